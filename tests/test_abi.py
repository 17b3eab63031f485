"""The C-ABI library loads and exports every function include/mk.h declares; host-side argument
checks work without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
mk = pytest.importorskip("persistent_megakernel_decode_sm_gb300")


def header_functions():
    text = open(os.path.join(ROOT, "include", "mk.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_function_is_exported():
    names = header_functions()
    assert len(names) >= 15
    lib = ctypes.CDLL(mk.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(mk.EXPORTS)


def test_build_schedule_rejects_bad_arguments():
    from workload import small_config
    with pytest.raises(mk.MkError) as e:
        mk.Schedule(small_config(n_kv_heads=3), 4)
    assert e.value.status == mk.MK_ERR_ARG
    with pytest.raises(mk.MkError):
        mk.Schedule(small_config(), 0)
    with pytest.raises(mk.MkError):
        mk.Schedule(small_config(head_dim=24), 4)
    with pytest.raises(mk.MkError):
        mk.Schedule(small_config(batch=9), 4)
    with pytest.raises(mk.MkError):
        mk.Schedule(small_config(), 4, rows_qkv=65)       # more rows than head_dim
    with pytest.raises(mk.MkError):
        mk.Schedule(small_config(hidden=1024), 4, page_bytes=1024)   # holds no gate/up row
    with pytest.raises(mk.MkError):
        mk.Schedule(small_config(), 4, page_bytes=1000)
    # batch > 1: a page is a 16-row block over page_bytes / 32 <= 2048 positions, and a tile of
    # rows longer than 2048 keeps at most 64 rows of sums
    with pytest.raises(mk.MkError):
        mk.Schedule(small_config(batch=2), 4, page_bytes=131072)
    with pytest.raises(mk.MkError):
        mk.Schedule(small_config(batch=2, ffn=4096), 4, rows_down=65)
    assert mk.Schedule(small_config(batch=2, ffn=4096), 4, rows_down=64).attn_chunk > 0


def test_patch_and_scratch_size():
    from workload import small_config
    s = mk.Schedule(small_config(), 3)
    q = s.queues()
    s.patch(1, 0, 5, 77)
    assert s.queues()[1, 0, 5] == 77 and q[1, 0, 5] != 77 or q[1, 0, 5] == 77
    with pytest.raises(mk.MkError):
        s.patch(3, 0, 0, 1)
    assert s.scratch_bytes > 0 and s.scratch_bytes % 256 == 0


def test_last_error_message_is_set():
    from workload import small_config
    with pytest.raises(mk.MkError) as e:
        mk.Schedule(small_config(n_q_heads=5, n_kv_heads=2), 4)
    assert "n_kv_heads" in str(e.value)


def test_step_calls_reject_null_and_bad_arguments_without_a_device():
    lib = mk.lib
    B = 1
    t = (ctypes.c_int32 * B)(1)
    p = (ctypes.c_int32 * B)(0)
    out = (ctypes.c_int32 * 8)()
    dummy = ctypes.c_void_p(256)   # never dereferenced: every call below fails its host checks first
    assert lib.mk_decode_steps(None, t, p, 0, dummy, dummy, out) == mk.MK_ERR_ARG      # n_steps < 1
    assert lib.mk_decode_steps(None, t, p, 2, dummy, None, out) == mk.MK_ERR_ARG       # no token buffer
    assert lib.mk_decode_steps(None, t, p, 2, dummy, dummy, None) == mk.MK_ERR_ARG     # no host copy
    assert lib.mk_decode_steps(None, t, p, 2, dummy, dummy, out) == mk.MK_ERR_ARG      # no context
    assert lib.mk_launch_step(None, t, p, dummy, None) == mk.MK_ERR_ARG
    assert lib.mk_decode_step(None, t, p, dummy, out) == mk.MK_ERR_ARG
    n = ctypes.c_int32(0)
    assert lib.mk_decode_persistent_start(None, t, p, 4, dummy, dummy) == mk.MK_ERR_ARG   # no context
    assert lib.mk_decode_persistent_stop(None) == mk.MK_ERR_ARG
    assert lib.mk_decode_persistent_progress(None, ctypes.byref(n)) == mk.MK_ERR_ARG
    assert lib.mk_decode_persistent_wait(None, ctypes.byref(n), out) == mk.MK_ERR_ARG
