"""Variable-length re-planning (schedule KV windows, mk_rebind_schedule) on the GPU.

- A batch-8 schedule whose attention tiles cover only each sequence's window decodes bit for bit
  like the full schedule (tokens, logits, appended K/V): chunks past pos never contribute.
- A step past a window is refused (MK_ERR_ARG) before anything is launched; after
  mk_rebind_schedule moves the binding to wider windows, decoding continues where it stopped and
  still equals the full-schedule run bit for bit, also through a persistent multi-step launch.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import persistent_megakernel_decode_sm_gb300 as mk  # noqa: E402
from gpu_helpers import make_setup  # noqa: E402
from workload import KVCache  # noqa: E402


def _clone_kv(kv):
    return KVCache(kv.k.clone(), kv.v.clone())


def _run_steps(dec, tokens, pos, n):
    out = []
    t = list(tokens)
    for i in range(n):
        t = dec.step(t, [p + i for p in pos])
        out.append(t)
    return out


@pytest.mark.parametrize("S", [None, 37])
def test_windowed_schedule_equals_full_schedule(S):
    s = make_setup("llama1b_batch8")
    S = S or mk.device_sm_count()
    n = 3
    kv_b = _clone_kv(s.kv)
    full = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, s.kv)
    ref = _run_steps(full, s.tokens, s.pos, n)
    win = mk.Schedule(s.cfg, S, kv_limit=[p + n for p in s.pos])
    assert (win.queues()[..., 0] == 2).sum() < (full.sched.queues()[..., 0] == 2).sum()   # fewer attention tiles
    dec = mk.Decoder(win, s.weights, kv_b)
    got = _run_steps(dec, s.tokens, s.pos, n)
    assert got == ref
    assert torch.equal(dec.logits, full.logits)
    assert torch.equal(s.kv.k, kv_b.k) and torch.equal(s.kv.v, kv_b.v)
    full.close()
    dec.close()


def test_step_past_the_window_is_refused_then_rebind_continues():
    s = make_setup("llama1b_batch8")
    S = mk.device_sm_count()
    kv_b = _clone_kv(s.kv)
    full = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, s.kv)
    ref = _run_steps(full, s.tokens, s.pos, 6)
    narrow = mk.Schedule(s.cfg, S, kv_limit=[p + 2 for p in s.pos])
    dec = mk.Decoder(narrow, s.weights, kv_b)
    got = _run_steps(dec, s.tokens, s.pos, 2)
    with pytest.raises(mk.MkError) as e:
        dec.step(got[-1], [p + 2 for p in s.pos])   # position p + 2 is outside [0, p + 2)
    assert e.value.status == mk.MK_ERR_ARG
    wide = mk.Schedule(s.cfg, S, kv_limit=[p + 64 for p in s.pos], shuffle_seed=3)
    dec.rebind(wide)
    got += _run_steps(dec, got[-1], [p + 2 for p in s.pos], 2)
    got += dec.persistent(got[-1], [p + 4 for p in s.pos], 2)
    assert got == ref
    assert torch.equal(dec.logits, full.logits)
    assert torch.equal(s.kv.k, kv_b.k) and torch.equal(s.kv.v, kv_b.v)
    with pytest.raises(mk.MkError) as e:   # another model's schedule is refused
        dec.rebind(mk.Schedule(s.cfg, S // 2))
    assert e.value.status == mk.MK_ERR_ARG
    dec.status()
    full.close()
    dec.close()
