"""mk_decode_step_static -- the decode step for callers that cannot allocate device memory (code
under a framework whose caching allocator owns the GPU, or a latency-critical loop where
cudaMalloc / cudaFree could synchronise the device).  It keeps its scratch in a fixed-size
library-owned device array instead of the scratch bound with the context.

Checked against mk_decode_step through the C ABI on two calls in a row, with the tolerance the
other parity tests use (the two run the same kernel, so the results are in fact identical).
This file is collected last so that a failure here never hides another test's."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import persistent_megakernel_decode_sm_gb300 as mk  # noqa: E402
from gpu_helpers import REL_TOL, make_setup  # noqa: E402
from workload import empty_kv, make_weights, small_config  # noqa: E402


def _two_calls(name, use_static):
    s = make_setup(name)
    dec = mk.Decoder(mk.Schedule(s.cfg, mk.device_sm_count()), s.weights, s.kv)
    toks, pos = list(s.tokens), list(s.pos)
    out = []
    for _ in range(2):
        nxt = dec.step_static(toks, pos) if use_static else dec.step(toks, pos)
        out.append((dec.logits.cpu().numpy().copy(), list(nxt)))
        toks, pos = nxt, [p + 1 for p in pos]
    kv = (s.kv.k.cpu().clone(), s.kv.v.cpu().clone())
    dec.close()
    return out, kv


@pytest.mark.parametrize("name", ["tiny", "llama1b_ctx512"])
def test_static_scratch_step_matches_bound_scratch_step(name):
    ref, kv_ref = _two_calls(name, use_static=False)
    got, kv_got = _two_calls(name, use_static=True)
    for (lr, tr), (lg, tg) in zip(ref, got):
        scale = float(np.max(np.abs(lr)))
        assert float(np.max(np.abs(lg - lr))) <= REL_TOL * scale
        assert tg == tr
    assert torch.equal(kv_ref[0], kv_got[0]) and torch.equal(kv_ref[1], kv_got[1])


def test_static_scratch_rejects_a_step_larger_than_the_array():
    cfg = small_config(max_seq=131072)   # the RoPE table alone needs 32 MiB
    w = make_weights(cfg, seed=0, device="cuda")
    kv = empty_kv(cfg, device="cuda")
    dec = mk.Decoder(mk.Schedule(cfg, mk.device_sm_count()), w, kv)
    with pytest.raises(mk.MkError) as e:
        dec.step_static([1], [0])
    assert e.value.status == mk.MK_ERR_CAPACITY
    dec.step([1], [0])   # the context is still usable through its bound scratch
    dec.close()


def _tokens_logits_kv(dec, s, kinds):
    """Runs one step per entry of `kinds` ("b": the bound scratch, "s": the static array),
    teacher-forced from the set-up's first token; returns every step's logits and tokens and the
    final cache."""
    toks, pos = list(s.tokens), list(s.pos)
    out = []
    for k in kinds:
        nxt = dec.step_static(toks, pos) if k == "s" else dec.step(toks, pos)
        out.append((dec.logits.cpu().clone(), list(nxt)))
        toks, pos = nxt, [p + 1 for p in pos]
    return out, (s.kv.k.cpu().clone(), s.kv.v.cpu().clone())


def test_static_and_bound_steps_interleaved_on_one_context():
    # six static steps between two bound steps: the SwiGLU output's 3-bit step tag repeats every
    # seven steps, so the bound scratch left behind by the first step must not pass for the
    # eighth step's data.  Bit-identical to eight bound steps.
    kinds = "bssssssb"
    runs = []
    for pattern in (kinds, "b" * len(kinds)):
        s = make_setup("tiny")
        dec = mk.Decoder(mk.Schedule(s.cfg, mk.device_sm_count()), s.weights, s.kv)
        runs.append(_tokens_logits_kv(dec, s, pattern))
        dec.close()
    (got, kv_got), (ref, kv_ref) = runs
    for (lg, tg), (lr, tr) in zip(got, ref):
        assert torch.equal(lg, lr) and tg == tr
    assert torch.equal(kv_got[0], kv_ref[0]) and torch.equal(kv_got[1], kv_ref[1])


def test_two_contexts_share_the_static_array_alternately():
    # each call finds the other context's contents in the array and must not read them
    sa, sb = make_setup("tiny"), make_setup("tiny", seed=1)
    da = mk.Decoder(mk.Schedule(sa.cfg, mk.device_sm_count()), sa.weights, sa.kv)
    db = mk.Decoder(mk.Schedule(sb.cfg, mk.device_sm_count()), sb.weights, sb.kv)
    ta, pa, tb, pb = list(sa.tokens), list(sa.pos), list(sb.tokens), list(sb.pos)
    got_a, got_b = [], []
    for _ in range(3):
        na = da.step_static(ta, pa)
        got_a.append(da.logits.cpu().clone())
        nb = db.step_static(tb, pb)
        got_b.append(db.logits.cpu().clone())
        ta, pa, tb, pb = na, [p + 1 for p in pa], nb, [p + 1 for p in pb]
    da.close()
    db.close()
    for s, got in ((make_setup("tiny"), got_a), (make_setup("tiny", seed=1), got_b)):
        dec = mk.Decoder(mk.Schedule(s.cfg, mk.device_sm_count()), s.weights, s.kv)
        ref, _ = _tokens_logits_kv(dec, s, "bbb")
        dec.close()
        for g, (r, _) in zip(got, ref):
            assert torch.equal(g, r)

