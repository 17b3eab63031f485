"""GPU parity of the megakernel against the CPU oracle, through the C ABI (libmk.so).

Tolerances (the parity criterion of this decoder): logits within
max |error| <= 1e-2 * max |oracle logit| per sequence; the greedy token equal wherever the
oracle's top-2 logit margin exceeds 0.05; appended K/V equal to the oracle's bf16 codes up to one
unit in the last place (the fp32 sums behind them are ordered differently).  Outputs are
bit-identical across SM counts, queue placements and the two synchronisation modes
(epoch-tagged activations, completion counters).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import persistent_megakernel_decode_sm_gb300 as mk  # noqa: E402
from gpu_helpers import REL_TOL, kv_agreement, make_setup, run_parity  # noqa: E402
from workload import get_workload  # noqa: E402


def _assert_parity(r):
    assert r["rel"] <= REL_TOL, r
    assert not r["token_mismatch"], r


def test_smoke():
    import __graft_entry__
    __graft_entry__.smoke()


def test_tiny_greedy_decode_parity():
    s = make_setup("tiny")
    dec = mk.Decoder(mk.Schedule(s.cfg, mk.device_sm_count()), s.weights, s.kv)
    r = run_parity(s, dec, steps=get_workload("tiny").decode_steps)
    _assert_parity(r)
    assert r["token_checked"] >= 4
    kv = kv_agreement(s, [list(range(16, 24))])
    assert kv["worst_in_steps"] <= 1.0 and kv["frac_equal"] > 0.97, kv


@pytest.mark.parametrize("S_div,shuffle", [(1, 0), (2, 0), (0, 0), (1, 99)])
def test_tiny_bit_identical_across_sm_counts(S_div, shuffle):
    full = mk.device_sm_count()
    S = 37 if S_div == 0 else full // S_div
    outs = []
    for s_count, seed in ((full, 0), (S, shuffle)):
        s = make_setup("tiny")
        dec = mk.Decoder(mk.Schedule(s.cfg, s_count, shuffle_seed=seed), s.weights, s.kv)
        toks, pos = list(s.tokens), list(s.pos)
        res = []
        for _ in range(3):
            nxt = dec.step(toks, pos)
            res.append(dec.logits.cpu().clone())
            toks, pos = nxt, [p + 1 for p in pos]
        res.append(s.kv.k.cpu().clone())
        res.append(s.kv.v.cpu().clone())
        outs.append(res)
        dec.close()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_llama1b_ctx512_parity():
    # 16 teacher-forced steps, every fourth (and the last) compared with the oracle in full
    s = make_setup("llama1b_ctx512")
    dec = mk.Decoder(mk.Schedule(s.cfg, mk.device_sm_count()), s.weights, s.kv)
    r = run_parity(s, dec, steps=16, check_every=4)
    _assert_parity(r)
    assert r["token_checked"] >= 2
    kv = kv_agreement(s, [list(range(512, 528))])
    assert kv["worst_in_steps"] <= 1.0 and kv["frac_equal"] > 0.97, kv


def _llama1b_outputs(name, s_count, seed, steps):
    s = make_setup(name)
    dec = mk.Decoder(mk.Schedule(s.cfg, s_count, shuffle_seed=seed), s.weights, s.kv)
    out = _steps(dec, s, steps)
    dec.close()
    del s, dec
    torch.cuda.empty_cache()
    return out


@pytest.mark.parametrize("S_spec,shuffle", [("half", 0), ("37", 0), ("full", 7), ("8", 11)])
def test_llama1b_bit_identical_across_sm_counts(S_spec, shuffle):
    # the full-size paths: two segments per row (the segment sums meet in shared memory), the
    # MLP down projection's eight-segment rows polled per warp, ten-chunk attention groups combined
    # in chunk order -- identical logits and caches whatever the SM count and placement (at 8
    # queues, shuffled, every queue holds about ten attention chunk tiles of a layer, and the
    # combining tile waits inside the wave for chunks that other queues run)
    full = mk.device_sm_count()
    S = {"half": full // 2, "37": 37, "full": full, "8": 8}[S_spec]
    ref = _llama1b_outputs("llama1b_ctx512", full, 0, 2)
    got = _llama1b_outputs("llama1b_ctx512", S, shuffle, 2)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def test_device_timeout_is_reported_and_gpu_stays_usable():
    s = make_setup("tiny")
    sched = mk.Schedule(s.cfg, mk.device_sm_count())
    q = sched.queues()
    # plant an unsatisfiable wait (need one more than the producers ever publish) in the first
    # instruction that waits on something
    sm, slot = [(i, j) for i in range(q.shape[0]) for j in range(q.shape[1]) if q[i, j, 6] > 0][0]
    sched.patch(sm, slot, 8, int(q[sm, slot, 8]) + 1)
    dec = mk.Decoder(sched, s.weights, s.kv, timeout_ns=20_000_000)
    dec.set_sync("counters")   # every instruction waits its counters
    with pytest.raises(mk.MkError) as ei:
        dec.step(s.tokens, s.pos)
    assert ei.value.status == mk.MK_ERR_TIMEOUT
    with pytest.raises(mk.MkError) as ei:
        dec.step(s.tokens, s.pos)
    assert ei.value.status == mk.MK_ERR_POISONED
    dec.close()
    # the GPU and a fresh context still work
    s2 = make_setup("tiny")
    dec2 = mk.Decoder(mk.Schedule(s2.cfg, mk.device_sm_count()), s2.weights, s2.kv)
    _assert_parity(run_parity(s2, dec2, steps=1))


def test_invalid_opcode_is_reported():
    s = make_setup("tiny")
    sched = mk.Schedule(s.cfg, mk.device_sm_count())
    sched.patch(0, 0, 0, 99)
    dec = mk.Decoder(sched, s.weights, s.kv, timeout_ns=50_000_000)
    with pytest.raises(mk.MkError) as ei:
        dec.step(s.tokens, s.pos)
    assert ei.value.status == mk.MK_ERR_OPCODE
    dec.close()
    s2 = make_setup("tiny")
    dec2 = mk.Decoder(mk.Schedule(s2.cfg, mk.device_sm_count()), s2.weights, s2.kv)
    _assert_parity(run_parity(s2, dec2, steps=1))


def _steps(dec, s, n):
    toks, pos = list(s.tokens), list(s.pos)
    res = []
    for _ in range(n):
        nxt = dec.step(toks, pos)
        res.append(dec.logits.cpu().clone())
        toks, pos = nxt, [p + 1 for p in pos]
    res.append(s.kv.k.cpu().clone())
    res.append(s.kv.v.cpu().clone())
    return res


@pytest.mark.parametrize("name,steps", [("tiny", 3), ("llama1b_ctx512", 2)])
def test_sync_modes_bit_identical(name, steps):
    outs = []
    for mode in ("tags", "counters"):
        s = make_setup(name)
        dec = mk.Decoder(mk.Schedule(s.cfg, mk.device_sm_count()), s.weights, s.kv)
        dec.set_sync(mode)
        outs.append(_steps(dec, s, steps))
        dec.close()
        del s
        torch.cuda.empty_cache()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_tagged_wait_timeout_is_reported():
    # shift the rows of one last-layer MLP-down tile onto its neighbour's: the tile still
    # publishes its completion, so the LM-head tiles pass their counter waits, but some words of
    # the final residual stream never receive this step's tag and the LM-head tiles, reading
    # them, give up after the time budget (the argmax sits behind them: no other wait is open)
    s = make_setup("tiny")
    sched = mk.Schedule(s.cfg, 16)   # 16 queues: every one holds LM-head tiles
    q = sched.queues()
    am = [(i, j) for i in range(q.shape[0]) for j in range(q.shape[1]) if q[i, j, 0] == 8][0]
    assert 7 in q[am[0], :am[1], 0], "the argmax must queue behind an LM-head tile"
    last = s.cfg.n_layers - 1
    sm, slot = [(i, j) for i in range(q.shape[0]) for j in range(q.shape[1])
                if q[i, j, 0] == 6 and q[i, j, 1] == last and q[i, j, 3] == 0][0]
    sched.patch(sm, slot, 3, int(q[sm, slot, 4]))
    dec = mk.Decoder(sched, s.weights, s.kv, timeout_ns=20_000_000)
    with pytest.raises(mk.MkError) as ei:
        dec.step(s.tokens, s.pos)
    assert ei.value.status == mk.MK_ERR_TIMEOUT
    st, info = dec.status_code()
    assert st == mk.MK_ERR_TIMEOUT and info[6] == 5, (st, info)   # a tagged-data poll gave up
    dec.close()
    s2 = make_setup("tiny")
    dec2 = mk.Decoder(mk.Schedule(s2.cfg, mk.device_sm_count()), s2.weights, s2.kv)
    _assert_parity(run_parity(s2, dec2, steps=1))


def test_lm_partials_of_ctas_without_lm_rows_are_cleared_at_bind():
    # only four CTAs hold LM-head tiles; every other CTA's per-warp (max, index, epoch) partials
    # must come from the bind's clearing, not from whatever the scratch held before: fill the
    # scratch with entries (1e30, index 0, epoch 0) -- they would win the first step's argmax if
    # the bind left any of them in place
    s = make_setup("tiny")
    sched = mk.Schedule(s.cfg, mk.device_sm_count(), rows_lm=s.cfg.vocab // 4)
    poison = torch.zeros((sched.scratch_bytes // 16 + 16, 4), dtype=torch.int32, device="cuda")
    poison[:, 0] = int(np.array([1e30], dtype=np.float32).view(np.int32)[0])
    dec = mk.Decoder(sched, s.weights, s.kv, scratch=poison.view(-1))
    r = run_parity(s, dec, steps=2)
    _assert_parity(r)
    assert r["token_checked"] >= 1
    dec.close()


def test_decode_from_position_zero():
    # an empty cache: the first position attends to itself only (the attention output is v0)
    s = make_setup("tiny")
    from workload import empty_kv
    s.kv = empty_kv(s.cfg, device="cuda")
    s.kh[...] = 0
    s.vh[...] = 0
    s.pos = [0]
    dec = mk.Decoder(mk.Schedule(s.cfg, mk.device_sm_count()), s.weights, s.kv)
    r = run_parity(s, dec, steps=4)
    _assert_parity(r)
    kv = kv_agreement(s, [[0, 1, 2, 3]])
    assert kv["worst_in_steps"] <= 1.0 and kv["frac_equal"] > 0.97, kv
    dec.close()


@pytest.mark.parametrize("name", ["tiny", "llama1b_ctx512"])
def test_repeated_runs_bit_identical(name):
    # the same steps on fresh contexts, four times: logits and caches must not depend on timing
    def run():
        s = make_setup(name)
        dec = mk.Decoder(mk.Schedule(s.cfg, mk.device_sm_count()), s.weights, s.kv)
        out = _steps(dec, s, 3)
        dec.close()
        return out
    ref = run()
    for _ in range(3):
        for a, b in zip(run(), ref):
            assert torch.equal(a, b)
