"""Persistent multi-step decoding through the C ABI (mk_decode_persistent_*): ONE resident launch
runs up to n steps, each step's greedy token feeding the next step's embedding on the device,
and a host stop request ends it at a step boundary.

- A persistent launch of n steps matches n chained launches (mk_decode_steps) bit for bit:
  tokens, last logits and the appended K/V, at batch 1 and batch 8, in both sync modes and on a
  grid smaller than the device.
- A stop requested before the launch starts running ends it after exactly one step; a stop
  requested mid-run ends it within two steps of the progress the host saw, with the tokens of
  the steps it ran equal to the chained run's.
- The context continues after a stopped run: the next launch starts at the following epoch and
  position and again matches the chained reference bit for bit.
- While a launch is in flight the other entry points refuse the context.
"""
import time

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import persistent_megakernel_decode_sm_gb300 as mk  # noqa: E402
from gpu_helpers import MARGIN, make_setup  # noqa: E402
from oracle import Oracle  # noqa: E402
from workload import KVCache  # noqa: E402


def _clone_kv(kv):
    return KVCache(kv.k.clone(), kv.v.clone())


@pytest.mark.parametrize("name,n,S,sync", [("tiny", 8, None, "tags"), ("tiny", 8, None, "counters"),
                                           ("tiny", 8, 5, "tags"), ("llama1b_ctx512", 16, None, "tags"),
                                           ("llama1b_ctx512", 6, 37, "tags"), ("llama1b_batch8", 4, None, "tags")])
def test_persistent_run_equals_chained_steps(name, n, S, sync):
    s = make_setup(name)
    S = S or mk.device_sm_count()
    kv_b = _clone_kv(s.kv)
    a = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, s.kv)
    a.set_sync(sync)
    toks_a = a.persistent(s.tokens, s.pos, n)
    b = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, kv_b)
    b.set_sync(sync)
    toks_b = b.steps(s.tokens, s.pos, n)
    assert toks_a == toks_b
    assert torch.equal(a.logits, b.logits)
    assert torch.equal(s.kv.k, kv_b.k) and torch.equal(s.kv.v, kv_b.v)
    assert a.persistent_progress() == n
    a.close()
    b.close()


def test_tiny_persistent_run_follows_the_oracle():
    s = make_setup("tiny")
    dec = mk.Decoder(mk.Schedule(s.cfg, mk.device_sm_count()), s.weights, s.kv)
    n = 8
    toks = dec.persistent(s.tokens, s.pos, n)
    assert len(toks) == n
    orc = Oracle("f32")
    tokens, pos, checked = list(s.tokens), list(s.pos), 0
    for i in range(n):
        o_logits, o_next = orc.decode_step(s.cfg, s.host, s.kh, s.vh, tokens, pos)
        top = np.sort(o_logits[0])[-2:]
        if top[1] - top[0] > MARGIN:
            checked += 1
            assert toks[i] == list(o_next), (i, toks[i], o_next)
        tokens, pos = list(toks[i]), [p + 1 for p in pos]
    assert checked >= n // 2
    dec.close()


def test_stop_before_the_launch_runs_ends_after_one_step():
    s = make_setup("llama1b_ctx512")
    S = mk.device_sm_count()
    kv_b = _clone_kv(s.kv)
    dec = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, s.kv)
    torch.cuda._sleep(200_000_000)   # ~0.1 s of device time ahead of the launch on the bound stream
    dec.persistent_start(s.tokens, s.pos, 8)
    dec.persistent_stop()            # set while the sleep still holds the launch back
    toks = dec.persistent_wait()
    assert len(toks) == 1
    ref = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, kv_b)
    assert toks == [ref.step(s.tokens, s.pos)]
    assert torch.equal(dec.logits, ref.logits)
    assert torch.equal(s.kv.k, kv_b.k) and torch.equal(s.kv.v, kv_b.v)
    dec.close()
    ref.close()


def test_stop_mid_run_then_continue():
    s = make_setup("llama1b_ctx512")
    S = mk.device_sm_count()
    n = 100
    kv_b = _clone_kv(s.kv)
    dec = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, s.kv)
    dec.persistent_start(s.tokens, s.pos, n)
    seen, t0 = 0, time.time()
    while seen < 3 and time.time() - t0 < 30:
        seen = dec.persistent_progress()
    dec.persistent_stop()
    toks = dec.persistent_wait()
    done = len(toks)
    assert 3 <= done <= n
    assert done == n or done <= seen + 2, (done, seen)
    # the chained reference over the same steps, then both continue for 4 more
    m = 4
    ref = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, kv_b)
    ref_toks = ref.steps(s.tokens, s.pos, min(done + m, s.cfg.max_seq - s.pos[0]))
    assert toks == ref_toks[:done]
    more = dec.persistent(toks[-1], [p + done for p in s.pos], m)
    assert more == ref_toks[done:done + m]
    assert torch.equal(dec.logits, ref.logits)
    assert torch.equal(s.kv.k, kv_b.k) and torch.equal(s.kv.v, kv_b.v)
    dec.close()
    ref.close()


def test_in_flight_launch_refuses_other_calls():
    s = make_setup("tiny")
    dec = mk.Decoder(mk.Schedule(s.cfg, mk.device_sm_count()), s.weights, s.kv)
    with pytest.raises(mk.MkError) as e:
        dec.persistent_wait()                      # nothing in flight
    assert e.value.status == mk.MK_ERR_ARG
    with pytest.raises(mk.MkError) as e:
        dec.persistent_start(s.tokens, [s.cfg.max_seq - 2], 3)   # positions past the cache
    assert e.value.status == mk.MK_ERR_ARG
    torch.cuda._sleep(50_000_000)
    dec.persistent_start(s.tokens, s.pos, 4)
    for call in (lambda: dec.step(s.tokens, s.pos), lambda: dec.step_static(s.tokens, s.pos),
                 lambda: dec.persistent_start(s.tokens, s.pos, 2), lambda: dec.status()):
        with pytest.raises(mk.MkError) as e:
            call()
        assert e.value.status == mk.MK_ERR_ARG
    toks = dec.persistent_wait()
    assert len(toks) == 4
    dec.status()   # the context is healthy
    dec.close()
