"""Chained multi-step decoding through the C ABI (mk_decode_steps): each step's greedy token
feeds the next step's embedding on the device, with one host synchronisation per call.

- The steps match single steps bit for bit (same tokens, logits and appended K/V as
  mk_decode_step called once per step with the previous step's token).
- Fed the megakernel's own tokens, the CPU oracle picks the same token wherever its top-2 margin
  exceeds 0.05, and the last step's logits agree within max |error| <= 1e-2 * max |oracle logit|.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import persistent_megakernel_decode_sm_gb300 as mk  # noqa: E402
from gpu_helpers import MARGIN, REL_TOL, compare_step, make_setup  # noqa: E402
from oracle import Oracle  # noqa: E402
from workload import KVCache  # noqa: E402


def _clone_kv(kv):
    return KVCache(kv.k.clone(), kv.v.clone())


@pytest.mark.parametrize("name,n", [("tiny", 8), ("llama1b_ctx512", 3)])
def test_chained_steps_equal_single_steps(name, n):
    s = make_setup(name)
    S = mk.device_sm_count()
    kv_b = _clone_kv(s.kv)
    a = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, s.kv)
    toks_a = a.steps(s.tokens, s.pos, n)
    b = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, kv_b)
    t, toks_b = list(s.tokens), []
    for i in range(n):
        t = b.step(t, [p + i for p in s.pos])
        toks_b.append(t)
    assert toks_a == toks_b
    assert torch.equal(a.logits, b.logits)
    assert torch.equal(s.kv.k, kv_b.k) and torch.equal(s.kv.v, kv_b.v)
    a.close()
    b.close()


def test_tiny_chained_steps_follow_the_oracle():
    s = make_setup("tiny")
    dec = mk.Decoder(mk.Schedule(s.cfg, mk.device_sm_count()), s.weights, s.kv)
    n = 8
    toks = dec.steps(s.tokens, s.pos, n)
    orc = Oracle("f32")
    tokens, pos, checked = list(s.tokens), list(s.pos), 0
    for i in range(n):
        o_logits, o_next = orc.decode_step(s.cfg, s.host, s.kh, s.vh, tokens, pos)
        top = np.sort(o_logits[0])[-2:]
        if top[1] - top[0] > MARGIN:
            checked += 1
            assert toks[i] == list(o_next), (i, toks[i], o_next)
        tokens, pos = list(toks[i]), [p + 1 for p in pos]
    r = compare_step(dec.logits.cpu().numpy(), o_logits, toks[-1], list(o_next))
    assert r["rel"] <= REL_TOL, r
    assert checked >= n // 2
    dec.close()


def test_chained_steps_reject_positions_past_the_cache():
    s = make_setup("tiny")
    dec = mk.Decoder(mk.Schedule(s.cfg, mk.device_sm_count()), s.weights, s.kv)
    with pytest.raises(mk.MkError) as e:
        dec.steps(s.tokens, [s.cfg.max_seq - 2], 3)
    assert e.value.status == mk.MK_ERR_ARG
    assert len(dec.steps(s.tokens, s.pos, 1)) == 1   # nothing was launched by the rejected call
    dec.close()
