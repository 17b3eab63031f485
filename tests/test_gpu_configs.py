"""GPU parity of the megakernel against the CPU oracle on the larger configurations, through the
C ABI (libmk.so): a long context (17 attention chunks of 512 positions per group, combined over
partials in L2), batch 8 with uneven KV lengths (the tensor-core kernel: 16-row TMA pages, every
sequence's inputs staged once per range, COMB tiles), and the 8B shape (8 chunks per lane, untied
LM head).

Tolerances as in test_gpu_parity: logits within max |error| <= 1e-2 * max |oracle logit| per
sequence, the greedy token equal wherever the oracle's top-2 margin exceeds 0.05, appended K/V
within one bf16 step of the oracle's codes (scale-aware, see gpu_helpers.kv_agreement).
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import persistent_megakernel_decode_sm_gb300 as mk  # noqa: E402
from gpu_helpers import REL_TOL, kv_agreement, make_setup, run_parity  # noqa: E402


def _run(name: str, steps: int):
    s = make_setup(name)
    dec = mk.Decoder(mk.Schedule(s.cfg, mk.device_sm_count()), s.weights, s.kv)
    r = run_parity(s, dec, steps=steps)
    assert r["rel"] <= REL_TOL, r
    assert not r["token_mismatch"], r
    kv = kv_agreement(s, [list(range(p, p + steps)) for p in s.pos])
    assert kv["worst_in_steps"] <= 1.0 and kv["frac_equal"] > 0.97, kv
    dec.close()
    del s, dec
    torch.cuda.empty_cache()
    return r


def test_llama1b_long_context_parity():
    _run("llama1b_ctx8192", steps=2)


def test_llama1b_long_context_bit_identical_across_sm_counts():
    # 17 attention chunks of 512 positions per group, combined in chunk order
    outs = []
    for S in (mk.device_sm_count(), 76):
        s = make_setup("llama1b_ctx8192")
        dec = mk.Decoder(mk.Schedule(s.cfg, S), s.weights, s.kv)
        dec.step(s.tokens, s.pos)
        outs.append((dec.logits.cpu().clone(), s.kv.k[:, :, :, s.pos[0]].cpu().clone(),
                     s.kv.v[:, :, :, s.pos[0]].cpu().clone()))
        dec.close()
        del s, dec
        torch.cuda.empty_cache()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_llama1b_batch8_parity():
    r = _run("llama1b_batch8", steps=2)
    assert r["token_checked"] >= 1


def test_llama8b_parity():
    _run("llama8b_ctx2048", steps=1)
