"""The batch > 1 kernel (and the attention body both kernels share) on small shapes chosen to
reach their edge cases, against the oracle.

Each case runs teacher-forced steps through the C ABI and compares logits and tokens with the
oracle (tolerances of test_gpu_parity), then checks that a schedule for another SM count gives
bit-identical outputs.  The shapes cover:
- row lengths that are no multiple of the 256-element tensor box edge (688: boxes of 16);
- a page of 512 positions, so the last slice of a row is partly past the matrix (zero fill);
- rows longer than one 2048-position staging range with a short last range (2560);
- two query heads per KV group (padded head columns), and eight (the wide head path) at
  head_dim 32; head_dim 128;
- 3 and 5 sequences (MMA columns past the batch), with uneven KV lengths over several chunks.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import persistent_megakernel_decode_sm_gb300 as mk  # noqa: E402
from gpu_helpers import REL_TOL, make_setup, run_parity  # noqa: E402
from workload import small_config  # noqa: E402

CASES = {
    "b3_ffn688": (dict(batch=3, max_seq=300), [17, 130, 259], {}),
    "b3_ffn688_p16k": (dict(batch=3, max_seq=300), [5, 200, 64], dict(page_bytes=16384)),
    "b5_ffn2560": (dict(batch=5, ffn=2560, max_seq=200), [40, 1, 129, 77, 150], {}),
    "b2_hpg8_d32": (dict(batch=2, n_q_heads=16, n_kv_heads=2, head_dim=32, max_seq=260), [100, 240], {}),
    "b2_d128": (dict(batch=2, n_q_heads=4, n_kv_heads=2, head_dim=128, max_seq=300), [129, 3], {}),
    # the same attention body in the batch-1 kernel
    "b1_hpg8_d32": (dict(batch=1, n_q_heads=16, n_kv_heads=2, head_dim=32, max_seq=300), [257], {}),
    "b1_d128": (dict(batch=1, n_q_heads=4, n_kv_heads=2, head_dim=128, max_seq=300), [200], {}),
}


@pytest.mark.parametrize("case", list(CASES))
def test_batched_edge_shapes_match_the_oracle(case):
    over, lens, opts = CASES[case]
    cfg = small_config(**over)
    s = make_setup("tiny", cfg=cfg, kv_len=lens)
    dec = mk.Decoder(mk.Schedule(cfg, mk.device_sm_count(), **opts), s.weights, s.kv)
    r = run_parity(s, dec, steps=3)
    assert r["rel"] <= REL_TOL, r
    assert not r["token_mismatch"], r
    dec.close()


@pytest.mark.parametrize("case", ["b3_ffn688", "b5_ffn2560"])
def test_batched_outputs_bit_identical_across_sm_counts(case):
    over, lens, opts = CASES[case]
    cfg = small_config(**over)
    outs = []
    for S in (mk.device_sm_count(), 37):
        s = make_setup("tiny", cfg=cfg, kv_len=lens)
        dec = mk.Decoder(mk.Schedule(cfg, S, **opts), s.weights, s.kv)
        toks = dec.step(s.tokens, s.pos)
        outs.append((toks, dec.logits.cpu().clone(), s.kv.k.cpu().clone(), s.kv.v.cpu().clone()))
        dec.close()
    assert outs[0][0] == outs[1][0]
    for a, b in zip(outs[0][1:], outs[1][1:]):
        assert torch.equal(a, b)
