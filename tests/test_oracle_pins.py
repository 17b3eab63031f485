"""Pins of the CPU oracle to things other than itself (no GPU).

Every check here is a closed form, an invariant, a special case that reduces to a textbook
result or a library routine (torch / numpy in float64), or brute force on a tiny input.  The
"Inference MegaKernel" page prints no worked example, so nothing here is a stored value from
it.  Each group names the operator of the page's opcode list it pins (section "Hand-written
whole-model MegaKernel": RMS_NORM, QKV_MATVEC, ATTENTION, MLP_UP_GATE, MLP_DOWN, LM_HEAD).
"""
import math

import numpy as np
import pytest
import torch

from oracle import HostWeights, Oracle, kv_to_host
from workload import empty_kv, get_workload, make_weights, prefilled_kv, small_config, token_ids


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def widen(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


ONE_BF16 = np.uint16(0x3F80)


# ---------------------------------------------------------------- bf16 rounding (KV append)
def test_bf16_round_matches_torch(oracle32):
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000),
                           [0.0, -0.0, 1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8,
                            65504.0, 3.0e38, 1e-40, -2.5]]).astype(np.float32)
    want = bits(torch.from_numpy(vals).to(torch.bfloat16))
    got = np.array([oracle32.bf16_round(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)
    # ties go to even
    assert oracle32.bf16_round(1.0 + 2 ** -8) == 0x3F80
    assert oracle32.bf16_round(1.0 + 3 * 2 ** -8) == 0x3F82


# ---------------------------------------------------------------- RMS_NORM
def test_rmsnorm_output_rms_is_one_before_gain(oracle64):
    rng = np.random.default_rng(1)
    for n in (7, 256, 2048):
        x = rng.standard_normal(n) * 3.0
        eps = 1e-5
        out = oracle64.rmsnorm(x, np.full(n, ONE_BF16), eps)
        ms = np.mean(x * x)
        assert math.isclose(np.sqrt(np.mean(out * out)), math.sqrt(ms / (ms + eps)), rel_tol=1e-12)


def test_rmsnorm_eps_inside_sqrt_and_gain_per_element(oracle64):
    c, eps = 1e-3, 1e-5
    out = oracle64.rmsnorm(np.full(16, c), np.full(16, ONE_BF16), eps)
    assert np.allclose(out, c / math.sqrt(c * c + eps), rtol=1e-13)
    rng = np.random.default_rng(2)
    x = rng.standard_normal(64)
    g = bits(torch.from_numpy(rng.standard_normal(64)).to(torch.bfloat16))
    base = oracle64.rmsnorm(x, np.full(64, ONE_BF16), eps)
    assert np.allclose(oracle64.rmsnorm(x, g, eps), base * widen(g), rtol=1e-14, atol=0)
    # library routine: torch rms_norm in float64
    want = torch.nn.functional.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(widen(g)), eps)
    assert np.allclose(oracle64.rmsnorm(x, g, eps), want.numpy(), rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- matvec (QKV/O/MLP/LM_HEAD)
def test_matvec_one_hot_selects_column(oracle32, oracle64):
    rng = np.random.default_rng(3)
    W = bits(torch.from_numpy(rng.standard_normal((37, 300))).to(torch.bfloat16))
    for j in (0, 5, 299):
        x = np.zeros(300)
        x[j] = 1.0
        for o in (oracle32, oracle64):
            assert np.array_equal(o.matvec(W, x), widen(W[:, j]).astype(o.dtype))


def test_matvec_vs_numpy_float64(oracle32, oracle64):
    rng = np.random.default_rng(4)
    W = bits(torch.from_numpy(rng.standard_normal((53, 777)) * 0.02).to(torch.bfloat16))
    x = rng.standard_normal(777)
    want = widen(W) @ x
    assert np.allclose(oracle64.matvec(W, x), want, rtol=1e-12, atol=1e-13)
    bound = 777 * 2 ** -23 * (np.abs(widen(W)) @ np.abs(x)) * 2
    assert np.all(np.abs(oracle32.matvec(W, x.astype(np.float32)) - want) <= bound + 1e-6)


# ---------------------------------------------------------------- RoPE (QKV_MATVEC prologue)
def test_rope_identity_at_zero_and_pair_norms(oracle64):
    rng = np.random.default_rng(5)
    d, nh = 64, 3
    v = rng.standard_normal(nh * d)
    assert np.array_equal(oracle64.rope(v, nh, d, 0, 10000.0), v)
    r = oracle64.rope(v, nh, d, 1234, 500000.0).reshape(nh, d)
    v = v.reshape(nh, d)
    h = d // 2
    assert np.allclose(r[:, :h] ** 2 + r[:, h:] ** 2, v[:, :h] ** 2 + v[:, h:] ** 2, rtol=1e-12)


def test_rope_rotate_half_pairing_and_frequencies(oracle64):
    d, theta, pos = 8, 10000.0, 3
    for i in range(d // 2):
        e = np.zeros(d)
        e[i] = 1.0
        r = oracle64.rope(e, 1, d, pos, theta)
        a = pos * theta ** (-2.0 * i / d)
        want = np.zeros(d)
        want[i], want[i + d // 2] = math.cos(a), math.sin(a)
        assert np.allclose(r, want, atol=1e-15)
    # the complex-number form: (x_i + j x_{i+d/2}) * exp(j a_i)
    rng = np.random.default_rng(6)
    d = 64
    x = rng.standard_normal(d)
    z = (x[: d // 2] + 1j * x[d // 2:]) * np.exp(1j * 77 * 500000.0 ** (-2.0 * np.arange(d // 2) / d))
    r = oracle64.rope(x, 1, d, 77, 500000.0)
    assert np.allclose(r, np.concatenate([z.real, z.imag]), atol=1e-13)


def test_rope_scores_depend_only_on_relative_position(oracle64):
    rng = np.random.default_rng(7)
    d = 64
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    s1 = oracle64.rope(q, 1, d, 40, 10000.0) @ oracle64.rope(k, 1, d, 13, 10000.0)
    s2 = oracle64.rope(q, 1, d, 540, 10000.0) @ oracle64.rope(k, 1, d, 513, 10000.0)
    assert math.isclose(s1, s2, rel_tol=1e-10, abs_tol=1e-12)


# ---------------------------------------------------------------- ATTENTION
def _cache(rng, nkv, S, d, scale=1.0):
    return bits(torch.from_numpy(rng.standard_normal((nkv, S, d)) * scale).to(torch.bfloat16))


def test_attention_bruteforce_torch_softmax(oracle64):
    rng = np.random.default_rng(8)
    nq, nkv, d, S = 4, 2, 4, 8
    for pos in range(S):
        kc, vc = _cache(rng, nkv, S, d), _cache(rng, nkv, S, d)
        q = rng.standard_normal(nq * d)
        out, probs = oracle64.attention(q, kc, vc, nq, nkv, d, S, pos, want_probs=True)
        for h in range(nq):
            g = h // (nq // nkv)
            K = torch.from_numpy(widen(kc[g, : pos + 1]))
            V = torch.from_numpy(widen(vc[g, : pos + 1]))
            p = torch.softmax(K @ torch.from_numpy(q[h * d:(h + 1) * d]) / math.sqrt(d), dim=0)
            assert np.allclose(probs[h], p.numpy(), rtol=1e-12, atol=1e-15)
            assert np.allclose(out[h * d:(h + 1) * d], (p @ V).numpy(), rtol=1e-12, atol=1e-14)


def test_attention_special_cases(oracle32, oracle64):
    rng = np.random.default_rng(9)
    nq, nkv, d, S = 8, 2, 16, 12
    kc, vc = _cache(rng, nkv, S, d), _cache(rng, nkv, S, d)
    q = rng.standard_normal(nq * d)
    # a single position: o = v_0 exactly
    for o in (oracle32, oracle64):
        out = o.attention(q, kc, vc, nq, nkv, d, S, 0)
        for h in range(nq):
            assert np.array_equal(out[h * d:(h + 1) * d], widen(vc[h // 4, 0]).astype(o.dtype))
    # rows sum to one
    _, probs = oracle64.attention(q, kc, vc, nq, nkv, d, S, 9, want_probs=True)
    assert np.allclose(probs.sum(axis=1), 1.0, atol=1e-14)
    # equal keys: the output is the mean of the values over 0..pos
    kc2 = kc.copy()
    kc2[:, :] = kc[:, :1]
    out = oracle64.attention(q, kc2, vc, nq, nkv, d, S, 6)
    for h in range(nq):
        assert np.allclose(out[h * d:(h + 1) * d], widen(vc[h // 4, :7]).mean(axis=0), atol=1e-14)
    # positions after pos never matter; GQA: head h reads KV head h // (nq / nkv)
    vc3 = np.empty_like(vc)
    for g in range(nkv):
        vc3[g] = bits(torch.full((S, d), float(g + 1), dtype=torch.bfloat16))
    kc3 = kc.copy()
    kc3[:, 7:] = bits(torch.full((nkv, S - 7, d), 3.0e4, dtype=torch.bfloat16))
    out = oracle64.attention(q, kc3, vc3, nq, nkv, d, S, 6)
    for h in range(nq):
        assert np.allclose(out[h * d:(h + 1) * d], h // 4 + 1.0, atol=1e-13)
    # one dominant score: one-hot weights
    kc4 = np.zeros_like(kc)
    kc4[:, 3] = bits(torch.full((nkv, d), 50.0, dtype=torch.bfloat16))
    qq = np.ones(nq * d)
    _, probs = oracle64.attention(qq, kc4, vc, nq, nkv, d, S, 5, want_probs=True)
    assert np.allclose(probs[:, 3], 1.0, atol=1e-12)


# ---------------------------------------------------------------- MLP_UP_GATE (SiLU) / argmax
def test_silu_and_swiglu(oracle64):
    assert oracle64.silu(0.0) == 0.0
    assert math.isclose(oracle64.silu(1.0), 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)
    assert math.isclose(oracle64.silu(40.0), 40.0, rel_tol=1e-15)
    assert abs(oracle64.silu(-40.0)) < 1e-15
    rng = np.random.default_rng(10)
    a, u = rng.standard_normal(50), rng.standard_normal(50)
    want = torch.nn.functional.silu(torch.from_numpy(a)).numpy() * u
    assert np.allclose(oracle64.swiglu(a, u), want, rtol=1e-14, atol=1e-16)


def test_argmax_bruteforce_lowest_index_on_ties(oracle32):
    rng = np.random.default_rng(11)
    for _ in range(20):
        v = rng.integers(0, 5, 40).astype(np.float32)   # many ties
        assert oracle32.argmax(v) == int(np.argmax(v))   # numpy returns the first maximum
    assert oracle32.argmax(np.array([1.0, 3.0, 3.0], dtype=np.float32)) == 1


# ---------------------------------------------------------------- whole decode step
def _run(cfg, w, kv, tokens, pos, precision="f64"):
    o = Oracle(precision)
    hw = HostWeights(w)
    k, v = kv_to_host(kv)
    logits, nxt = o.decode_step(cfg, hw, k, v, tokens, pos)
    return logits, nxt, k, v


def _t64(b):
    return torch.from_numpy(widen(b))


def test_decode_zero_blocks_reduce_to_embedding_head():
    cfg = small_config(n_layers=2)
    w = make_weights(cfg, seed=3)
    for l in range(cfg.n_layers):
        w.wo[l].zero_()
        w.wdown[l].zero_()
    kv = prefilled_kv(cfg, [5], seed=3)
    tok = 1234
    logits, nxt, _, _ = _run(cfg, w, kv, [tok], [5])
    e = _t64(bits(w.embed[tok]))
    xn = torch.nn.functional.rms_norm(e, (cfg.hidden,), _t64(bits(w.final_norm)), cfg.rms_eps)
    want = _t64(bits(w.lm_head)) @ xn
    assert np.allclose(logits[0], want.numpy(), rtol=1e-11, atol=1e-12)
    assert nxt[0] == int(torch.argmax(want))


def _rope_complex(x, nh, d, pos, theta):
    x = x.reshape(nh, d)
    a = pos * theta ** (-2.0 * np.arange(d // 2) / d)
    z = (x[:, : d // 2] + 1j * x[:, d // 2:]) * np.exp(1j * a)
    return np.concatenate([z.real, z.imag], axis=1).reshape(-1)


def test_decode_kv_append_layout_rope_and_rounding():
    cfg = small_config(n_layers=1)
    w = make_weights(cfg, seed=4, gain_std=0.1)
    kv = prefilled_kv(cfg, [9], seed=4)
    tok, pos = 77, 9
    _, _, k, v = _run(cfg, w, kv, [tok], [pos])
    d, nq, nkv = cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads
    e = _t64(bits(w.embed[tok]))
    xn = torch.nn.functional.rms_norm(e, (cfg.hidden,), _t64(bits(w.attn_norm[0])), cfg.rms_eps)
    qkv = (_t64(bits(w.wqkv[0])) @ xn).numpy()
    kk = _rope_complex(qkv[nq * d: nq * d + nkv * d], nkv, d, pos, cfg.rope_theta)
    vv = qkv[nq * d + nkv * d:]
    want_k = bits(torch.from_numpy(kk.astype(np.float32)).to(torch.bfloat16)).reshape(nkv, d)
    want_v = bits(torch.from_numpy(vv.astype(np.float32)).to(torch.bfloat16)).reshape(nkv, d)
    # f64 oracle rounds through binary32; allow one bf16 ulp where the two paths straddle a tie
    assert np.max(np.abs(k[0, 0, :, pos].astype(np.int32) - want_k.astype(np.int32))) <= 1
    assert np.mean(k[0, 0, :, pos] == want_k) > 0.98
    assert np.max(np.abs(v[0, 0, :, pos].astype(np.int32) - want_v.astype(np.int32))) <= 1
    # every other position is untouched
    k0, v0 = kv_to_host(kv)
    mask = np.ones(cfg.max_seq, bool)
    mask[pos] = False
    assert np.array_equal(k[..., mask, :], k0[..., mask, :])
    assert np.array_equal(v[..., mask, :], v0[..., mask, :])


def test_decode_uniform_attention_is_mean_over_causal_range():
    """q rows zero -> all scores 0 -> softmax uniform over 0..pos (the new token included).
    Wo is a permutation, the MLP is off: x1 = e + P o, o_h = mean_t V[h // group][t]."""
    cfg = small_config(n_layers=1)
    H, d, nq, nkv = cfg.hidden, cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads
    assert H == nq * d
    w = make_weights(cfg, seed=5)
    w.wqkv[0][: nq * d].zero_()
    perm = torch.randperm(H, generator=torch.Generator().manual_seed(1))
    wo = torch.zeros(H, H)
    wo[torch.arange(H), perm] = 1.0
    w.wo[0].copy_(wo.to(torch.bfloat16))
    w.wgate_up[0].zero_()
    pos = 11
    kv = prefilled_kv(cfg, [pos], seed=5)
    kv.k[0, :, :, pos + 1:] = 1.0e4   # garbage past pos must be ignored
    kv.v[0, :, :, pos + 1:] = 1.0e4
    logits, _, k, v = _run(cfg, w, kv, [42], [pos])
    vals = widen(v[0, 0, :, : pos + 1])            # includes the appended token
    o = np.concatenate([vals[h // (nq // nkv)].mean(axis=0) for h in range(nq)])
    x1 = _t64(bits(w.embed[42])) + torch.from_numpy(o)[perm]
    xn = torch.nn.functional.rms_norm(x1, (H,), _t64(bits(w.final_norm)), cfg.rms_eps)
    want = _t64(bits(w.lm_head)) @ xn
    assert np.allclose(logits[0], want.numpy(), rtol=1e-10, atol=1e-11)


def test_decode_mlp_block_gate_then_up_rows():
    cfg = small_config(n_layers=2)
    w = make_weights(cfg, seed=6, gain_std=0.1)
    for l in range(cfg.n_layers):
        w.wo[l].zero_()
    kv = prefilled_kv(cfg, [3], seed=6)
    logits, _, _, _ = _run(cfg, w, kv, [9], [3])
    F, H = cfg.ffn, cfg.hidden
    x = _t64(bits(w.embed[9]))
    for l in range(cfg.n_layers):
        xn = torch.nn.functional.rms_norm(x, (H,), _t64(bits(w.mlp_norm[l])), cfg.rms_eps)
        gu = _t64(bits(w.wgate_up[l])) @ xn
        x = x + _t64(bits(w.wdown[l])) @ (torch.nn.functional.silu(gu[:F]) * gu[F:])
    xn = torch.nn.functional.rms_norm(x, (H,), _t64(bits(w.final_norm)), cfg.rms_eps)
    want = _t64(bits(w.lm_head)) @ xn
    assert np.allclose(logits[0], want.numpy(), rtol=1e-10, atol=1e-11)


def test_decode_fp32_oracle_within_rounding_of_fp64():
    wl = get_workload("tiny")
    cfg = wl.cfg
    w = make_weights(cfg, seed=0)
    kv = prefilled_kv(cfg, [16], seed=0)
    toks = token_ids(cfg, 1)
    l32, n32, _, _ = _run(cfg, w, kv, toks, [16], "f32")
    l64, n64, _, _ = _run(cfg, w, kv, toks, [16], "f64")
    scale = np.max(np.abs(l64))
    assert np.max(np.abs(l32 - l64)) <= 1e-4 * scale
    top2 = np.sort(l64[0])[-2:]
    if top2[1] - top2[0] > 1e-3:
        assert n32 == n64


def test_decode_batch_sequences_independent():
    cfg = small_config(batch=3, max_seq=20)
    w = make_weights(cfg, seed=7)
    kv = prefilled_kv(cfg, [4, 9, 0], seed=7)
    toks, pos = [5, 6, 7], [4, 9, 0]
    logits, nxt, k, v = _run(cfg, w, kv, toks, pos)
    one = small_config(batch=1, max_seq=20)
    for b in range(3):
        kvb = empty_kv(one)
        kvb.k[0] = kv.k[b]
        kvb.v[0] = kv.v[b]
        lb, nb, kb, vb = _run(one, w, kvb, [toks[b]], [pos[b]])
        assert np.array_equal(lb[0], logits[b]) and nb[0] == nxt[b]
        assert np.array_equal(kb[0], k[b]) and np.array_equal(vb[0], v[b])


def test_swiglu_step_tag_stays_inside_the_parity_tolerance(oracle32, oracle64):
    """The megakernel stores the SwiGLU output in fp32 with its three lowest mantissa bits
    replaced by a step tag (1..7).  Restated here on the oracle's own swiglu outputs: every tagged
    value lies within 2^-20 (relative) of the untagged one, and the change it makes to a
    down-projection row of the 1B shape (8192 inputs, weights ~N(0, 0.02)) is below 1e-5 of the
    row's magnitude -- three orders of magnitude inside the parity tolerance of 1e-2 * max|logit|."""
    rng = np.random.default_rng(5)
    a = rng.normal(0, 2.0, 8192).astype(np.float32)
    u = rng.normal(0, 2.0, 8192).astype(np.float32)
    h = oracle32.swiglu(a, u).astype(np.float32)
    bits = h.view(np.uint32)
    for tag in range(1, 8):
        tagged = ((bits & np.uint32(0xFFFFFFF8)) | np.uint32(tag)).view(np.float32)
        rel = np.abs(tagged.astype(np.float64) - h) / np.maximum(np.abs(h.astype(np.float64)), 1e-30)
        assert rel.max() < 2.0 ** -20
        w = rng.normal(0, 0.02, (4, 8192)).astype(np.float32)
        exact = w.astype(np.float64) @ h.astype(np.float64)
        moved = w.astype(np.float64) @ tagged.astype(np.float64)
        scale = np.abs(w.astype(np.float64)) @ np.abs(h.astype(np.float64))
        assert np.all(np.abs(moved - exact) <= 1e-5 * scale)
    # (the fp64 oracle agrees with the fp32 one far inside the same bound)
    h64 = oracle64.swiglu(a.astype(np.float64), u.astype(np.float64))
    assert np.max(np.abs(h64 - h) / np.maximum(np.abs(h64), 1e-30)) < 2.0 ** -20
