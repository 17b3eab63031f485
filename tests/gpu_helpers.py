"""Shared helpers of the GPU parity tests: build a workload on the device, run the megakernel
and the CPU oracle side by side (teacher-forced: both consume the oracle's token)."""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional

import numpy as np
import torch

from oracle import HostWeights, Oracle, kv_to_host
from workload import KVCache, empty_kv, get_workload, make_weights, prefilled_kv, token_ids

REL_TOL = 1e-2        # max |logit error| <= REL_TOL * max |oracle logit|, per sequence
MARGIN = 0.05         # tokens must agree where the oracle's top-2 margin exceeds this


@dataclass
class Setup:
    cfg: object
    weights: object       # workload.Weights on cuda
    host: HostWeights
    kv: KVCache           # on cuda (the megakernel's cache)
    kh: np.ndarray        # oracle's cache (uint16)
    vh: np.ndarray
    tokens: List[int]
    pos: List[int]


def make_setup(name: str, seed: int = 0, cfg=None, kv_len=None) -> Setup:
    wl = get_workload(name)
    cfg = cfg or wl.cfg
    w = make_weights(cfg, seed=seed, device="cuda")
    hw = HostWeights(w)
    if wl.prompt_len and cfg.batch == 1:
        orc = Oracle("f32")
        kh, vh = kv_to_host(empty_kv(cfg))
        prompt = token_ids(cfg, wl.prompt_len, seed=seed, tag="prompt")
        nxt = None
        for i, t in enumerate(prompt):
            _, nxt = orc.decode_step(cfg, hw, kh, vh, [t], [i])
        kv = empty_kv(cfg, device="cuda")
        kv.k.copy_(torch.from_numpy(kh.view(np.int16)).view(torch.bfloat16))
        kv.v.copy_(torch.from_numpy(vh.view(np.int16)).view(torch.bfloat16))
        return Setup(cfg, w, hw, kv, kh, vh, list(nxt), [wl.prompt_len])
    lens = list(kv_len if kv_len is not None else wl.kv_len)
    kv = prefilled_kv(cfg, lens, seed=seed, device="cuda")
    kh, vh = kv_to_host(kv)
    toks = token_ids(cfg, cfg.batch, seed=seed, tag="first")
    return Setup(cfg, w, hw, kv, kh, vh, toks, lens)


def compare_step(g_logits: np.ndarray, o_logits: np.ndarray, g_next: List[int], o_next: List[int]) -> Dict:
    out = {"max_err": 0.0, "rel": 0.0, "token_checked": 0, "token_mismatch": []}
    for b in range(o_logits.shape[0]):
        err = float(np.max(np.abs(g_logits[b].astype(np.float64) - o_logits[b])))
        scale = float(np.max(np.abs(o_logits[b])))
        out["max_err"] = max(out["max_err"], err)
        out["rel"] = max(out["rel"], err / scale)
        top = np.sort(o_logits[b])[-2:]
        if top[1] - top[0] > MARGIN:
            out["token_checked"] += 1
            if g_next[b] != o_next[b]:
                out["token_mismatch"].append((b, g_next[b], o_next[b]))
    return out


def run_parity(s: Setup, dec, steps: int, oracle: Optional[Oracle] = None, check_every: int = 1) -> Dict:
    """Runs `steps` teacher-forced steps; returns the worst relative error and token stats."""
    orc = oracle or Oracle("f32")
    tokens, pos = list(s.tokens), list(s.pos)
    worst = {"rel": 0.0, "token_checked": 0, "token_mismatch": [], "steps": 0}
    for i in range(steps):
        g_next = dec.step(tokens, pos)
        o_logits, o_next = orc.decode_step(s.cfg, s.host, s.kh, s.vh, tokens, pos)
        if i % check_every == 0 or i == steps - 1:
            r = compare_step(dec.logits.cpu().numpy(), o_logits, g_next, o_next)
            worst["rel"] = max(worst["rel"], r["rel"])
            worst["token_checked"] += r["token_checked"]
            worst["token_mismatch"] += r["token_mismatch"]
        worst["steps"] += 1
        tokens = list(o_next)
        pos = [p + 1 for p in pos]
    worst["final_pos"] = pos
    return worst


def kv_agreement(s: Setup, positions_per_seq: List[List[int]]) -> Dict:
    """Compares the megakernel's appended K/V with the oracle's.  Both round an fp32 value to
    bf16, but the fp32 sums behind them are ordered differently, so a value may land one bf16
    step apart; near zero (cancellation) a step is tiny in absolute terms.  Reports the fraction
    of identical codes and the worst |difference| in units of (one bf16 step at the value's
    magnitude + 1e-3 * the head vector's RMS)."""
    k = s.kv.k.cpu().float().numpy()
    v = s.kv.v.cpu().float().numpy()
    kh = (s.kh.astype(np.uint32) << 16).view(np.float32)
    vh = (s.vh.astype(np.uint32) << 16).view(np.float32)
    worst, n, same = 0.0, 0, 0
    for b, ps in enumerate(positions_per_seq):
        for p in ps:
            for a, r in ((k, kh), (v, vh)):
                ga, ra = a[b, :, :, p].astype(np.float64), r[b, :, :, p].astype(np.float64)
                rms = np.sqrt(np.mean(ra * ra, axis=-1, keepdims=True))
                step = 2.0 ** -7 * np.maximum(np.abs(ga), np.abs(ra)) + 1e-3 * rms
                worst = max(worst, float(np.max(np.abs(ga - ra) / step)))
                n += ga.size
                same += int(np.sum(ga == ra))
    return {"worst_in_steps": worst, "frac_equal": same / max(n, 1)}
