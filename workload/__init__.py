"""Seeded synthetic workloads for the decode megakernel and its oracle.

This module is the only code that both sides share. It holds the model
configurations (plain numbers) and seeded generators of weights, KV-cache
contents and token ids. It holds none of the decoder's arithmetic: no norm, no
projection, no attention, no scheduling.

Shapes and value distributions follow the workloads named in the
"Inference MegaKernel" page (section "Hand-written whole-model MegaKernel":
a Llama-3.2-1B-shaped decoder at batch 1), widened to the five configurations
this library is tested on:

* ``tiny``          2 layers, hidden 256, 4 Q / 2 KV heads, head_dim 64, FFN 688,
                    vocab 4096; a 16-token random prompt prefilled by the oracle,
                    then 8 greedy decode steps.
* ``llama1b_ctx512``  Llama-3.2-1B shape (16 layers, hidden 2048, 32 Q / 8 KV
                    heads, head_dim 64, FFN 8192, vocab 128256, tied embeddings,
                    RoPE theta 500000); KV prefilled to 512 positions; 128 steps.
* ``llama1b_ctx8192`` same shape, KV prefilled to 8192 positions; 64 steps.
* ``llama1b_batch8``  same shape, 8 sequences with KV lengths uniform in
                    [256, 4096]; 64 steps.
* ``llama8b_ctx2048`` Llama-3.1-8B shape (32 layers, hidden 4096, head_dim 128,
                    FFN 14336, untied LM head); KV prefilled to 2048; 64 steps.

Two profiling cases (not benchmark lines) keep the 1B layer shapes with 2 layers
and vocab 32000: ``llama1b_reduced`` (batch 1, KV 512) and
``llama1b_reduced_batch8`` (the batch-8 KV lengths).

Value recipe: every matrix ~ N(0, 0.02) rounded to bf16 (round to nearest
even); every RMSNorm gain = 1.0; prefilled K/V ~ N(0, 1) rounded to bf16 and
taken as already-rotated cache contents; token ids uniform in [0, vocab).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch


@dataclass(frozen=True)
class ModelConfig:
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    tied_embeddings: bool
    batch: int
    max_seq: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def qkv_rows(self) -> int:
        return self.q_dim + 2 * self.kv_dim

    def weight_bytes(self) -> int:
        """bf16 bytes of every weight one decode step reads (norm gains included)."""
        L, H, F, V = self.n_layers, self.hidden, self.ffn, self.vocab
        per_layer = self.qkv_rows * H + H * self.q_dim + 2 * F * H + H * F + 2 * H
        return 2 * (L * per_layer + V * H + H)

    def kv_bytes(self, pos: List[int]) -> int:
        """KV-cache bytes one step moves: read positions 0..pos, write position pos."""
        per_pos = self.n_layers * 2 * self.kv_dim * 2
        return sum(per_pos * (p + 1) for p in pos) + per_pos * len(pos)

    def step_bytes(self, pos: List[int]) -> int:
        return self.weight_bytes() + self.kv_bytes(pos)


@dataclass(frozen=True)
class Workload:
    name: str
    cfg: ModelConfig
    prompt_len: int          # tiny: prompt tokens prefilled by the oracle; else 0
    kv_len: List[int]        # per sequence: positions already in the cache at step 0
    decode_steps: int
    seed: int = 0
    description: str = ""


def _kv_lengths_batch8(seed: int) -> List[int]:
    g = torch.Generator().manual_seed(seed + 7919)
    return [int(v) for v in torch.randint(256, 4097, (8,), generator=g)]


def get_workload(name: str) -> Workload:
    if name == "tiny":
        cfg = ModelConfig(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                          ffn=688, vocab=4096, tied_embeddings=True, batch=1,
                          max_seq=16 + 8, rms_eps=1e-5, rope_theta=10000.0)
        return Workload(name, cfg, prompt_len=16, kv_len=[16], decode_steps=8,
                        description="tiny Llama-style decoder, 16-token prompt, 8 greedy steps")
    if name == "llama1b_ctx512":
        cfg = _llama1b(batch=1, max_seq=512 + 128)
        return Workload(name, cfg, prompt_len=0, kv_len=[512], decode_steps=128,
                        description="Llama-3.2-1B shape, batch 1, KV 512, 128 steps")
    if name == "llama1b_ctx8192":
        cfg = _llama1b(batch=1, max_seq=8192 + 64)
        return Workload(name, cfg, prompt_len=0, kv_len=[8192], decode_steps=64,
                        description="Llama-3.2-1B shape, batch 1, KV 8192, 64 steps")
    if name == "llama1b_batch8":
        lens = _kv_lengths_batch8(0)
        cfg = _llama1b(batch=8, max_seq=4096 + 64)
        return Workload(name, cfg, prompt_len=0, kv_len=lens, decode_steps=64,
                        description="Llama-3.2-1B shape, batch 8, KV U[256,4096], 64 steps")
    if name == "llama1b_reduced":
        # profiling case (not a benchmark line): Llama-3.2-1B layer shapes, 2 layers, vocab 32000;
        # ~380 MB of weights, larger than L2, small enough for many-pass profiler captures
        cfg = ModelConfig(n_layers=2, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=64, ffn=8192,
                          vocab=32000, tied_embeddings=True, batch=1, max_seq=512 + 128, rms_eps=1e-5,
                          rope_theta=500000.0)
        return Workload(name, cfg, prompt_len=0, kv_len=[512], decode_steps=128,
                        description="reduced Llama-3.2-1B shape for profiling: 2 layers, vocab 32000")
    if name == "llama1b_reduced_batch8":
        # profiling case (not a benchmark line): the batch-8 workload's shapes and KV lengths with 2
        # layers and vocab 32000 (~520 MB of weights and KV cache on the device)
        lens = _kv_lengths_batch8(0)
        cfg = ModelConfig(n_layers=2, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=64, ffn=8192,
                          vocab=32000, tied_embeddings=True, batch=8, max_seq=4096 + 64, rms_eps=1e-5,
                          rope_theta=500000.0)
        return Workload(name, cfg, prompt_len=0, kv_len=lens, decode_steps=64,
                        description="reduced batch-8 Llama-3.2-1B shape for profiling: 2 layers, vocab 32000")
    if name == "llama8b_ctx2048":
        cfg = ModelConfig(n_layers=32, hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
                          ffn=14336, vocab=128256, tied_embeddings=False, batch=1,
                          max_seq=2048 + 64, rms_eps=1e-5, rope_theta=500000.0)
        return Workload(name, cfg, prompt_len=0, kv_len=[2048], decode_steps=64,
                        description="Llama-3.1-8B shape, batch 1, KV 2048, 64 steps")
    raise KeyError(name)


def _llama1b(batch: int, max_seq: int) -> ModelConfig:
    return ModelConfig(n_layers=16, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=64,
                       ffn=8192, vocab=128256, tied_embeddings=True, batch=batch,
                       max_seq=max_seq, rms_eps=1e-5, rope_theta=500000.0)


WORKLOADS = ["tiny", "llama1b_ctx512", "llama1b_ctx8192", "llama1b_batch8", "llama8b_ctx2048"]


def small_config(**over) -> ModelConfig:
    """A configurable small shape for unit tests (defaults: the tiny decoder)."""
    base = dict(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=688,
                vocab=4096, tied_embeddings=True, batch=1, max_seq=24, rms_eps=1e-5,
                rope_theta=10000.0)
    base.update(over)
    return ModelConfig(**base)


# --------------------------------------------------------------------------------------
# Seeded tensors.  Every tensor gets its own generator stream derived from (seed, tag), so
# shapes can be generated in any order and on any device.
# --------------------------------------------------------------------------------------

def _stream_seed(seed: int, tag: str) -> int:
    h = 1469598103934665603
    for ch in f"{seed}:{tag}".encode():
        h = ((h ^ ch) * 1099511628211) & 0xFFFFFFFFFFFFFFFF
    return h & 0x7FFFFFFFFFFFFFFF


def _normal_bf16(shape, std: float, seed: int, tag: str, device) -> torch.Tensor:
    g = torch.Generator(device=device).manual_seed(_stream_seed(seed, tag))
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


@dataclass
class Weights:
    """Decoder weights, bf16, row-major, in the layouts the library documents.

    wqkv[l]     [(nq + 2 nkv) d, H]   rows: q heads, then k heads, then v heads
    wo[l]       [H, nq d]
    wgate_up[l] [2F, H]               rows: gate (F rows), then up (F rows)
    wdown[l]    [H, F]
    embed       [V, H]; lm_head is embed itself when tied.
    """
    embed: torch.Tensor
    lm_head: torch.Tensor
    final_norm: torch.Tensor
    attn_norm: List[torch.Tensor]
    wqkv: List[torch.Tensor]
    wo: List[torch.Tensor]
    mlp_norm: List[torch.Tensor]
    wgate_up: List[torch.Tensor]
    wdown: List[torch.Tensor]

    def to(self, device) -> "Weights":
        f = lambda t: t.to(device)
        emb = f(self.embed)
        lm = emb if self.lm_head is self.embed else f(self.lm_head)
        return Weights(emb, lm, f(self.final_norm), [f(t) for t in self.attn_norm],
                       [f(t) for t in self.wqkv], [f(t) for t in self.wo],
                       [f(t) for t in self.mlp_norm], [f(t) for t in self.wgate_up],
                       [f(t) for t in self.wdown])

    @property
    def tied(self) -> bool:
        return self.lm_head is self.embed


def make_weights(cfg: ModelConfig, seed: int = 0, device="cpu", std: float = 0.02,
                 gain_std: float = 0.0) -> Weights:
    """Seeded weights. Gains are 1.0 (or 1 + N(0, gain_std) when a test asks for it)."""
    H, F, V = cfg.hidden, cfg.ffn, cfg.vocab

    def gain(tag):
        if gain_std == 0.0:
            return torch.ones(H, dtype=torch.bfloat16, device=device)
        return (1.0 + _normal_bf16((H,), gain_std, seed, tag, device).float()).to(torch.bfloat16)

    embed = _normal_bf16((V, H), std, seed, "embed", device)
    lm = embed if cfg.tied_embeddings else _normal_bf16((V, H), std, seed, "lm_head", device)
    L = cfg.n_layers
    return Weights(
        embed=embed, lm_head=lm, final_norm=gain("final_norm"),
        attn_norm=[gain(f"attn_norm{l}") for l in range(L)],
        wqkv=[_normal_bf16((cfg.qkv_rows, H), std, seed, f"wqkv{l}", device) for l in range(L)],
        wo=[_normal_bf16((H, cfg.q_dim), std, seed, f"wo{l}", device) for l in range(L)],
        mlp_norm=[gain(f"mlp_norm{l}") for l in range(L)],
        wgate_up=[_normal_bf16((2 * F, H), std, seed, f"wgu{l}", device) for l in range(L)],
        wdown=[_normal_bf16((H, F), std, seed, f"wdown{l}", device) for l in range(L)],
    )


@dataclass
class KVCache:
    """K and V caches, bf16, shape [B, L, n_kv_heads, max_seq, head_dim] each."""
    k: torch.Tensor
    v: torch.Tensor

    def clone(self) -> "KVCache":
        return KVCache(self.k.clone(), self.v.clone())

    def to(self, device) -> "KVCache":
        return KVCache(self.k.to(device), self.v.to(device))


def empty_kv(cfg: ModelConfig, device="cpu") -> KVCache:
    shape = (cfg.batch, cfg.n_layers, cfg.n_kv_heads, cfg.max_seq, cfg.head_dim)
    return KVCache(torch.zeros(shape, dtype=torch.bfloat16, device=device),
                   torch.zeros(shape, dtype=torch.bfloat16, device=device))


def prefilled_kv(cfg: ModelConfig, kv_len: List[int], seed: int = 0, device="cpu") -> KVCache:
    """Positions [0, kv_len[b]) of sequence b hold N(0,1) bf16 values; the rest are zero."""
    kv = empty_kv(cfg, device)
    for b, n in enumerate(kv_len):
        if n == 0:
            continue
        shape = (cfg.n_layers, cfg.n_kv_heads, n, cfg.head_dim)
        kv.k[b, :, :, :n] = _normal_bf16(shape, 1.0, seed, f"kcache{b}", device)
        kv.v[b, :, :, :n] = _normal_bf16(shape, 1.0, seed, f"vcache{b}", device)
    return kv


def token_ids(cfg: ModelConfig, n: int, seed: int = 0, tag: str = "tokens") -> List[int]:
    g = torch.Generator().manual_seed(_stream_seed(seed, tag))
    return [int(t) for t in torch.randint(0, cfg.vocab, (n,), generator=g)]


def config_dict(cfg: ModelConfig) -> Dict:
    return dataclasses.asdict(cfg)
