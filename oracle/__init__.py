"""ORACLE -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` import
this package.  The library's product path never does, and this package imports nothing from
the library.

* ``Oracle``       ctypes front end of ``oracle.c`` (plain fp32 / fp64 CPU decode step and its
                   building blocks), built with gcc by ``build()``.
* ``schedule_ref`` an independent restatement of the tile scheduler, the schedule validator and
                   a host simulator of the per-SM queue interpreter.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (OpenMP when available)."""
    src = os.path.join(_HERE, "oracle.c")
    dep = [src, os.path.join(_HERE, "oracle_impl.h")]
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(p) for p in dep)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-shared", "-fPIC", "-std=c11", src, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:2] + ["-fopenmp"] + base[2:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
                 "batch", "max_seq")] + [("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double)]


_P = ctypes.c_void_p


class _W(ctypes.Structure):
    _fields_ = [("embed", _P), ("lm_head", _P), ("final_norm", _P), ("attn_norm", _P),
                ("wqkv", _P), ("wo", _P), ("mlp_norm", _P), ("wgate_up", _P), ("wdown", _P)]


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_LIB_PATH)
        for pfx in ("or_f32_", "or_f64_"):
            real = ctypes.c_float if pfx == "or_f32_" else ctypes.c_double
            getattr(_lib, pfx + "bf16_round").restype = ctypes.c_uint16
            getattr(_lib, pfx + "bf16_round").argtypes = [real]
            getattr(_lib, pfx + "silu").restype = real
            getattr(_lib, pfx + "silu").argtypes = [real]
            getattr(_lib, pfx + "argmax").restype = ctypes.c_int
            getattr(_lib, pfx + "argmax").argtypes = [_P, ctypes.c_int]
            getattr(_lib, pfx + "rmsnorm").argtypes = [_P, _P, ctypes.c_int, ctypes.c_double, _P]
            getattr(_lib, pfx + "matvec").argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, _P]
            getattr(_lib, pfx + "rope").argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_double]
            getattr(_lib, pfx + "attention").argtypes = [_P, _P, _P] + [ctypes.c_int] * 5 + [_P, _P]
            getattr(_lib, pfx + "swiglu").argtypes = [_P, _P, ctypes.c_int, _P]
            getattr(_lib, pfx + "decode_step").restype = ctypes.c_int
            getattr(_lib, pfx + "decode_step").argtypes = [ctypes.POINTER(_Cfg), ctypes.POINTER(_W),
                                                           _P, _P, _P, _P, _P, _P]
        _lib.or_set_threads.restype = ctypes.c_int
        _lib.or_set_threads.argtypes = [ctypes.c_int]
    return _lib


def set_threads(n: int = 0) -> int:
    """Set (n > 0) and return the number of host threads the oracle uses."""
    return _load().or_set_threads(n)


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (CPU) -> contiguous uint16 numpy view of its bit patterns."""
    assert t.dtype == torch.bfloat16
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16)


class Oracle:
    """fp32 (``precision='f32'``) or fp64 (``'f64'``) oracle."""

    def __init__(self, precision: str = "f32"):
        assert precision in ("f32", "f64")
        self.lib = _load()
        self.pfx = "or_" + precision + "_"
        self.dtype = np.float32 if precision == "f32" else np.float64

    def _f(self, name):
        return getattr(self.lib, self.pfx + name)

    def _arr(self, x) -> np.ndarray:
        return np.ascontiguousarray(np.asarray(x, dtype=self.dtype))

    # ---- building blocks ------------------------------------------------------------
    def bf16_round(self, v: float) -> int:
        return int(self._f("bf16_round")(float(v)))

    def rmsnorm(self, x, gain_bf16: np.ndarray, eps: float) -> np.ndarray:
        x = self._arr(x)
        g = np.ascontiguousarray(gain_bf16, dtype=np.uint16)
        out = np.empty_like(x)
        self._f("rmsnorm")(_ptr(x), _ptr(g), x.size, eps, _ptr(out))
        return out

    def matvec(self, w_bf16: np.ndarray, x) -> np.ndarray:
        w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
        x = self._arr(x)
        rows, cols = w.shape
        assert cols == x.size
        y = np.empty(rows, dtype=self.dtype)
        self._f("matvec")(_ptr(w), rows, cols, _ptr(x), _ptr(y))
        return y

    def rope(self, v, n_heads: int, d: int, pos: int, theta: float) -> np.ndarray:
        v = self._arr(v).copy()
        self._f("rope")(_ptr(v), n_heads, d, pos, theta)
        return v

    def attention(self, q, kc: np.ndarray, vc: np.ndarray, nq: int, nkv: int, d: int,
                  max_seq: int, pos: int, want_probs: bool = False):
        q = self._arr(q)
        kc = np.ascontiguousarray(kc, dtype=np.uint16)
        vc = np.ascontiguousarray(vc, dtype=np.uint16)
        out = np.empty(nq * d, dtype=self.dtype)
        probs = np.empty(nq * (pos + 1), dtype=self.dtype) if want_probs else None
        self._f("attention")(_ptr(q), _ptr(kc), _ptr(vc), nq, nkv, d, max_seq, pos, _ptr(out),
                             _ptr(probs) if probs is not None else None)
        return (out, probs.reshape(nq, pos + 1)) if want_probs else out

    def silu(self, z: float) -> float:
        return float(self._f("silu")(float(z)))

    def swiglu(self, a, u) -> np.ndarray:
        a, u = self._arr(a), self._arr(u)
        out = np.empty_like(a)
        self._f("swiglu")(_ptr(a), _ptr(u), a.size, _ptr(out))
        return out

    def argmax(self, v) -> int:
        v = self._arr(v)
        return int(self._f("argmax")(_ptr(v), v.size))

    # ---- whole decode step ----------------------------------------------------------
    def decode_step(self, cfg, weights, kv_k: np.ndarray, kv_v: np.ndarray,
                    tokens: Sequence[int], pos: Sequence[int]) -> Tuple[np.ndarray, List[int]]:
        """One step for every sequence.  ``weights`` is a HostWeights; kv_k / kv_v are uint16
        arrays [B, L, nkv, max_seq, d] updated in place at pos.  Returns (logits [B, V], next)."""
        c = _Cfg(cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn,
                 cfg.vocab, cfg.batch, cfg.max_seq, float(cfg.rms_eps), float(cfg.rope_theta))
        assert kv_k.dtype == np.uint16 and kv_k.flags["C_CONTIGUOUS"] and kv_v.flags["C_CONTIGUOUS"]
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        ps = np.ascontiguousarray(pos, dtype=np.int32)
        assert tok.size == cfg.batch and ps.size == cfg.batch
        logits = np.empty((cfg.batch, cfg.vocab), dtype=self.dtype)
        nxt = np.empty(cfg.batch, dtype=np.int32)
        rc = self._f("decode_step")(ctypes.byref(c), ctypes.byref(weights.cstruct), _ptr(kv_k),
                                    _ptr(kv_v), _ptr(tok), _ptr(ps), _ptr(logits), _ptr(nxt))
        if rc != 0:
            raise ValueError("oracle decode_step rejected its arguments")
        return logits, [int(t) for t in nxt]


class HostWeights:
    """Host (uint16) copies of a workload.Weights, kept alive for the C structure."""

    def __init__(self, w):
        self.embed = _u16(w.embed)
        self.lm_head = self.embed if w.lm_head is w.embed else _u16(w.lm_head)
        self.final_norm = _u16(w.final_norm)
        self.layers = {k: [_u16(t) for t in getattr(w, k)]
                       for k in ("attn_norm", "wqkv", "wo", "mlp_norm", "wgate_up", "wdown")}
        self._tables = {k: (ctypes.c_void_p * len(v))(*[_ptr(a) for a in v])
                        for k, v in self.layers.items()}
        self.cstruct = _W(_ptr(self.embed), _ptr(self.lm_head), _ptr(self.final_norm),
                          *[ctypes.cast(self._tables[k], ctypes.c_void_p)
                            for k in ("attn_norm", "wqkv", "wo", "mlp_norm", "wgate_up", "wdown")])


def kv_to_host(kv) -> Tuple[np.ndarray, np.ndarray]:
    """workload.KVCache -> (k, v) uint16 numpy arrays (copies)."""
    return _u16(kv.k).copy(), _u16(kv.v).copy()
