"""Python binding of the persistent decode megakernel's C ABI (include/mk.h).

Argument marshalling only: every step of the decode runs in the CUDA kernels of libmk.so.
PyTorch supplies device memory and the stream.  There is no fallback: if libmk.so is missing
or fails to load, importing this package raises.

Low level: the mk_* functions of the C ABI under the same names (``lib.mk_bind`` ...).
High level:
    sched = Schedule(cfg, sm_count)               # mk_build_schedule
    dec = Decoder(sched, weights, kv)             # allocates counters/scratch with torch, mk_bind
    nxt = dec.step(tokens, pos, logits)           # mk_decode_step (synchronous)
    dec.launch(tokens, pos, logits, next_dev)     # mk_launch_step (asynchronous)
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmk.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
lib = ctypes.CDLL(LIB_PATH)

MK_OK, MK_ERR_ARG, MK_ERR_CAPACITY, MK_ERR_RESOURCES, MK_ERR_CUDA, MK_ERR_TIMEOUT, MK_ERR_OPCODE, \
    MK_ERR_BOUNDS, MK_ERR_POISONED = range(9)
STATUS_NAMES = ["MK_OK", "MK_ERR_ARG", "MK_ERR_CAPACITY", "MK_ERR_RESOURCES", "MK_ERR_CUDA", "MK_ERR_TIMEOUT",
                "MK_ERR_OPCODE", "MK_ERR_BOUNDS", "MK_ERR_POISONED"]
SYNC_TAGS, SYNC_COUNTERS = 0, 1   # mk_sync_mode

EXPORTS = ["mk_build_schedule", "mk_schedule_queues", "mk_schedule_counters", "mk_schedule_patch",
           "mk_scratch_bytes", "mk_schedule_free", "mk_bind", "mk_set_timeout", "mk_decode_step",
           "mk_launch_step", "mk_ctx_status", "mk_device_sm_count", "mk_last_error", "mk_unbind", "mk_set_trace",
           "mk_decode_step_static", "mk_set_sync", "mk_decode_steps", "mk_bind_paged", "mk_schedule_attn_chunk",
           "mk_decode_persistent_start", "mk_decode_persistent_stop", "mk_decode_persistent_progress",
           "mk_decode_persistent_wait", "mk_rebind_schedule"]


class MkError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES[status] if 0 <= status < 9 else status}: {msg}")
        self.status = status


class mk_model_cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim",
                                              "ffn", "vocab", "tied_embeddings", "batch", "max_seq")] + \
               [("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double)]


class mk_sched_opts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("page_bytes", "tile_bytes", "attn_chunk", "rows_qkv", "rows_o",
                                              "pairs_up", "rows_down", "rows_lm")] + \
               [("shuffle_seed", ctypes.c_uint64), ("kv_limit", ctypes.c_int32 * 8)]


_P = ctypes.c_void_p


class mk_weights(ctypes.Structure):
    _fields_ = [("embed", _P), ("lm_head", _P), ("final_norm", _P), ("attn_norm", _P), ("wqkv", _P),
                ("wo", _P), ("mlp_norm", _P), ("wgate_up", _P), ("wdown", _P)]


class mk_kv(ctypes.Structure):
    _fields_ = [("k", _P), ("v", _P), ("batch_stride", ctypes.c_int64), ("layer_stride", ctypes.c_int64),
                ("head_stride", ctypes.c_int64)]


class mk_kv_pages(ctypes.Structure):
    _fields_ = [("block_table", _P), ("block_size", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("n_blocks", ctypes.c_int32)]


_I32P = ctypes.POINTER(ctypes.c_int32)
lib.mk_build_schedule.restype = ctypes.c_int
lib.mk_build_schedule.argtypes = [ctypes.POINTER(mk_model_cfg), ctypes.c_int32, ctypes.POINTER(mk_sched_opts),
                                  ctypes.POINTER(_P)]
lib.mk_schedule_queues.restype = ctypes.c_int
lib.mk_schedule_queues.argtypes = [_P, ctypes.POINTER(_I32P), _I32P, _I32P]
lib.mk_schedule_counters.restype = ctypes.c_int
lib.mk_schedule_counters.argtypes = [_P, ctypes.POINTER(ctypes.POINTER(ctypes.c_uint32)), _I32P]
lib.mk_schedule_attn_chunk.restype = ctypes.c_int
lib.mk_schedule_attn_chunk.argtypes = [_P, _I32P]
lib.mk_schedule_patch.restype = ctypes.c_int
lib.mk_schedule_patch.argtypes = [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
lib.mk_scratch_bytes.restype = ctypes.c_size_t
lib.mk_scratch_bytes.argtypes = [_P]
lib.mk_schedule_free.restype = None
lib.mk_schedule_free.argtypes = [_P]
lib.mk_bind.restype = ctypes.c_int
lib.mk_bind.argtypes = [_P, ctypes.POINTER(mk_weights), ctypes.POINTER(mk_kv), _P, _P, _P, ctypes.POINTER(_P)]
lib.mk_bind_paged.restype = ctypes.c_int
lib.mk_bind_paged.argtypes = [_P, ctypes.POINTER(mk_weights), ctypes.POINTER(mk_kv), ctypes.POINTER(mk_kv_pages), _P,
                              _P, _P, ctypes.POINTER(_P)]
lib.mk_set_timeout.restype = ctypes.c_int
lib.mk_set_timeout.argtypes = [_P, ctypes.c_uint64]
lib.mk_decode_step.restype = ctypes.c_int
lib.mk_decode_step.argtypes = [_P, _I32P, _I32P, _P, _I32P]
lib.mk_launch_step.restype = ctypes.c_int
lib.mk_launch_step.argtypes = [_P, _I32P, _I32P, _P, _P]
lib.mk_decode_steps.restype = ctypes.c_int
lib.mk_decode_steps.argtypes = [_P, _I32P, _I32P, ctypes.c_int32, _P, _P, _I32P]
lib.mk_decode_persistent_start.restype = ctypes.c_int
lib.mk_decode_persistent_start.argtypes = [_P, _I32P, _I32P, ctypes.c_int32, _P, _P]
lib.mk_decode_persistent_stop.restype = ctypes.c_int
lib.mk_decode_persistent_stop.argtypes = [_P]
lib.mk_decode_persistent_progress.restype = ctypes.c_int
lib.mk_decode_persistent_progress.argtypes = [_P, _I32P]
lib.mk_decode_persistent_wait.restype = ctypes.c_int
lib.mk_decode_persistent_wait.argtypes = [_P, _I32P, _I32P]
lib.mk_rebind_schedule.restype = ctypes.c_int
lib.mk_rebind_schedule.argtypes = [_P, _P]
lib.mk_ctx_status.restype = ctypes.c_int
lib.mk_ctx_status.argtypes = [_P, _I32P]
lib.mk_device_sm_count.restype = ctypes.c_int
lib.mk_device_sm_count.argtypes = [_I32P]
lib.mk_last_error.restype = ctypes.c_char_p
lib.mk_last_error.argtypes = []
lib.mk_decode_step_static.restype = ctypes.c_int
lib.mk_decode_step_static.argtypes = [_P, _I32P, _I32P, _P, _I32P]
lib.mk_set_trace.restype = ctypes.c_int
lib.mk_set_trace.argtypes = [_P, _P]
lib.mk_set_sync.restype = ctypes.c_int
lib.mk_set_sync.argtypes = [_P, ctypes.c_int32]
lib.mk_unbind.restype = None
lib.mk_unbind.argtypes = [_P]


def _check(st: int):
    if st != MK_OK:
        raise MkError(st, lib.mk_last_error().decode(errors="replace"))


def make_cfg(cfg) -> mk_model_cfg:
    """workload.ModelConfig (or any object with the same fields) -> mk_model_cfg."""
    return mk_model_cfg(cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn, cfg.vocab,
                        int(cfg.tied_embeddings), cfg.batch, cfg.max_seq, float(cfg.rms_eps), float(cfg.rope_theta))


def device_sm_count() -> int:
    n = ctypes.c_int32()
    _check(lib.mk_device_sm_count(ctypes.byref(n)))
    return n.value


class Schedule:
    """Host schedule object (mk_build_schedule); frees itself."""

    def __init__(self, cfg, sm_count: int, page_bytes: int = 0, tile_bytes: int = 0, attn_chunk: int = 0,
                 rows_qkv: int = 0, rows_o: int = 0, pairs_up: int = 0, rows_down: int = 0, rows_lm: int = 0,
                 shuffle_seed: int = 0, kv_limit: Optional[Sequence[int]] = None):
        self.cfg = cfg
        self._c = make_cfg(cfg)
        lim = list(kv_limit or []) + [0] * (8 - len(kv_limit or []))
        o = mk_sched_opts(page_bytes, tile_bytes, attn_chunk, rows_qkv, rows_o, pairs_up, rows_down, rows_lm,
                          shuffle_seed, (ctypes.c_int32 * 8)(*lim))
        h = _P()
        _check(lib.mk_build_schedule(ctypes.byref(self._c), int(sm_count), ctypes.byref(o), ctypes.byref(h)))
        self.handle = h

    def __del__(self):
        if getattr(self, "handle", None):
            lib.mk_schedule_free(self.handle)
            self.handle = None

    def queues(self) -> np.ndarray:
        q, S, Q = _I32P(), ctypes.c_int32(), ctypes.c_int32()
        _check(lib.mk_schedule_queues(self.handle, ctypes.byref(q), ctypes.byref(S), ctypes.byref(Q)))
        return np.ctypeslib.as_array(q, shape=(S.value, Q.value, 32)).copy()

    def totals(self) -> np.ndarray:
        t, n = ctypes.POINTER(ctypes.c_uint32)(), ctypes.c_int32()
        _check(lib.mk_schedule_counters(self.handle, ctypes.byref(t), ctypes.byref(n)))
        return np.ctypeslib.as_array(t, shape=(n.value,)).copy()

    @property
    def n_counters(self) -> int:
        return int(self.totals().size)

    @property
    def attn_chunk(self) -> int:
        """KV positions per split-K attention tile (the block size of a paged KV cache)."""
        v = ctypes.c_int32()
        _check(lib.mk_schedule_attn_chunk(self.handle, ctypes.byref(v)))
        return v.value

    @property
    def scratch_bytes(self) -> int:
        return int(lib.mk_scratch_bytes(self.handle))

    def patch(self, sm: int, slot: int, word: int, value: int):
        _check(lib.mk_schedule_patch(self.handle, sm, slot, word, value))


def _ptr(t) -> int:
    return t.data_ptr()


class Decoder:
    """A bound context: borrows the weights / KV tensors, owns counters, scratch and logits (torch).

    ``pages`` (optional) binds a paged KV cache: a tuple (block_table, block_size, n_blocks) with
    block_table a CUDA int32 tensor [batch, max_blocks]; kv.k / kv.v are then the block pools,
    shaped [n_layers, n_kv_heads, n_blocks * block_size, head_dim].  ``scratch`` (optional) is the
    caller's device scratch (at least ``sched.scratch_bytes`` bytes, 256-byte aligned); by default
    one is allocated."""

    def __init__(self, sched: Schedule, weights, kv, stream=None, timeout_ns: Optional[int] = None, pages=None,
                 scratch=None):
        import torch
        cfg = sched.cfg
        dev = weights.embed.device
        assert dev.type == "cuda", "weights must be CUDA tensors"
        self.cfg, self.sched, self.weights, self.kv = cfg, sched, weights, kv
        L = cfg.n_layers
        self._tabs = {k: (_P * L)(*[_ptr(t) for t in getattr(weights, k)])
                      for k in ("attn_norm", "wqkv", "wo", "mlp_norm", "wgate_up", "wdown")}
        self._w = mk_weights(_ptr(weights.embed), _ptr(weights.lm_head), _ptr(weights.final_norm),
                             *[ctypes.cast(self._tabs[k], _P)
                               for k in ("attn_norm", "wqkv", "wo", "mlp_norm", "wgate_up", "wdown")])
        for t in (kv.k, kv.v):
            assert t.is_contiguous() and t.dtype == torch.bfloat16 and t.device == dev
        st = kv.k.stride()
        if pages is None:
            self._kv = mk_kv(_ptr(kv.k), _ptr(kv.v), st[0], st[1], st[2])
            self._pages = None
        else:
            table, block_size, n_blocks = pages
            assert table.dtype == torch.int32 and table.device == dev and table.is_contiguous()
            self._kv = mk_kv(_ptr(kv.k), _ptr(kv.v), 0, st[0], st[1])
            self._pages = mk_kv_pages(_ptr(table), int(block_size), int(table.shape[-1]), int(n_blocks))
            self._table = table
        self.counters = torch.zeros(sched.n_counters, dtype=torch.int32, device=dev)
        if scratch is None:
            scratch = torch.empty(sched.scratch_bytes // 4 + 64, dtype=torch.int32, device=dev)
        assert scratch.device == dev and scratch.numel() * scratch.element_size() >= sched.scratch_bytes
        self.scratch = scratch
        self.logits = torch.empty((cfg.batch, cfg.vocab), dtype=torch.float32, device=dev)
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)
        h = _P()
        _check(lib.mk_bind_paged(sched.handle, ctypes.byref(self._w), ctypes.byref(self._kv),
                                 ctypes.byref(self._pages) if self._pages is not None else None, _ptr(self.counters),
                                 _ptr(self.scratch), ctypes.c_void_p(self.stream.cuda_stream), ctypes.byref(h)))
        self.handle = h
        if timeout_ns is not None:
            self.set_timeout(timeout_ns)

    def close(self):
        if getattr(self, "handle", None):
            lib.mk_unbind(self.handle)
            self.handle = None

    def __del__(self):
        self.close()

    def set_timeout(self, ns: int):
        _check(lib.mk_set_timeout(self.handle, int(ns)))

    def _arrays(self, tokens, pos):
        B = self.cfg.batch
        t = (ctypes.c_int32 * B)(*[int(v) for v in tokens])
        p = (ctypes.c_int32 * B)(*[int(v) for v in pos])
        assert len(tokens) == B and len(pos) == B
        return t, p

    def step(self, tokens: Sequence[int], pos: Sequence[int], logits=None) -> List[int]:
        """mk_decode_step: one synchronous step; logits land in ``logits`` (default self.logits)."""
        lg = self.logits if logits is None else logits
        t, p = self._arrays(tokens, pos)
        out = (ctypes.c_int32 * self.cfg.batch)()
        _check(lib.mk_decode_step(self.handle, t, p, _ptr(lg), out))
        return list(out)

    def step_static(self, tokens: Sequence[int], pos: Sequence[int], logits=None) -> List[int]:
        """mk_decode_step_static: one synchronous step using the library's static device scratch."""
        lg = self.logits if logits is None else logits
        t, p = self._arrays(tokens, pos)
        out = (ctypes.c_int32 * self.cfg.batch)()
        _check(lib.mk_decode_step_static(self.handle, t, p, _ptr(lg), out))
        return list(out)

    def steps(self, tokens: Sequence[int], pos: Sequence[int], n_steps: int, logits=None,
              tokens_dev=None) -> List[List[int]]:
        """mk_decode_steps: n_steps chained greedy steps (each step's token feeds the next on the
        device), one host synchronisation.  Returns the greedy tokens per step ([n_steps][batch]);
        ``logits`` (default self.logits) holds the last step's logits."""
        import torch
        B = self.cfg.batch
        lg = self.logits if logits is None else logits
        if tokens_dev is None:
            tokens_dev = torch.empty(n_steps * B, dtype=torch.int32, device=lg.device)
        t, p = self._arrays(tokens, pos)
        out = (ctypes.c_int32 * (max(n_steps, 1) * B))()
        _check(lib.mk_decode_steps(self.handle, t, p, int(n_steps), _ptr(lg), _ptr(tokens_dev), out))
        return [list(out[i * B:(i + 1) * B]) for i in range(n_steps)]

    def rebind(self, sched: "Schedule"):
        """mk_rebind_schedule: continue on another schedule of the same model and SM count (new KV
        windows: the variable-length re-planning).  The schedule object must outlive its use."""
        _check(lib.mk_rebind_schedule(self.handle, sched.handle))
        self.sched = sched

    def persistent_start(self, tokens: Sequence[int], pos: Sequence[int], n_steps: int, logits=None,
                         tokens_dev=None):
        """mk_decode_persistent_start: one resident launch of up to n_steps chained greedy steps,
        enqueued on the bound stream.  Returns the device token buffer ([n_steps * batch] int32);
        keep it alive until persistent_wait."""
        import torch
        B = self.cfg.batch
        lg = self.logits if logits is None else logits
        if tokens_dev is None:
            tokens_dev = torch.empty(max(int(n_steps), 1) * B, dtype=torch.int32, device=lg.device)
        t, p = self._arrays(tokens, pos)
        _check(lib.mk_decode_persistent_start(self.handle, t, p, int(n_steps), _ptr(lg), _ptr(tokens_dev)))
        self._run = (int(n_steps), tokens_dev)
        return tokens_dev

    def persistent_stop(self):
        """mk_decode_persistent_stop: the launch in flight ends after the step it is deciding."""
        _check(lib.mk_decode_persistent_stop(self.handle))

    def persistent_progress(self) -> int:
        """mk_decode_persistent_progress: steps finished so far (no wait)."""
        out = ctypes.c_int32(0)
        _check(lib.mk_decode_persistent_progress(self.handle, ctypes.byref(out)))
        return out.value

    def persistent_wait(self) -> List[List[int]]:
        """mk_decode_persistent_wait: waits for the launch; returns the greedy tokens of the steps
        it ran ([steps][batch])."""
        B = self.cfg.batch
        n_steps = self._run[0] if getattr(self, "_run", None) else 1
        done = ctypes.c_int32(0)
        out = (ctypes.c_int32 * (n_steps * B))()
        st = lib.mk_decode_persistent_wait(self.handle, ctypes.byref(done), out)
        self._run = None
        _check(st)
        return [list(out[i * B:(i + 1) * B]) for i in range(done.value)]

    def persistent(self, tokens: Sequence[int], pos: Sequence[int], n_steps: int, logits=None,
                   tokens_dev=None) -> List[List[int]]:
        """One persistent launch of n_steps steps, waited for: the tokens per step."""
        self.persistent_start(tokens, pos, n_steps, logits, tokens_dev)
        return self.persistent_wait()

    def launch(self, tokens: Sequence[int], pos: Sequence[int], logits=None, next_dev=None):
        """mk_launch_step: enqueue one step on the bound stream."""
        lg = self.logits if logits is None else logits
        t, p = self._arrays(tokens, pos)
        _check(lib.mk_launch_step(self.handle, t, p, _ptr(lg), _ptr(next_dev) if next_dev is not None else None))

    def status(self) -> List[int]:
        """mk_ctx_status: waits for the stream; raises MkError on a device error. Returns the info words."""
        info = (ctypes.c_int32 * 8)()
        st = lib.mk_ctx_status(self.handle, info)
        if st != MK_OK:
            raise MkError(st, lib.mk_last_error().decode(errors="replace"))
        return list(info)

    def set_sync(self, mode: str):
        """mk_set_sync: "tags" (epoch-tagged activations, the default) or "counters" (every
        instruction waits its completion counters first)."""
        modes = {"tags": SYNC_TAGS, "counters": SYNC_COUNTERS}
        if mode not in modes:
            raise ValueError(f"sync mode {mode!r}: expected one of {sorted(modes)}")
        _check(lib.mk_set_sync(self.handle, modes[mode]))

    def set_trace(self, buf):
        """mk_set_trace: buf is a CUDA int64 tensor of S*Q*8 elements, or None to stop tracing."""
        _check(lib.mk_set_trace(self.handle, _ptr(buf) if buf is not None else None))

    def status_code(self):
        info = (ctypes.c_int32 * 8)()
        st = lib.mk_ctx_status(self.handle, info)
        return st, list(info)
