"""ORACLE -- test infrastructure only.  An independent restatement of the offline tile
scheduler, a schedule validator and a host simulator of the per-SM queue interpreter.

The "Inference MegaKernel" page (section "Hand-written whole-model MegaKernel", paragraphs on
principle/scheduling and the object table) describes the scheduler only in outline: cut every
operator of a fixed Llama configuration into tiles, build the tile dependency DAG, assign
"waves" and a memory/compute pool, and tensorise each SM's plan into an instruction queue of
shape [S, Q, 32] int32 held in HBM for the life of the kernel; the runtime waits on counters
before an instruction and adds to counters after it.  The exact rules below are this library's
reading of that outline (the page fixes none of them):

Tiles (per layer l, in this order; ids are assigned in enumeration order):
  QKV     rows [r, r+R_qkv) of Wqkv (q heads, k heads, v heads); R_qkv <= head_dim, so a tile
          touches one or two KV groups' q, k or v ranges and completes each group it touches.
          RMSNorm of the layer input is its prologue.
  ATTN    (b, g, c): sequence b, KV group g, KV positions [c*C, (c+1)*C) -- split-K decode
          attention; c runs over the chunks of the sequence's window [0, kv_limit[b]) (default
          max_seq; chunks past pos do no work).  At batch 1 the tile whose chunk holds the
          step's position (known at run time only) also does the fixed-order log-sum-exp combine
          of the group's chunk partials, reading the lower chunks' partials as they land, and
          alone carries the tile's completion (a conditional completion); at batch > 1 the
          chunk tiles complete nothing and
  COMB    (b, g) (batch > 1 only, after every ATTN tile of the layer, in the same wave) does
          that combine for the group and carries its completion.
  OPROJ   rows of Wo, residual add.
  UPGATE  row pairs [r, r+R_up) of gate and of up, SiLU(gate)*up epilogue.
  DOWN    rows of Wdown, residual add.  At batch > 1 with rows longer than MMV_RANGE: one tile
          per (staging range a2, row block), all tiles of range 0 first, then range 1, ...; a
          tile of a lower range stores its partial sums, the tile of the last range (so of
          higher id than every partial it needs) adds them in range order, writes the rows and
          alone carries the completion.
then LMHEAD (rows of the LM head, final RMSNorm prologue, per-tile max/argmax partial) and
ARGMAX (b).
Waves: the DAG's longest-path level; per layer QKV=5l, ATTN=5l+1, OPROJ=5l+2, UPGATE=5l+3,
DOWN=5l+4; LMHEAD=5L, ARGMAX=5L+1.
Pools: memory pool = tiles that stream weights or KV (QKV, ATTN, OPROJ, UPGATE, DOWN,
LMHEAD); compute pool = COMB and ARGMAX.  Within a wave memory tiles are placed before compute
tiles.
Rows per tile: (tile_bytes 0) about one tile per operator per SM -- such a tile streams through
the page ring page by page (at batch > 1 a page is a 16-row block over page_bytes / 32
positions); at batch > 1 the down projection of rows longer than MMV_RANGE takes about
H * ranges / S rows per tile (whole 16-row blocks, at most 64); any other tile of rows longer
than MMV_RANGE (its sums held over several
staging ranges) takes at most 64 rows; otherwise tiles of about tile_bytes.
Assignment, wave by wave: memory tiles sorted by (cost desc, tile id asc), then compute tiles
likewise; the k-th tile of that order (from 0) goes to the SM with the smallest accumulated cost
(ties: lowest SM id) among the SMs holding at most k // S of the pool's tiles in this wave -- the
placement runs in rounds of S tiles, one per SM -- and the accumulated cost carries across waves.
cost = streamed bytes + TILE_OVERHEAD.
With a non-zero shuffle seed the wave's tiles are instead put in a splitmix64 Fisher-Yates
order (pools still kept apart) -- the "shuffled assignment" used to test determinism.
Queue of an SM: its tiles wave by wave, in tile-id order within a wave (so the combining
attention tile, which waits inside its wave on lower chunks of its group, only ever waits on tiles
every queue runs before it), padded with END (all-zero words).
"""
from __future__ import annotations

import heapq
import random
from dataclasses import dataclass
from typing import Dict, List, Optional, Tuple

import numpy as np

# opcodes
END, QKV, ATTN, COMB, OPROJ, UPGATE, DOWN, LMHEAD, ARGMAX = range(9)
OPNAMES = ["END", "QKV", "ATTN", "COMB", "OPROJ", "UPGATE", "DOWN", "LMHEAD", "ARGMAX"]
WORDS = 32
MAX_WAIT = 4
MAX_PUB = 2
TILE_OVERHEAD = 1024
MEMORY_OPS = (QKV, ATTN, OPROJ, UPGATE, DOWN, LMHEAD)
U32 = 1 << 32
M64 = (1 << 64) - 1


@dataclass
class SchedOpts:
    page_bytes: int = 0     # 0: 32768 at batch 1, 65536 at batch > 1 (a 16-row block over 2048 positions)
    tile_bytes: int = 0     # 0: per-SM tiles (batch > 1: at most 64 down rows when F > MMV_RANGE)
    attn_chunk: int = 0     # 0: 128 positions, doubled up to 512 while B * n_kv * chunks > 152
    shuffle_seed: int = 0
    rows_qkv: int = 0   # 0: derived from tile_bytes
    rows_o: int = 0
    pairs_up: int = 0
    rows_down: int = 0
    rows_lm: int = 0
    kv_limit: Tuple[int, ...] = (0,) * 8   # per sequence: positions served, [0, kv_limit) (0: max_seq)


def kv_window(cfg, o: SchedOpts, b: int) -> int:
    """Positions [0, window) of sequence b the schedule serves (variable-length re-planning)."""
    lim = o.kv_limit[b] if b < len(o.kv_limit) else 0
    return lim if lim else cfg.max_seq


MMV_RANGE = 2048   # batch > 1: positions of the inputs staged at a time (longer rows: several ranges)


def tile_rows(cfg, o: SchedOpts, S: int) -> Dict[str, int]:
    """Rows (pairs for gate/up) per matvec tile.  tile_bytes 0: about one tile per operator per SM,
    at batch 1 rounded up to whole consumer groups (two pages of whole rows -- for gate/up a gate
    page and its up page -- at most 16 rows or 8 pairs), at batch > 1 only the QKV rows, to a
    16-row MMA block; QKV tiles at most head_dim rows, so a tile touches one or two KV groups; at batch > 1 the down
    (and output) projection, when its rows are longer than MMV_RANGE (its sums held over several
    staging ranges), takes at most 64 rows.  Otherwise tiles of about tile_bytes.  Explicit rows_*
    override either."""
    H, F, V, d = cfg.hidden, cfg.ffn, cfg.vocab, cfg.head_dim
    qd = cfg.n_q_heads * cfg.head_dim
    nqkv = qd + 2 * cfg.n_kv_heads * d
    if o.tile_bytes == 0:
        pb = page_bytes_of(cfg, o)

        def grp(K, pair):   # rows (pairs) a tile is rounded up to
            if cfg.batch > 1:
                return 1
            rpp = max(1, pb // (2 * K))
            return min(rpp, 8) if pair else min(2 * rpp, 16)

        def up_to(r, m):
            return ceil_div(r, m) * m

        o_rows = up_to(ceil_div(H, S), grp(qd, False))
        if cfg.batch > 1 and qd > MMV_RANGE:
            o_rows = min(64, o_rows)
        nrg = down_ranges(cfg)
        down = min(64, up_to(ceil_div(H * nrg, S), 16)) if nrg > 1 else up_to(ceil_div(H, S), grp(F, False))
        R = dict(qkv=min(d, up_to(ceil_div(nqkv, S), 16 if cfg.batch > 1 else grp(H, False))), o=o_rows,
                 up=up_to(ceil_div(F, S), grp(H, True)), down=down, lm=up_to(ceil_div(V, S), grp(H, False)))
    else:
        tb = o.tile_bytes

        def fit(limit, nbytes_per_row):
            return max(1, min(limit, tb // nbytes_per_row))

        r_qkv = fit(8, 2 * H)
        while d % r_qkv:
            r_qkv -= 1
        R = dict(qkv=r_qkv, o=fit(8, 2 * qd), up=fit(16, 4 * H), down=fit(8, 2 * F), lm=fit(32, 2 * H))
    for k, v in (("qkv", o.rows_qkv), ("o", o.rows_o), ("up", o.pairs_up), ("down", o.rows_down),
                 ("lm", o.rows_lm)):
        if v:
            R[k] = v
    return R


def ceil_div(a, b):
    return -(-a // b)


class Counters:
    def __init__(self, cfg):
        L, nkv, B = cfg.n_layers, cfg.n_kv_heads, cfg.batch
        self.L, self.nkv, self.B = L, nkv, B
        self.base2 = L * nkv
        self.n = self.base2 + 4 * L + 2

    def qkv(self, l, g): return l * self.nkv + g
    def comb(self, l): return self.base2 + l
    def o(self, l): return self.base2 + self.L + l
    def up(self, l): return self.base2 + 2 * self.L + l
    def down(self, l): return self.base2 + 3 * self.L + l
    def lm(self): return self.base2 + 4 * self.L
    def final(self): return self.base2 + 4 * self.L + 1


@dataclass
class Tile:
    op: int
    layer: int
    b: int
    a0: int
    a1: int
    a2: int
    wave: int
    waits: List[Tuple[int, int]]
    pubs: List[Tuple[int, int]]
    stream_bytes: int
    tid: int = -1
    cond: bool = False   # ATTN: pubs only from the tile that combines its group

    @property
    def memory(self) -> bool:
        return self.op in MEMORY_OPS

    @property
    def cost(self) -> int:
        return self.stream_bytes + TILE_OVERHEAD


ATTN_CHUNK_TILES = 152   # the default chunk grows while a layer has more chunks than this


def attn_chunk(cfg, o: SchedOpts, S: int) -> int:
    """KV positions per split-K attention tile: the option, else 128 doubled (at most to 512) as
    long as the chunks of all sequences and KV heads outnumber ATTN_CHUNK_TILES -- a property of
    the configuration, independent of the queue count S."""
    if o.attn_chunk:
        return o.attn_chunk
    C = 128
    while C < 512 and cfg.batch * cfg.n_kv_heads * ceil_div(cfg.max_seq, C) > ATTN_CHUNK_TILES:
        C *= 2
    return C


def enumerate_tiles(cfg, o: SchedOpts, S: int) -> Tuple[List[Tile], Counters, Dict[str, int]]:
    L, H, F, V, B = cfg.n_layers, cfg.hidden, cfg.ffn, cfg.vocab, cfg.batch
    nq, nkv, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    qd, kvd = nq * d, nkv * d
    hpg = nq // nkv
    R = tile_rows(cfg, o, S)
    C = attn_chunk(cfg, o, S)
    nchunk = ceil_div(cfg.max_seq, C)
    cnt = Counters(cfg)
    n_qkv_rows = qd + 2 * kvd
    n_qkv = ceil_div(n_qkv_rows, R["qkv"])
    n_o = ceil_div(H, R["o"])
    n_up = ceil_div(F, R["up"])
    n_dn = ceil_div(H, R["down"])
    n_lm = ceil_div(V, R["lm"])
    tiles: List[Tile] = []

    def group_of_row(r):
        if r < qd:
            return (r // d) // hpg
        if r < qd + kvd:
            return (r - qd) // d
        return (r - qd - kvd) // d

    # a QKV tile (<= head_dim rows) touches one or two KV groups and completes each of them
    def groups_of_tile(r0, n):
        g0, g1 = group_of_row(r0), group_of_row(r0 + n - 1)
        return [g0] if g0 == g1 else [g0, g1]

    qkv_tiles_of_group = [0] * nkv
    for t in range(n_qkv):
        r0 = t * R["qkv"]
        for g in groups_of_tile(r0, min(R["qkv"], n_qkv_rows - r0)):
            qkv_tiles_of_group[g] += 1

    for l in range(L):
        wq = [] if l == 0 else [(cnt.down(l - 1), n_dn)]
        for t in range(n_qkv):
            r0 = t * R["qkv"]
            n = min(R["qkv"], n_qkv_rows - r0)
            tiles.append(Tile(QKV, l, 0, r0, n, 0, 5 * l, list(wq),
                              [(cnt.qkv(l, g), 1) for g in groups_of_tile(r0, n)], n * H * 2))
        for b in range(B):
            for g in range(nkv):
                for c in range(nchunk):
                    if c * C >= kv_window(cfg, o, b):   # chunks past the sequence's window: no tile
                        break
                    rows = min(C, kv_window(cfg, o, b) - c * C)   # the chunk's K/V rows in the window
                    if B == 1:   # the chunk holding pos combines and completes
                        tiles.append(Tile(ATTN, l, b, g, c, C, 5 * l + 1,
                                          [(cnt.qkv(l, g), qkv_tiles_of_group[g])],
                                          [(cnt.comb(l), 1)], 2 * rows * d * 2, cond=True))
                    else:        # combined by the group's COMB tile
                        tiles.append(Tile(ATTN, l, b, g, c, C, 5 * l + 1,
                                          [(cnt.qkv(l, g), qkv_tiles_of_group[g])], [], 2 * rows * d * 2))
        if B > 1:
            for b in range(B):
                for g in range(nkv):
                    tiles.append(Tile(COMB, l, b, g, 0, C, 5 * l + 1, [], [(cnt.comb(l), 1)], 0))
        for t in range(n_o):
            r0 = t * R["o"]
            n = min(R["o"], H - r0)
            tiles.append(Tile(OPROJ, l, 0, r0, n, 0, 5 * l + 2, [(cnt.comb(l), B * nkv)],
                              [(cnt.o(l), 1)], n * qd * 2))
        for t in range(n_up):
            r0 = t * R["up"]
            n = min(R["up"], F - r0)
            tiles.append(Tile(UPGATE, l, 0, r0, n, 0, 5 * l + 3, [(cnt.o(l), n_o)],
                              [(cnt.up(l), 1)], 2 * n * H * 2))
        nrg = down_ranges(cfg)
        for r in range(nrg):
            kr = min(MMV_RANGE, F - r * MMV_RANGE) if nrg > 1 else F
            for t in range(n_dn):
                r0 = t * R["down"]
                n = min(R["down"], H - r0)
                tiles.append(Tile(DOWN, l, 0, r0, n, r, 5 * l + 4, [(cnt.up(l), n_up)],
                                  [(cnt.down(l), 1)] if r == nrg - 1 else [], n * kr * 2))
    for t in range(n_lm):
        r0 = t * R["lm"]
        n = min(R["lm"], V - r0)
        tiles.append(Tile(LMHEAD, L, 0, r0, n, t, 5 * L, [(cnt.down(L - 1), n_dn)],
                          [(cnt.lm(), 1)], n * H * 2))
    for b in range(B):
        tiles.append(Tile(ARGMAX, L, b, 0, n_lm, 0, 5 * L + 1, [(cnt.lm(), n_lm)],
                          [(cnt.final(), 1)], 0))
    for i, t in enumerate(tiles):
        t.tid = i
    return tiles, cnt, R


class SplitMix64:
    def __init__(self, seed: int):
        self.s = seed & M64

    def next(self) -> int:
        self.s = (self.s + 0x9E3779B97F4A7C15) & M64
        z = self.s
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        return z ^ (z >> 31)


def _shuffle(xs: List[Tile], rng: SplitMix64) -> List[Tile]:
    xs = list(xs)
    for i in range(len(xs) - 1, 0, -1):
        j = rng.next() % (i + 1)
        xs[i], xs[j] = xs[j], xs[i]
    return xs


def down_ranges(cfg) -> int:
    """Staging ranges of the down projection's rows when it runs one tile per (range, row block):
    at batch > 1 with rows longer than MMV_RANGE; else 1."""
    return ceil_div(cfg.ffn, MMV_RANGE) if cfg.batch > 1 and cfg.ffn > MMV_RANGE else 1


def page_bytes_of(cfg, o: SchedOpts) -> int:
    return o.page_bytes or (65536 if cfg.batch > 1 else 32768)


def tile_pages(t: Tile, cfg, o: SchedOpts) -> int:
    """Pages of a tile's stream: at batch 1 a matvec tile streams whole rows per page (gate/up:
    gate and up row groups in alternate pages), at batch > 1 one 16-row block (gate/up: 8 gate
    rows and the 8 up rows of the same pairs) over page_bytes / 32 positions per page; an
    attention tile streams its bytes contiguously."""
    if t.op in (QKV, OPROJ, UPGATE, DOWN, LMHEAD):
        K = cfg.q_dim if t.op == OPROJ else (cfg.ffn if t.op == DOWN else cfg.hidden)
        if cfg.batch > 1:   # 16-row blocks (gate/up: 8 pairs) over page_bytes / 32 positions
            kp = page_bytes_of(cfg, o) // 32
            if t.op == DOWN and down_ranges(cfg) > 1:   # one staging range of the rows
                K = min(MMV_RANGE, K - t.a2 * MMV_RANGE)
            return ceil_div(t.a1, 8 if t.op == UPGATE else 16) * ceil_div(K, kp)
        rpp = page_bytes_of(cfg, o) // (2 * K)
        return ceil_div(t.a1, rpp) * (2 if t.op == UPGATE else 1)
    return ceil_div(t.stream_bytes, page_bytes_of(cfg, o))


def encode(t: Tile, n_pages: int) -> List[int]:
    w = [0] * WORDS
    w[0], w[1], w[2], w[3], w[4], w[5] = t.op, t.layer, t.b, t.a0, t.a1, t.a2
    w[6] = len(t.waits)
    for i, (c, need) in enumerate(t.waits):
        w[7 + 2 * i], w[8 + 2 * i] = c, need
    w[15] = len(t.pubs)
    for i, (c, delta) in enumerate(t.pubs):
        w[16 + 2 * i], w[17 + 2 * i] = c, delta
    w[20] = n_pages
    w[21] = t.tid
    w[22] = t.wave
    if t.cond:   # completions only from the tile that combines its group
        w[23] = 1
    return w


def build_schedule(cfg, S: int, opts: Optional[SchedOpts] = None):
    """Returns (queues int32 [S, Q, 32], per-step counter totals uint32 [n_counters], info)."""
    o = opts or SchedOpts()
    if S < 1:
        raise ValueError("sm_count must be >= 1")
    tiles, cnt, R = enumerate_tiles(cfg, o, S)
    by_wave: Dict[int, List[Tile]] = {}
    for t in tiles:
        by_wave.setdefault(t.wave, []).append(t)
    rng = SplitMix64(o.shuffle_seed) if o.shuffle_seed else None
    # each tile, in order, to the SM with the smallest accumulated cost (ties: lowest SM) among
    # those holding at most k // S of the wave's tiles of its pool (rounds of S tiles, one per SM)
    acc = np.zeros(S, dtype=np.int64)
    per_sm: List[List[Tile]] = [[] for _ in range(S)]
    for wv in sorted(by_wave):
        mem = [t for t in by_wave[wv] if t.memory]
        cmp_ = [t for t in by_wave[wv] if not t.memory]
        if rng is None:
            pools = [sorted(mem, key=lambda t: (-t.cost, t.tid)), sorted(cmp_, key=lambda t: (-t.cost, t.tid))]
        else:
            pools = [_shuffle(mem, rng), _shuffle(cmp_, rng)]
        start = [len(q) for q in per_sm]
        for pool in pools:
            in_wave = np.zeros(S, dtype=np.int64)
            big = np.iinfo(np.int64).max
            for k, t in enumerate(pool):
                cap = k // S + 1   # round k // S: every SM takes a tile of it before any takes another
                s = int(np.argmin(np.where(in_wave < cap, acc, big)))   # first minimum: lowest SM
                per_sm[s].append(t)
                acc[s] += t.cost
                in_wave[s] += 1
        for s in range(S):   # a queue runs its tiles of a wave in id order
            per_sm[s][start[s]:] = sorted(per_sm[s][start[s]:], key=lambda t: t.tid)
    Q = 1 + max(len(q) for q in per_sm)
    queues = np.zeros((S, Q, WORDS), dtype=np.int32)
    for s in range(S):
        for i, t in enumerate(per_sm[s]):
            queues[s, i] = encode(t, tile_pages(t, cfg, o))
    totals = np.zeros(cnt.n, dtype=np.uint64)
    for t in tiles:
        if t.cond and t.a1 != 0:   # a group's completion counts once
            continue
        for c, dl in t.pubs:
            totals[c] += dl
    info = dict(rows=R, n_tiles=len(tiles), counters=cnt, tiles=tiles,
                n_chunks=ceil_div(cfg.max_seq, attn_chunk(cfg, o, S)))
    return queues, totals.astype(np.uint32), info


# --------------------------------------------------------------------------------------
# Validator
# --------------------------------------------------------------------------------------

def _decode(w) -> Tile:
    waits = [(int(w[7 + 2 * i]), int(w[8 + 2 * i])) for i in range(int(w[6]))]
    pubs = [(int(w[16 + 2 * i]), int(w[17 + 2 * i])) for i in range(int(w[15]))]
    t = Tile(int(w[0]), int(w[1]), int(w[2]), int(w[3]), int(w[4]), int(w[5]), int(w[22]),
             waits, pubs, 0, int(w[21]))
    t.cond = int(w[23]) == 1
    return t


def validate(queues: np.ndarray, totals: np.ndarray, cfg, opts: Optional[SchedOpts] = None,
             page_bytes_capacity: Optional[int] = None) -> List[str]:
    """Checks the contract a schedule must satisfy; returns a list of violations (empty = valid).

    * every tile of the model appears exactly once; END only as padding, at least one END per SM;
    * each counter's per-step total equals the sum of the deltas published into it, and every
      wait asks for exactly that total (a consumer waits for all producers of its counter);
    * waits point only at counters produced in strictly lower waves, and each SM's queue is in
      non-decreasing wave order (the forward-progress rule: a waiter never holds an SM that a
      producer it waits on still needs);
    * within a wave each SM's tiles are in increasing tile-id order, and at batch 1 the
      attention chunk tiles of a group carry conditional completions (exactly one completion per
      group is counted): the combining chunk tile's wait inside its wave is on lower chunks of
      its group, i.e. on lower ids, which no queue runs after a higher id of that wave (at
      batch > 1 the COMB tile of the group waits likewise on the chunk tiles, all of lower id, and
      a down tile of the last staging range on the same rows' tiles of the other ranges);
    * (DAG + per-SM program order) is acyclic -- implied by the points above;
    * capacity: at most 4 waits and 2 completions per instruction; no attention tile needs more
      pages than the ring holds.
    """
    o = opts or SchedOpts()
    errs: List[str] = []
    S, Q, W = queues.shape
    if W != WORDS:
        return [f"instruction width {W} != {WORDS}"]
    ref_tiles, cnt, _ = enumerate_tiles(cfg, o, S)
    seen: Dict[int, Tuple[int, int]] = {}
    pub_sum = np.zeros(cnt.n, dtype=np.int64)
    producer_wave: Dict[int, int] = {}
    for s in range(S):
        ended = False
        last_wave = -1
        last_tid = -1
        for i in range(Q):
            w = queues[s, i]
            if w[0] == END:
                if np.any(w != 0):
                    errs.append(f"sm {s} slot {i}: END with non-zero words")
                ended = True
                continue
            if ended:
                errs.append(f"sm {s} slot {i}: instruction after END")
            t = _decode(w)
            if not (0 < t.op <= ARGMAX):
                errs.append(f"sm {s} slot {i}: bad opcode {t.op}")
                continue
            if t.tid in seen:
                errs.append(f"tile {t.tid} appears twice")
            seen[t.tid] = (s, i)
            if t.wave < last_wave:
                errs.append(f"sm {s} slot {i}: wave {t.wave} after wave {last_wave}")
            elif t.wave == last_wave and t.tid < last_tid:
                errs.append(f"sm {s} slot {i}: tile {t.tid} after tile {last_tid} of the same wave")
            last_wave, last_tid = t.wave, t.tid
            if len(t.waits) > MAX_WAIT or len(t.pubs) > MAX_PUB:
                errs.append(f"tile {t.tid}: too many waits/completions")
            if t.cond != (t.op == ATTN and cfg.batch == 1):
                errs.append(f"tile {t.tid}: conditional completions on a {OPNAMES[t.op]} tile"
                            if t.cond else f"tile {t.tid}: batch-1 attention tile without conditional completions")
            # conditional completions: one per group, counted at its chunk 0 (which tile fires it
            # is decided at run time)
            produced = [] if (t.cond and t.a1 != 0) else list(t.pubs)
            for c, dl in produced:
                pub_sum[c] += dl
                pw = producer_wave.setdefault(c, t.wave)
                if pw != t.wave:
                    errs.append(f"counter {c} produced in waves {pw} and {t.wave}")
            # an attention tile holds its pages until it is done: it must fit the ring (a matvec
            # tile streams through the ring page by page)
            if page_bytes_capacity is not None and t.op == ATTN and w[20] * page_bytes_of(cfg, o) > page_bytes_capacity:
                errs.append(f"tile {t.tid}: needs {w[20]} pages, ring too small")
            ref = ref_tiles[t.tid] if 0 <= t.tid < len(ref_tiles) else None
            if ref is None or (ref.op, ref.layer, ref.b, ref.a0, ref.a1, ref.a2) != \
                    (t.op, t.layer, t.b, t.a0, t.a1, t.a2):
                errs.append(f"tile {t.tid}: fields do not match the model's tile")
        if not ended:
            errs.append(f"sm {s}: queue not END-terminated")
    if len(seen) != len(ref_tiles):
        errs.append(f"{len(seen)} tiles scheduled, model has {len(ref_tiles)}")
    if not np.array_equal(pub_sum.astype(np.uint32), np.asarray(totals, dtype=np.uint32)):
        errs.append("per-step counter totals differ from the sum of published deltas")
    for s in range(S):
        for i in range(Q):
            w = queues[s, i]
            if w[0] == END:
                continue
            t = _decode(w)
            for c, need in t.waits:
                if c not in producer_wave:
                    errs.append(f"tile {t.tid}: waits on counter {c} that nobody produces")
                    continue
                if producer_wave[c] >= t.wave:
                    errs.append(f"tile {t.tid}: waits on counter {c} of wave {producer_wave[c]}")
                if need != pub_sum[c]:
                    errs.append(f"tile {t.tid}: waits for {need} on counter {c}, total {pub_sum[c]}")
    return errs


# --------------------------------------------------------------------------------------
# Host simulator of the queue interpreter (page section "principle, scheduling and data flow":
# fetch instruction -> END? -> wait counters -> lease pages -> run body -> fence ->
# add completions -> release pages -> next), with abstract data tracking.
# --------------------------------------------------------------------------------------

def _reads_writes(t: Tile, cfg):
    """Abstract buffers a tile reads and writes, as (key, rows) pairs: a write adds its rows to
    the key's count; a read requires the key's count to have reached the given number of rows
    (its writers have all run).  Used to check every read follows its write."""
    L, H, nq, nkv, d = cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    F, hpg = cfg.ffn, nq // nkv
    l, op = t.layer, t.op
    R, W = [], []
    if op == QKV:
        if l > 0:
            R.append((("x_out", l - 1), H))
        qd, kvd = nq * d, nkv * d

        def group(r):
            return (r // d) // hpg if r < qd else ((r - qd) // d if r < qd + kvd else (r - qd - kvd) // d)

        for r in range(t.a0, t.a0 + t.a1):   # rows counted per KV group (a tile may touch two)
            W.append((("qkv", l, group(r)), 1))
    elif op == ATTN:   # (its partial and the combine's output: in the simulator, by position)
        R.append((("qkv", l, t.a0), (hpg + 2) * d))
    elif op == OPROJ:
        R.append((("o", l), cfg.batch * nkv))
        if l > 0:
            R.append((("x_out", l - 1), H))
        W.append((("x_attn", l), t.a1))
    elif op == UPGATE:
        R.append((("x_attn", l), H))
        W.append((("h", l), t.a1))
    elif op == DOWN:
        R.append((("h", l), F))
        nrg = down_ranges(cfg)
        if t.a2 + 1 < nrg:   # a partial of range a2 (the last range's tile reads it: in the simulator)
            W.append((("dpart", l, t.a0), 1))
        else:
            R.append((("x_attn", l), H))
            W.append((("x_out", l), t.a1))
    elif op == LMHEAD:
        R.append((("x_out", L - 1), H))
        W.append((("lmpart",), 1))
    elif op == ARGMAX:
        R.append((("lmpart",), t.a1))
        W.append((("token", t.b), 1))
    return R, W


def simulate(queues: np.ndarray, totals: np.ndarray, cfg, n_epochs: int = 2, seed: int = 0,
             track_data: bool = True, pos: Optional[List[int]] = None) -> List[str]:
    """Runs the S queues on the host under a random interleaving, for n_epochs consecutive steps
    with epoch-offset counter targets (target = epoch * total + need, compared modulo 2^32).
    Sequence b decodes position pos[b] (default: the last position its scheduled chunks cover): the
    chunk tiles past it do nothing, the others write their partial, and the tile of the chunk
    holding it waits (inside its wave) until the lower chunks of its group have written theirs,
    then writes the group's attention output and fires the completion (at batch > 1 the group's
    COMB tile waits for every active chunk's partial and does that; a batch > 1 down tile of the
    last staging range waits likewise for the partials of its rows' other ranges).  Reports a deadlock (no
    SM can progress before all reach END) and any read of a buffer whose writer has not yet run
    in the current step."""
    S, Q, _ = queues.shape
    decoded0 = [_decode(queues[s, i]) for s in range(S) for i in range(Q) if queues[s, i, 0] != END]
    if pos is None:   # the last position each sequence's scheduled chunks cover
        pos = [min(cfg.max_seq - 1, max([(t.a1 + 1) * t.a2 - 1 for t in decoded0 if t.op == ATTN and t.b == b],
                                        default=cfg.max_seq - 1)) for b in range(cfg.batch)]
    rng = random.Random(seed)
    counters = np.zeros(len(totals), dtype=np.int64)
    errs: List[str] = []
    decoded = [[_decode(queues[s, i]) if queues[s, i, 0] != END else None for i in range(Q)]
               for s in range(S)]
    rw_cache: Dict[int, Tuple[list, list]] = {}
    for epoch in range(n_epochs):
        pc = [0] * S
        written: Dict[tuple, int] = {}
        live = [s for s in range(S)]
        while live:
            rng.shuffle(live)
            progressed = False
            nxt = []
            for s in live:
                t = decoded[s][pc[s]]
                if t is None:
                    continue  # reached END
                ok = all(((int(counters[c]) - (epoch * int(totals[c]) + need)) % U32) < (U32 >> 1)
                         for c, need in t.waits)
                c_pos = pos[t.b] // t.a2 if t.op in (ATTN, COMB) else -1   # the chunk holding pos
                part_key = ("part", t.layer, t.b, t.a0)
                combines = (t.op == ATTN and t.cond and t.a1 == c_pos) or t.op == COMB
                if ok and combines:   # the combine reads chunks 0 .. c_pos - 1 (COMB: 0 .. c_pos)
                    ok = written.get(part_key, 0) >= (c_pos if t.op == ATTN else c_pos + 1)
                nrg = down_ranges(cfg) if t.op == DOWN else 1
                if ok and nrg > 1 and t.a2 == nrg - 1:   # the last range's tile reads the other partials
                    ok = written.get(("dpart", t.layer, t.a0), 0) >= nrg - 1
                if ok:
                    if track_data:
                        if t.tid not in rw_cache:
                            rw_cache[t.tid] = _reads_writes(t, cfg)
                        rd, wr = rw_cache[t.tid]
                        for key, need_rows in rd:
                            if written.get(key, 0) < need_rows:
                                errs.append(f"epoch {epoch}: tile {t.tid} ({OPNAMES[t.op]}) read "
                                            f"{key} before all of it was written")
                                return errs
                        for key, n in wr:
                            written[key] = written.get(key, 0) + n
                    pubs = t.pubs
                    if t.op == ATTN:
                        if t.a1 <= c_pos:
                            written[part_key] = written.get(part_key, 0) + 1
                        if combines:
                            written[("o", t.layer)] = written.get(("o", t.layer), 0) + 1
                        elif t.cond:
                            pubs = []
                    elif t.op == COMB:
                        written[("o", t.layer)] = written.get(("o", t.layer), 0) + 1
                    for c, dl in pubs:
                        counters[c] += dl
                    pc[s] += 1
                    progressed = True
                nxt.append(s)
            live = [s for s in nxt if decoded[s][pc[s]] is not None]
            if live and not progressed:
                blocked = live[0]
                return errs + [f"epoch {epoch}: deadlock, sm {blocked} stuck at slot {pc[blocked]}"]
    return errs
