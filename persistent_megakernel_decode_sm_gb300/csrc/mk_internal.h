// Internal definitions shared by the library's translation units (scheduler, binding, kernel).
#pragma once

#include <stddef.h>
#include <stdint.h>
#include <vector_types.h>

#include "mk.h"

#ifdef __CUDACC__
#define MK_HD __host__ __device__
#else
#define MK_HD
#endif

namespace mk {

// ---- instruction encoding ([S, Q, 32] int32, see mk_schedule_queues) ---------------------
enum Op : int32_t { OP_END = 0, OP_QKV = 1, OP_ATTN = 2, OP_COMB = 3, OP_OPROJ = 4, OP_UPGATE = 5,
                    OP_DOWN = 6, OP_LMHEAD = 7, OP_ARGMAX = 8, OP_COUNT = 9 };
enum Word : int {
    W_OP = 0, W_LAYER = 1, W_B = 2, W_A0 = 3, W_A1 = 4, W_A2 = 5, W_NWAIT = 6, W_WAIT = 7,
    W_NPUB = 15, W_PUB = 16, W_NPAGES = 20, W_TILE = 21, W_WAVE = 22,
    W_COND = 23,   // 1: completions only from the tile that combines its group (ATTN: the chunk holding pos)
    W_SRC0 = 26, W_SRC1 = 28, W_BYTES0 = 30, W_BYTES1 = 31   // device copy: resolved weight stream (matvec)
};
constexpr int kWords = 32;
constexpr int kMaxWait = 4;
constexpr int kMaxPub = 2;
constexpr int kMaxBatch = 8;
constexpr int kMaxHpg = 8;         // query heads per KV head
constexpr int kMaxHeadDim = 128;
constexpr int kMaxK = 16384;       // longest matvec row (elements)
constexpr int64_t kTileOverhead = 1024;

// shared-memory layout of one CTA (after the page ring)
constexpr int kNumConsumerWarps = 8;
constexpr int kConsumerThreads = kNumConsumerWarps * 32;
constexpr int kLoaderWarp = 8;
constexpr int kPublisherWarp = 9;
constexpr int kThreads = 320;
constexpr int kSlots = 16;   // instruction slots in flight
constexpr int kQWin = 16;    // instructions per queue-window buffer (two buffers, bulk-copied)
constexpr int kMaxLayersSmem = 40;   // layer pointer table cached in shared memory
constexpr int kDone = 64;            // completion records the publisher may lag behind
constexpr int kTraceWords = 8;       // trace stamps per instruction
constexpr unsigned kPollBackoffNs = 0;     // pause between two polling rounds of tagged data (a round
                                           // re-reads only stale chunks; measured against 32 and 100 ns:
                                           // batch-1 step 681 us against 686 and 684, batch 8 unchanged)
constexpr int kMaxCpl = 8;           // 16-byte chunks a lane holds of its row segment (at most)
constexpr int kMaxSeg = 8;           // row segments of a matvec (a power of two dividing the warp count)
constexpr int kDirectMinK = 4097;    // rows this long take their input per warp, not through the shared buffer
constexpr int kXChunks = 2;          // 8-element input chunks a consumer thread polls per round
constexpr int kCombWords = 12;       // partial words a consumer thread polls per round of the attention combine
constexpr int kResBuf = 64;          // residual words of a tile's rows staged in shared memory (per buffer)
constexpr int kMaxRingPages = 64;    // cap on the page ring's length (the shared memory sets the rest)
constexpr int kMinXBuf = 3072;       // floats of the shared input buffer at least (attention scores, combine)
constexpr int kMmvRange = 2048;      // batch > 1: positions of a row staged at a time (longer rows: ranges)
// batch > 1: staging ranges of the MLP down projection's rows when it is cut into one tile per
// (range, row block) -- rows longer than kMmvRange -- else 1 (whole-row tiles)
MK_HD inline int mmv_down_ranges(int B, int F) { return B > 1 && F > kMmvRange ? (F + kMmvRange - 1) / kMmvRange : 1; }
constexpr int kAttnChunkTiles = 152; // default attention chunk: grown while a layer has more chunks


// ---- resolved schedule parameters -----------------------------------------------------------
struct Geometry {
    int32_t page_bytes, tile_bytes, attn_chunk;
    int32_t r_qkv, r_o, r_up, r_dn, r_lm;    // rows (pairs for up) per tile
    int32_t n_qkv, n_o, n_up, n_dn, n_lm;    // tiles per layer (n_lm: LM head)
    int32_t n_chunk;                          // attention chunks per (sequence, group)
    int32_t n_counters;
    uint64_t shuffle_seed;
    int32_t kv_limit[kMaxBatch];              // per sequence: positions [0, kv_limit) served
};

// counter ids
struct CounterMap {
    int32_t L, nkv, B, base2;
    explicit CounterMap(const mk_model_cfg& c)
        : L(c.n_layers), nkv(c.n_kv_heads), B(c.batch), base2(c.n_layers * c.n_kv_heads) {}
    int32_t qkv(int l, int g) const { return l * nkv + g; }
    int32_t comb(int l) const { return base2 + l; }
    int32_t o(int l) const { return base2 + L + l; }
    int32_t up(int l) const { return base2 + 2 * L + l; }
    int32_t down(int l) const { return base2 + 3 * L + l; }
    int32_t lm() const { return base2 + 4 * L; }
    int32_t fin() const { return base2 + 4 * L + 1; }
    int32_t count() const { return base2 + 4 * L + 2; }
};

// ---- scratch layout, each region 256-byte aligned ----------------------------------------------
// The activation vectors a step hands from one operator to the next (qkv, o, x_attn, x_out) are
// epoch-tagged: one 64-bit word per element, fp32 value in the low half, the step's tag in the high
// half, written and read as single 64-bit accesses.  A reader that sees this step's tag has the
// value of this step -- the element needs no separate flag, fence or counter to be consumed.
struct ScratchLayout {
    size_t err, tokens, x_attn, x_out, qkv, part, o, h, dpart, lm_part, rope, total;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

inline ScratchLayout scratch_layout(const mk_model_cfg& c, const Geometry& g, int S) {
    const size_t L = c.n_layers, B = c.batch, H = c.hidden, d = c.head_dim;
    const size_t qd = size_t(c.n_q_heads) * d, kvd = size_t(c.n_kv_heads) * d;
    const size_t hpg = c.n_q_heads / c.n_kv_heads;
    ScratchLayout s{};
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t r = off; off = align256(off + bytes); return r; };
    s.err = take(256);            // int32 err[16] at 0, int32 tokens[8] at byte 64 (one readback)
    s.tokens = s.err + 64;
    s.x_attn = take(L * B * H * 8);                   // tagged
    s.x_out = take(L * B * H * 8);                    // tagged
    s.qkv = take(L * B * (qd + 2 * kvd) * 8);         // tagged
    s.part = take(L * B * size_t(c.n_kv_heads) * g.n_chunk * hpg * (d + 2) * 8);   // tagged chunk partials
    s.o = take(L * B * qd * 8);                       // tagged
    s.h = take(L * B * size_t(c.ffn) * 4);            // fp32 with a 3-bit tag
    s.dpart = take(L * size_t(mmv_down_ranges(c.batch, c.ffn) - 1) * B * H * 4);   // down partial sums, 3-bit tag
    s.lm_part = take(B * size_t(S) * kNumConsumerWarps * 16);   // per (sequence, CTA, warp): max, index, epoch
    s.rope = take(size_t(c.max_seq) * (d / 2) * 8);
    s.total = off;
    return s;
}

// per-layer device pointers (bf16)
struct LayerPtrs {
    const uint16_t* attn_norm;
    const uint16_t* wqkv;
    const uint16_t* wo;
    const uint16_t* mlp_norm;
    const uint16_t* wgate_up;
    const uint16_t* wdown;
};

// Matvec shape per opcode, resolved at bind.  A row of K elements is cut into G segments of
// segch 16-byte chunks (the last one may be shorter); warp w always computes segment w mod G of
// every row, holding that segment of the input vector in registers (at most cpl chunks per lane;
// the kernel is built for cpl 4 and 8, and a model takes the smallest that holds its longest row in
// at most kMaxSeg segments).  G is the smallest power of two that keeps a segment within 32 * cpl
// chunks: a property of K and cpl alone, so the arithmetic of a row never depends on the tiling or
// the SM count.  Pages hold whole
// rows (rpp per page).
struct MvShape {
    int32_t K, chunks;       // row length: elements, 16-byte chunks
    int32_t G, logG;         // segments per row, log2
    int32_t segch;           // chunks per segment
    uint32_t rowbytes;       // 2 K
    int32_t rpp;             // rows per page (whole rows, or row slices)
    int32_t direct;          // 1: each warp polls its own input segment (no shared input buffer)
};

MK_HD inline MvShape mv_shape(int K, int cpl, int page_bytes, int xbuf_floats) {
    MvShape m{};
    m.K = K;
    m.chunks = K / 8;
    m.G = 1;
    m.logG = 0;
    while ((m.chunks + m.G - 1) / m.G > 32 * cpl && m.G < kMaxSeg) { m.G *= 2; ++m.logG; }
    m.segch = (m.chunks + m.G - 1) / m.G;
    m.rowbytes = uint32_t(K) * 2u;
    m.rpp = page_bytes / int(m.rowbytes);
    m.direct = K > xbuf_floats ? 1 : 0;
    return m;
}

// pages of a matvec tile of `rows` rows (pairs for gate/up).  Batch 1 (kp 0): whole rows per page,
// gate and up row groups in alternate pages.  Batch > 1: a page holds one 16-row block (gate/up:
// 8 gate rows, then the 8 up rows of the same pairs) over kp positions; every block of every
// slice, in the order (staging range, block, slice)
MK_HD inline int64_t mv_tile_pages(const MvShape& m, int kp, int64_t rows, bool pair) {
    if (kp) return ((rows + (pair ? 7 : 15)) / (pair ? 8 : 16)) * ((m.K + kp - 1) / kp);
    return ((rows + m.rpp - 1) / m.rpp) * (pair ? 2 : 1);
}
// batch > 1: pages of a tile over staging range r of rows of length K (16-row blocks)
MK_HD inline int64_t mmv_range_pages(int K, int kp, int64_t rows, int r) {
    const int64_t kr = K - int64_t(r) * kMmvRange < kMmvRange ? K - int64_t(r) * kMmvRange : kMmvRange;
    return ((rows + 15) / 16) * ((kr + kp - 1) / kp);
}

// ---- kernel parameters (passed by value) ----------------------------------------------------
struct Params {
    MvShape mv[OP_COUNT];    // matvec shapes by opcode (unused entries zero)
    // model
    int32_t L, H, nq, nkv, d, F, V, B, max_seq, hpg, qd, kvd, nqkv;
    float rms_eps, attn_scale;
    // geometry
    int32_t page_bytes, page_shift, n_pages, attn_chunk, n_chunk, n_lm;
    // queues and counters
    const int32_t* queues;
    int32_t Q, n_counters;
    const uint32_t* totals;
    uint32_t* counters;
    // weights
    const uint16_t* embed;
    const uint16_t* lm_head;
    const uint16_t* final_norm;
    const LayerPtrs* layers;
    // KV cache
    uint16_t* kc;
    uint16_t* vc;
    int64_t kv_bstride, kv_lstride, kv_hstride;
    const int32_t* kv_table;   // paged cache: DEVICE int32[B][kv_max_blocks] block table (null: contiguous)
    int32_t kv_max_blocks, kv_n_blocks;
    // scratch
    int32_t* err;
    int32_t* tokens_out;
    uint64_t* x_attn;   // tagged [L][B][H]: residual stream after attention
    uint64_t* x_out;    // tagged [L][B][H]: residual stream after the MLP
    uint64_t* qkv;      // tagged [L][B][nqkv]
    uint64_t* part;     // [L][B][nkv][n_chunk][hpg][d + 2] attention chunk partials (tagged)
    uint64_t* o;        // tagged [L][B][qd]: attention output
    uint32_t* h;        // [L][B][F]: SwiGLU output, fp32 with a 3-bit step tag in the low mantissa bits
    uint32_t* dpart;    // batch > 1: [L][ranges - 1][B][H] partial sums of the down projection's range tiles (3-bit tag)
    int4* lm_part;      // [B][S][kNumConsumerWarps]: (max bits, index, epoch, 0)
    const float2* rope; // [max_seq][d/2] (cos, sin)
    // step
    uint32_t epoch;
    uint32_t tag;            // epoch + 1: the tag of this step's activation words (0 = never written)
    int32_t sync_counters;   // 1: every counter wait acquires, every publish releases (MK_SYNC_COUNTERS)
    uint32_t acquire_ops;    // bit op: its counter waits acquire (it reads untagged inputs)
    uint32_t release_ops;    // bit op: its completions are published after a release fence
    int32_t tok[kMaxBatch];
    int32_t pos[kMaxBatch];
    float* logits;
    int32_t* next_dev;       // optional DEVICE int32[n_steps][B]: step s's greedy tokens at [s * B]
    const int32_t* tok_dev;  // optional DEVICE int32[B]: the first step's tokens (a chained step), else tok
    int32_t n_steps;         // steps this launch runs (>= 1): step s at epoch + s, positions pos + s
    uint32_t* step_bar;      // DEVICE word: every CTA adds 1 when it retires a step (e * grid at epoch e's start)
    volatile int32_t* ctl;   // optional host-mapped words: [0] stop request (host), [1] steps done (device)
    uint64_t timeout_ns;
    uint64_t* trace;         // optional [S][Q][8] globaltimer stamps (null: off)
    // shared-memory carve-up
    int32_t smem_misc_off;   // byte offset of the non-ring area
    int32_t qrot_floats;
    int32_t xbuf_floats;     // shared input buffer (floats)
    int32_t comb_stride;     // (row, segment) units of a page, at most: partial words per page slot
    int32_t mmv_kp;          // batch > 1: positions of a row in a page (page_bytes / 32: a page holds a
                             // 16-row block, rows 2 mmv_kp bytes apart); 0 at batch 1 (whole rows)
    const uint8_t* tmaps;    // batch > 1: TMA tensor maps (128 bytes each) over the matvec weights:
                             // [4 l + {QKV, O, gate/up, down}], then the LM head at [4 L]
};

// batch > 1: a [R][K] weight matrix is viewed as [R][K / g0][g0] elements, so that one tensor box
// of (g0, kp / g0, rows) is a block of rows over kp positions (every box edge at most 256)
MK_HD inline int mmv_g0(int K, int kp) {
    int g0 = 8;
    while (g0 < 256 && K % (2 * g0) == 0 && kp % (2 * g0) == 0) g0 *= 2;
    return g0;
}
MK_HD inline int tmap_index(int op, int layer) {   // the tensor map of a matvec operator
    return op == OP_LMHEAD ? 4 * layer : 4 * layer + (op == OP_QKV ? 0 : op == OP_OPROJ ? 1 : op == OP_UPGATE ? 2 : 3);
}

// one instruction slot: words + where its stream sits + the matvec shape.  16-byte aligned and
// sized: the loader fills the words of each slot of the array with 16-byte stores
struct alignas(16) SlotInfo {
    int32_t w[kWords];
    int32_t first_page;      // global page sequence number of the stream's first page
    int32_t n_pages;
    int32_t first_slot;      // ring slot of the first page
    int32_t first_phase;     // mbarrier phase parity of the first page
    int64_t kv_off;          // attention: element offset of the chunk's first K/V row in the cache
    int32_t rows;            // matvec: rows (gate/up: pairs) of the tile
    int32_t inter;           // matvec: 1 = gate/up, pages alternate gate rows and up rows
    MvShape mv;              // matvec: the operator's shape
};
static_assert(sizeof(SlotInfo) % 16 == 0 && offsetof(SlotInfo, w) == 0, "slot words must stay 16-byte aligned");

// byte offsets of the non-ring shared memory (after the page ring); shared by host and device
struct MiscLayout {
    uint32_t slots, qwin, layers, bars, comb, combcnt, pubinfo, red, lmbest, qrot, kv, res, xbuf, total;
};

MK_HD inline MiscLayout misc_layout(int n_pages, int qrot_floats, int xbuf_floats, int comb_stride) {
    MiscLayout m{};
    uint32_t o = 0;
    auto take = [&o](uint32_t bytes, uint32_t align) {
        o = (o + align - 1) & ~(align - 1);
        const uint32_t r = o;
        o += bytes;
        return r;
    };
    m.slots = take(uint32_t(sizeof(SlotInfo)) * kSlots, 16);
    m.qwin = take(2u * kQWin * kWords * 4u, 16);
    m.layers = take(uint32_t(sizeof(LayerPtrs)) * kMaxLayersSmem, 16);
    m.bars = take(8u * (2u + 2u * uint32_t(n_pages) + 2u * kSlots + kDone + 3u), 8);  // qfull, full, empty, ins, done, cbar, xfull, xfree
    m.comb = take(4u * 4u * uint32_t(n_pages) * uint32_t(comb_stride), 16);   // partials per (page slot, phase, unit)
    m.combcnt = take(4u * 2u * uint32_t(n_pages), 16);                        // arrivals per (page slot, phase)
    m.pubinfo = take(4u * kDone * 8u, 16);            // completion words of in-flight instructions
    m.red = take(4u * 64u, 16);                     // argmax scratch [0..31]; abort flag [32], published count [33],
                                                    // stream bytes the loader has issued [34..35] (u64),
                                                    // stop flag [41],
                                                    // per-warp sums of squares of the shared input [48..63]
    m.lmbest = take(8u * kNumConsumerWarps * kMaxBatch, 8);   // LM-head running (max, index) per warp / sequence
    m.qrot = take(4u * uint32_t(qrot_floats), 16);
    m.kv = take(2u * 2u * kMaxHeadDim, 16);         // new k, v (bf16)
    m.res = take(4u * 2u * kResBuf, 16);            // residual words of the tile's rows, two buffers
    m.xbuf = take(4u * uint32_t(xbuf_floats), 16);  // shared matvec input (raw), one per CTA
    m.total = (o + 255u) & ~255u;
    return m;
}

// Batch > 1 matvec inputs staged in shared memory, one range of at most kMmvRange positions at a
// time: per sequence a row of mmv_row_stride(range) bytes holding a 32-bit word per position
// (fp32 as polled, then a bf16 (hi, lo) pair), rounded to 128 bytes plus 16: the eight lanes of
// a quarter warp read 16 bytes each at (sequence g in {2j, 2j + 1}, 32 t4 bytes into a 128-byte
// step), distinct bank quads only when consecutive rows start 16 bytes apart in the banks
// (measured at batch 8 against 64 bytes apart, a two-way conflict: 1645 -> 1621 us a step); after the rows, the partial sums of two
// 16-row blocks from the 8 consumer warps.  A thread polls at most kMmvItems 8-element chunks of
// a range per round.
constexpr int kMmvItems = 8;
MK_HD inline uint32_t mmv_row_stride(int K) { return ((uint32_t((K + 31) / 32) * 128u + 127u) & ~127u) + 16u; }
constexpr uint32_t kMmvPartBytes = 2u * kNumConsumerWarps * 16u * 8u * 4u;

inline int smem_misc_bytes(int n_pages, int qrot_floats, int xbuf_floats, int comb_stride) {
    return int(misc_layout(n_pages, qrot_floats, xbuf_floats, comb_stride).total);
}

// records a message for mk_last_error() and returns st
mk_status fail(mk_status st, const char* fmt, ...);

}  // namespace mk

// host schedule object
#include <vector>
struct mk_schedule {
    mk_model_cfg cfg;
    mk::Geometry geo;
    int32_t S, Q;
    std::vector<int32_t> queues;     // [S, Q, 32]
    std::vector<uint32_t> totals;    // [n_counters]
    int32_t max_pages;               // largest n_pages of any instruction
};
