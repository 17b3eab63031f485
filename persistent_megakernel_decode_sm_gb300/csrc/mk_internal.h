// Internal definitions shared by the library's translation units (scheduler, binding, kernel).
#pragma once

#include <stddef.h>
#include <stdint.h>
#include <vector_types.h>

#include "mk.h"

namespace mk {

// ---- instruction encoding ([S, Q, 32] int32, see mk_schedule_queues) ---------------------
enum Op : int32_t { OP_END = 0, OP_QKV = 1, OP_ATTN = 2, OP_COMB = 3, OP_OPROJ = 4, OP_UPGATE = 5,
                    OP_DOWN = 6, OP_LMHEAD = 7, OP_ARGMAX = 8, OP_COUNT = 9 };
enum Word : int {
    W_OP = 0, W_LAYER = 1, W_B = 2, W_A0 = 3, W_A1 = 4, W_A2 = 5, W_NWAIT = 6, W_WAIT = 7,
    W_NPUB = 15, W_PUB = 16, W_NPAGES = 20, W_TILE = 21, W_WAVE = 22
};
constexpr int kWords = 32;
constexpr int kMaxWait = 4;
constexpr int kMaxPub = 2;
constexpr int kMaxBatch = 8;
constexpr int kMaxRows = 8;        // rows of one matvec tile
constexpr int kMaxHpg = 8;         // query heads per KV head
constexpr int kMaxHeadDim = 128;
constexpr int kMaxK = 16384;       // longest matvec row (elements)
constexpr int64_t kTileOverhead = 1024;

// ---- resolved schedule parameters -----------------------------------------------------------
struct Geometry {
    int32_t page_bytes, tile_bytes, attn_chunk;
    int32_t r_qkv, r_o, r_up, r_dn, r_lm;    // rows (pairs for up) per tile
    int32_t n_qkv, n_o, n_up, n_dn, n_lm;    // tiles per layer (n_lm: LM head)
    int32_t n_chunk;                          // attention chunks per (sequence, group)
    int32_t n_counters;
    uint64_t shuffle_seed;
};

// counter ids
struct CounterMap {
    int32_t L, nkv, B, base2;
    explicit CounterMap(const mk_model_cfg& c)
        : L(c.n_layers), nkv(c.n_kv_heads), B(c.batch), base2(c.n_layers * c.n_kv_heads * (1 + c.batch)) {}
    int32_t qkv(int l, int g) const { return l * nkv + g; }
    int32_t attn(int l, int b, int g) const { return L * nkv + (l * B + b) * nkv + g; }
    int32_t comb(int l) const { return base2 + l; }
    int32_t o(int l) const { return base2 + L + l; }
    int32_t up(int l) const { return base2 + 2 * L + l; }
    int32_t down(int l) const { return base2 + 3 * L + l; }
    int32_t lm() const { return base2 + 4 * L; }
    int32_t fin() const { return base2 + 4 * L + 1; }
    int32_t count() const { return base2 + 4 * L + 2; }
};

// ---- scratch layout (fp32 activations unless noted), each region 256-byte aligned -----------
struct ScratchLayout {
    size_t err, tokens, x_attn, x_out, qkv, part, o, h, lm_part, rope, total;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

inline ScratchLayout scratch_layout(const mk_model_cfg& c, const Geometry& g) {
    const size_t L = c.n_layers, B = c.batch, H = c.hidden, d = c.head_dim;
    const size_t qd = size_t(c.n_q_heads) * d, kvd = size_t(c.n_kv_heads) * d;
    const size_t hpg = c.n_q_heads / c.n_kv_heads;
    ScratchLayout s{};
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t r = off; off = align256(off + bytes); return r; };
    s.err = take(256);            // int32 err[16] at 0, int32 tokens[8] at byte 64 (one readback)
    s.tokens = s.err + 64;
    s.x_attn = take(L * B * H * 4);
    s.x_out = take(L * B * H * 4);
    s.qkv = take(L * B * (qd + 2 * kvd) * 4);
    s.part = take(L * B * size_t(c.n_kv_heads) * g.n_chunk * hpg * (d + 2) * 4);
    s.o = take(L * B * qd * 4);
    s.h = take(L * B * size_t(c.ffn) * 4);
    s.lm_part = take(B * size_t(g.n_lm) * 8);
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

// ---- kernel parameters (passed by value) ----------------------------------------------------
struct Params {
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
    // scratch
    int32_t* err;
    int32_t* tokens_out;
    float* x_attn;
    float* x_out;
    float* qkv;
    float* part;
    float* o;
    float* h;
    float2* lm_part;   // (value, index bits)
    const float2* rope; // [max_seq][d/2] (cos, sin)
    // step
    uint32_t epoch;
    int32_t tok[kMaxBatch];
    int32_t pos[kMaxBatch];
    float* logits;
    int32_t* next_dev;
    uint64_t timeout_ns;
    // shared-memory carve-up
    int32_t smem_misc_off;   // byte offset of the non-ring area
    int32_t attn_scratch_floats;
};

// shared-memory layout of one CTA (after the page ring)
constexpr int kNumConsumerWarps = 8;
constexpr int kConsumerThreads = kNumConsumerWarps * 32;
constexpr int kLoaderWarp = 8;
constexpr int kPublisherWarp = 9;
constexpr int kThreads = 320;
constexpr int kSlots = 16;   // instruction slots in flight

struct SlotInfo {            // one instruction slot: words + where its stream sits in the ring
    int32_t w[kWords];
    int32_t first_page;
    int32_t n_pages;
    int32_t pad[2];
};

// bytes of the non-ring shared memory (slots, barriers, reduction and attention scratch)
inline int smem_misc_bytes(int n_pages, int attn_scratch_floats) {
    size_t b = 0;
    b += sizeof(SlotInfo) * kSlots;
    b += 8 * (2 * size_t(n_pages) + 3 * kSlots);   // mbarriers
    b += 4 * (2 * kNumConsumerWarps * kMaxRows);   // matvec reduction (double buffered)
    b += 4 * 64;                                   // norm reduction, flags, misc
    b += 4 * size_t(kMaxHpg) * kMaxHeadDim;        // rotated q
    b += 4 * size_t(attn_scratch_floats);          // scores / combine factors
    b += 2 * 2 * kMaxHeadDim;                      // new k, v (bf16)
    b += 4 * 2 * kMaxHpg * 2;                      // (m, l) per head, combine (M, L)
    return int(align256(b + 256));
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
