// The persistent decode megakernel (sm_103a).
//
// One CTA per SM interprets that SM's instruction queue (page "Inference MegaKernel", section
// "Hand-written whole-model MegaKernel": fetch instruction -> END? -> wait counters -> lease
// shared-memory pages -> run the operator body -> memory fence -> add completions -> release
// pages -> next).  On GB300 the loop is split over three warp roles so that weight streaming
// never waits on a dependency:
//   * loader warp (one thread): walks the queue ahead of the consumers, copies each
//     instruction into a shared-memory slot and leases the pages of its stream, filling them
//     with cp.async.bulk global->shared copies (evict-first L2 policy) completed on the page's
//     mbarrier.  Weights and old KV rows do not depend on any counter, so they are fetched
//     before the instruction's dependencies resolve -- the page ring absorbs dependency stalls.
//  * 8 consumer warps: learn that the instruction's inputs are ready, run the body on the leased
//     pages, release the pages (mbarrier arrive), write outputs, and hand the instruction to
//     the publisher.  By default (epoch-tagged activations) a consumer polls the tagged words it
//     reads until they carry this step's tag; inputs without a tag (the argmax's partials,
//     segmented 64-bit inputs) and the counters mode wait the instruction's counters instead
//     (one thread spins with relaxed loads, then an acquire fence).
//  * publisher warp (one thread): adds the completions to the global counters, after a
//     fence.release.gpu where a reader will rely on the counter (data first, then the fence,
//     then the counter: the page's data-visibility contract), without stalling the consumers.
// Every wait (counter spin, page / slot barrier) has a time budget; when it runs out the CTA
// records the error, all roles leave their loops, the loader drains its copies in flight and
// the kernel returns (no trap, no endless spin).
#include <cuda_runtime.h>
#include <stdint.h>

#include "mk_internal.h"

namespace mk {
#ifdef MK_BATCHED_TU
constexpr bool kBatchedKernel = true;    // this unit holds the batch > 1 kernel
#else
constexpr bool kBatchedKernel = false;
#endif

enum Role : int { ROLE_LOADER = 1, ROLE_CONSUMER = 2, ROLE_PUBLISHER = 3, ROLE_COUNTER = 4, ROLE_DATA = 5 };

// ------------------------------------------------------------------------- PTX helpers ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t tx) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_u32(bar)),
                 "r"(tx)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// waits up to ~hint_ns for the phase (the thread is suspended, not spinning; completion wakes it)
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
// one box of a 3-d TMA tensor map (coordinates innermost first) into shared memory
__device__ __forceinline__ void tma_load_3d(void* dst, const void* map, int c0, int c1, int c2, uint64_t* bar,
                                            uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// acquire / release halves of the counter protocol (cheaper than a full acq_rel fence)
__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acquire.gpu;" ::: "memory"); }
__device__ __forceinline__ void fence_release_gpu() { asm volatile("fence.release.gpu;" ::: "memory"); }
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ void red_add_relaxed_gpu(uint32_t* p, uint32_t v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// host-mapped words (a multi-step launch's control block): system-scope accesses
__device__ __forceinline__ int32_t ld_sys(const volatile int32_t* a) {
    int32_t v;
    asm volatile("ld.relaxed.sys.global.b32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ void st_sys(volatile int32_t* a, int32_t v) {
    asm volatile("st.relaxed.sys.global.b32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// epoch-tagged activation words (q/k/v, attention chunk partials): fp32 bits low, tag high, one
// single-copy-atomic 64-bit access
__device__ __forceinline__ void st_tag(uint64_t* a, float v, uint32_t tag) {
    const uint64_t w = (uint64_t(tag) << 32) | uint64_t(__float_as_uint(v));
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(a), "l"(w) : "memory");
}
__device__ __forceinline__ uint64_t ld_tag(const uint64_t* a) {
    uint64_t w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(a));
    return w;
}
// two consecutive words (16-byte aligned); each 64-bit element is read atomically
__device__ __forceinline__ void ld_tag2(const uint64_t* a, uint64_t& w0, uint64_t& w1) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(w0), "=l"(w1) : "l"(a));
}
__device__ __forceinline__ float tag_val(uint64_t w) { return __uint_as_float(uint32_t(w)); }
__device__ __forceinline__ uint32_t tag_of(uint64_t w) { return uint32_t(w >> 32); }
// eight consecutive tagged elements (64-byte aligned): values into v, true when all carry `tag`
__device__ __forceinline__ bool ld8_tagged(const uint64_t* a, float* v, uint32_t tag) {
    uint64_t w[8];
    ld_tag2(a, w[0], w[1]);
    ld_tag2(a + 2, w[2], w[3]);
    ld_tag2(a + 4, w[4], w[5]);
    ld_tag2(a + 6, w[6], w[7]);
    bool ok = true;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        v[e] = tag_val(w[e]);
        ok &= tag_of(w[e]) == tag;
    }
    return ok;
}

// The SwiGLU output is read by the down projection a whole 2048-element segment per warp, where
// 64-bit words would not fit the registers next to x, and the residual streams and the attention
// output are read whole by every SM, where half the bytes shorten every poll (measured: batch-8
// step 1807 -> 1726 us, batch-1 708 -> 691 us): their elements are 32-bit words, fp32 with
// the three low mantissa bits replaced by a 3-bit step tag, (epoch mod 7) + 1 -- never 0 (the
// cleared scratch) and never the previous step's.  The stored value is the fp32 result with those
// bits cleared (a relative change below 2^-20).
__device__ __forceinline__ uint32_t htag(uint32_t tag) { return (tag - 1u) % 7u + 1u; }
__device__ __forceinline__ void st_htag(uint32_t* a, float v, uint32_t ht) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(a), "r"((__float_as_uint(v) & ~7u) | ht) : "memory");
}
// eight consecutive h-tagged elements (32-byte aligned): values into v, true when all carry ht
__device__ __forceinline__ bool ld8_htagged(const uint32_t* a, float* v, uint32_t ht) {
    uint32_t w[8];
    asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "l"(a));
    asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7]) : "l"(a + 4));
    uint32_t bad = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        v[e] = __uint_as_float(w[e] & ~7u);
        bad |= w[e] ^ ht;
    }
    return (bad & 7u) == 0;
}

// whole-CTA barrier reached by warps whose lanes diverged (loader / publisher lane 0 arrives late)
__device__ __forceinline__ void cta_sync_divergent() { asm volatile("barrier.sync 0;" ::: "memory"); }

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }
__device__ __forceinline__ uint16_t f2bf_rn(float f) {   // round to nearest even (finite inputs)
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7F800000u) == 0x7F800000u) return uint16_t((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
    u += 0x7FFFu + ((u >> 16) & 1u);
    return uint16_t(u >> 16);
}
__device__ __forceinline__ float dot8(uint4 w, const float* x, float acc) {
    acc = fmaf(bf_lo(w.x), x[0], acc);
    acc = fmaf(bf_hi(w.x), x[1], acc);
    acc = fmaf(bf_lo(w.y), x[2], acc);
    acc = fmaf(bf_hi(w.y), x[3], acc);
    acc = fmaf(bf_lo(w.z), x[4], acc);
    acc = fmaf(bf_hi(w.z), x[5], acc);
    acc = fmaf(bf_lo(w.w), x[6], acc);
    acc = fmaf(bf_hi(w.w), x[7], acc);
    return acc;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// optional per-instruction timeline: [0] slot published by the loader, [1] its pages issued,
// [2] dependencies satisfied, [3] body done, [4] completions published, [5] CTA start
__device__ __forceinline__ void stamp(const Params& p, int pc, int k) {
    if (p.trace) p.trace[(size_t(blockIdx.x) * p.Q + pc) * kTraceWords + k] = globaltimer();
}

// ------------------------------------------------------------------------- shared memory ----
struct Shared {
    uint8_t* ring;
    SlotInfo* slots;
    int32_t* qwin;     // [2][kQWin][32] queue window
    LayerPtrs* layers; // [L]
    uint64_t* qfull;   // [2]
    uint64_t* full;    // [n_pages]
    uint64_t* empty;   // [n_pages]
    uint64_t* ins_full;
    uint64_t* ins_empty;
    uint64_t* done;
    uint64_t* cbar;    // consumer-warp barrier (16 arrivals)
    uint64_t* xfull;   // shared input written (16 arrivals)
    uint64_t* xfree;   // shared input taken by every warp (16 arrivals)
    float* xbuf;       // [xbuf_floats] shared matvec input
    float* res;        // [2][kResBuf] residual words of a tile's rows
    float* comb;       // [n_pages][2 phases][comb_stride][2] row-segment partials
    int* combcnt;      // [n_pages][2 phases] arrivals of the warps on a page group
    int* pubinfo;      // [kDone][8]: opcode, #completions, (counter, delta) x 2
    float* red;        // [32] argmax scratch
    float2* lmbest;    // [kNumConsumerWarps][kMaxBatch] LM-head running (max, index) of the CTA's tiles
    int* abort;        // [1]
    int* stop;         // [1] a multi-step launch ends at a step boundary (not an error)
    int* published;    // [1] instructions the publisher has retired
    unsigned long long* issued;   // [1] stream bytes the loader has staged into pages
    float* qrot;       // [8][128]
    uint16_t* knew;    // [128]
    uint16_t* vnew;    // [128]
};

__device__ __forceinline__ Shared carve(uint8_t* base, const Params& p) {
    const MiscLayout m = misc_layout(p.n_pages, p.qrot_floats, p.xbuf_floats, p.comb_stride);
    uint8_t* b = base + p.smem_misc_off;
    Shared s;
    s.ring = base;
    s.slots = reinterpret_cast<SlotInfo*>(b + m.slots);
    s.qwin = reinterpret_cast<int32_t*>(b + m.qwin);
    s.layers = reinterpret_cast<LayerPtrs*>(b + m.layers);
    s.qfull = reinterpret_cast<uint64_t*>(b + m.bars);
    s.full = s.qfull + 2;
    s.empty = s.full + p.n_pages;
    s.ins_full = s.empty + p.n_pages;
    s.ins_empty = s.ins_full + kSlots;
    s.done = s.ins_empty + kSlots;
    s.cbar = s.done + kDone;
    s.xfull = s.cbar + 1;
    s.xfree = s.cbar + 2;
    s.xbuf = reinterpret_cast<float*>(b + m.xbuf);
    s.res = reinterpret_cast<float*>(b + m.res);
    s.comb = reinterpret_cast<float*>(b + m.comb);
    s.combcnt = reinterpret_cast<int*>(b + m.combcnt);
    s.pubinfo = reinterpret_cast<int*>(b + m.pubinfo);
    s.red = reinterpret_cast<float*>(b + m.red);
    s.lmbest = reinterpret_cast<float2*>(b + m.lmbest);
    s.abort = reinterpret_cast<int*>(b + m.red) + 32;
    s.stop = reinterpret_cast<int*>(b + m.red) + 41;
    s.published = reinterpret_cast<int*>(b + m.red) + 33;
    s.issued = reinterpret_cast<unsigned long long*>(reinterpret_cast<int*>(b + m.red) + 34);
    s.qrot = reinterpret_cast<float*>(b + m.qrot);
    s.knew = reinterpret_cast<uint16_t*>(b + m.kv);
    s.vnew = s.knew + kMaxHeadDim;
    return s;
}

__device__ void raise_error(const Params& p, const Shared& sh, int code, int role, int pc, int counter,
                            uint32_t have, uint32_t want) {
    if (atomicCAS(p.err, 0, code) == 0) {
        p.err[1] = blockIdx.x;
        p.err[2] = pc;
        p.err[3] = counter;
        p.err[4] = int(have);
        p.err[5] = int(want);
        p.err[6] = role;
        __threadfence();
    }
    *reinterpret_cast<volatile int*>(sh.abort) = 1;
}

// Time budget of a wait by its role.  Waits that can name the cause of a stall (a counter, a
// tagged element) get the configured budget; waits on this CTA's own consumers (consumer
// barriers) twice that, and the loader's and publisher's waits, which only follow the consumers,
// four times: the wait closest to the cause runs out first and is the one recorded.
__device__ __forceinline__ uint64_t budget(const Params& p, int role) {
    return role == ROLE_LOADER || role == ROLE_PUBLISHER ? 4ull * p.timeout_ns
         : role == ROLE_CONSUMER ? 2ull * p.timeout_ns : p.timeout_ns;
}

// bounded mbarrier wait: false when the CTA aborts or the budget runs out (error recorded)
// (the waiting thread sleeps in hardware between checks of the abort flag and the time budget)
__device__ __noinline__ bool wait_bar_slow(const Params& p, const Shared& sh, uint64_t* bar, uint32_t parity, int role,
                                           int pc) {
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*reinterpret_cast<volatile int*>(sh.abort) || *reinterpret_cast<volatile int*>(sh.stop)) return false;
        if (globaltimer() - t0 > budget(p, role)) {
            raise_error(p, sh, MK_ERR_TIMEOUT, role, pc, -1, 0, 0);
            return false;
        }
    }
}
__device__ __forceinline__ bool wait_bar(const Params& p, const Shared& sh, uint64_t* bar, uint32_t parity, int role,
                                         int pc) {
    return mbar_try_wait(bar, parity) || wait_bar_slow(p, sh, bar, parity, role, pc);
}

// ------------------------------------------------------------------------- streams ----------
struct Seg {
    const uint8_t* src;
    uint32_t off, bytes;   // offset of the segment inside the tile's stream
};
struct Stream {
    int64_t kv_off;                  // attention: element offset of the chunk's first K/V row
    Seg seg[2];
    int nseg;
    uint32_t total;
    int pages;
    int inter;                       // gate/up tile: page 2j = gate rows [j rpp, (j+1) rpp), 2j+1 = up rows
    uint32_t rows, rowbytes, rpp;    // matvec: whole rows per page (0 rows: a plain byte stream)
    uint32_t K, nblk;                // batch > 1: row length, 16-row blocks (gate/up: 8 pairs),
    uint32_t row0, g0, up;           // first row, innermost box edge, row offset of the up rows
    uint32_t r0;                     // the first staging range (a down tile of one range: its range)
    const uint8_t* tmap;             // and the weights' tensor map
};

__device__ __forceinline__ int attn_old_rows(const Params& p, int b, int c, int chunk, int dpos) {
    const int pos = p.pos[b] + dpos;
    const int c0 = c * chunk;
    if (c0 > pos) return -1;                 // chunk past pos: inactive
    return min(c0 + chunk, pos) - c0;        // cached positions strictly before pos
}

// Element offset of the first K/V row of attention chunk c (positions [c C, c C + C)) of
// sequence b, layer l, KV head g.  Contiguous cache: rows of a head are consecutive.  Paged cache:
// the chunk is one block of the pool, found through the block table; false when the table entry
// is outside the pool (nothing is read or written then).
__device__ __forceinline__ bool kv_chunk_off(const Params& p, int b, int l, int g, int c, int C, int64_t& off) {
    if (!p.kv_table) {
        off = int64_t(b) * p.kv_bstride + int64_t(l) * p.kv_lstride + int64_t(g) * p.kv_hstride + int64_t(c) * C * p.d;
        return true;
    }
    const int blk = __ldg(p.kv_table + size_t(b) * p.kv_max_blocks + c);
    if (unsigned(blk) >= unsigned(p.kv_n_blocks)) return false;
    off = int64_t(l) * p.kv_lstride + int64_t(g) * p.kv_hstride + int64_t(blk) * C * p.d;
    return true;
}

__device__ __forceinline__ const uint8_t* word_ptr(const int32_t* w) {
    return reinterpret_cast<const uint8_t*>((uint64_t(uint32_t(w[1])) << 32) | uint64_t(uint32_t(w[0])));
}
__device__ __forceinline__ bool is_matvec(int op) {
    return op == OP_QKV || op == OP_OPROJ || op == OP_UPGATE || op == OP_DOWN || op == OP_LMHEAD;
}

// The bytes an instruction's body streams.  Matvec tiles carry their resolved weight stream in
// words 26..31 (written and validated at bind); an attention chunk's cached KV rows depend on pos
// and are computed here (with the chunk's bounds checked).  Returns an mk_status.
__device__ int stream_of(const Params& p, const int32_t* w, Stream& st, int dpos) {
    st.nseg = 0;
    st.total = 0;
    st.pages = 0;
    st.kv_off = 0;
    st.inter = 0;
    st.rows = st.rowbytes = st.rpp = 0;
    st.K = st.nblk = st.row0 = st.g0 = st.up = st.r0 = 0;
    st.tmap = nullptr;
    const int op = w[W_OP];
    if (is_matvec(op)) {   // whole rows per page; gate/up: gate and up row groups in alternate pages
        const uint32_t b0 = uint32_t(w[W_BYTES0]), b1 = uint32_t(w[W_BYTES1]);
        st.seg[0] = {word_ptr(w + W_SRC0), 0u, b0};
        st.seg[1] = {word_ptr(w + W_SRC1), b0, b1};
        st.nseg = b1 ? 2 : 1;
        st.total = b0 + b1;
        st.inter = op == OP_UPGATE;
        st.rows = uint32_t(w[W_A1]);
        st.rowbytes = p.mv[op].rowbytes;
        st.rpp = uint32_t(p.mv[op].rpp);
        if (b0 == 0 || st.rpp == 0 || b0 != st.rows * st.rowbytes || b1 != (st.inter ? b0 : 0u)) return MK_ERR_BOUNDS;
        if (kBatchedKernel) {   // 16-row blocks over mmv_kp positions per page, through the tensor map
            st.K = uint32_t(p.mv[op].K);
            st.nblk = (st.rows + (st.inter ? 7u : 15u)) / (st.inter ? 8u : 16u);
            st.pages = int(mv_tile_pages(p.mv[op], p.mmv_kp, st.rows, st.inter));
            if (op == OP_DOWN && mmv_down_ranges(p.B, p.F) > 1) {   // one staging range of the rows
                st.r0 = uint32_t(w[W_A2]);
                if (st.r0 >= uint32_t(mmv_down_ranges(p.B, p.F))) return MK_ERR_BOUNDS;
                st.pages = int(mmv_range_pages(int(st.K), p.mmv_kp, st.rows, int(st.r0)));
            }
            st.row0 = uint32_t(w[W_A0]);
            st.g0 = uint32_t(mmv_g0(int(st.K), p.mmv_kp));
            st.up = uint32_t(p.F);
            st.tmap = p.tmaps + size_t(tmap_index(op, w[W_LAYER])) * 128u;
        } else {
            st.pages = int((st.rows + st.rpp - 1u) / st.rpp) * (st.inter ? 2 : 1);
        }
        if (st.pages > w[W_NPAGES]) return MK_ERR_CAPACITY;   // (matvec tiles stream through the ring)
        return MK_OK;
    } else if (op == OP_ATTN) {
        const int l = w[W_LAYER], b = w[W_B], g = w[W_A0], c = w[W_A1], C = w[W_A2];
        if (unsigned(l) >= unsigned(p.L) || unsigned(b) >= unsigned(p.B) || unsigned(g) >= unsigned(p.nkv) ||
            unsigned(c) >= unsigned(p.n_chunk) || C != p.attn_chunk)
            return MK_ERR_BOUNDS;
        const int n_old = attn_old_rows(p, b, c, C, dpos);
        if (n_old >= 0 && !kv_chunk_off(p, b, l, g, c, C, st.kv_off)) return MK_ERR_BOUNDS;
        if (n_old > 0) {
            const size_t base = size_t(st.kv_off);
            const uint32_t nb = uint32_t(n_old * p.d * 2);
            st.seg[0] = {reinterpret_cast<const uint8_t*>(p.kc + base), 0u, nb};
            st.seg[1] = {reinterpret_cast<const uint8_t*>(p.vc + base), nb, nb};
            st.nseg = 2;
            st.total = 2 * nb;
        }
    } else if (op != OP_ARGMAX && op != OP_END && !(kBatchedKernel && op == OP_COMB)) {
        return MK_ERR_OPCODE;
    }
    st.pages = int((st.total + uint32_t(p.page_bytes) - 1u) >> p.page_shift);
    // an attention tile's consumers hold all its pages at once: it must fit the ring
    if (st.pages > w[W_NPAGES] || (op == OP_ATTN && st.pages > p.n_pages)) return MK_ERR_CAPACITY;
    return MK_OK;
}

// ------------------------------------------------------------------------- loader -----------
// Page pg of a matvec stream: its source and bytes (whole rows; a gate/up tile alternates gate
// pages and up pages of the same row group).
__device__ __forceinline__ const uint8_t* mv_page(const Stream& st, uint32_t pg, uint32_t& bytes) {
    const uint32_t r0 = (st.inter ? pg >> 1 : pg) * st.rpp;
    bytes = min(st.rpp, st.rows - r0) * st.rowbytes;
    return ((st.inter && (pg & 1u)) ? st.seg[1].src : st.seg[0].src) + size_t(r0) * st.rowbytes;
}

// Another CTA's error reaches this CTA through the global error word; reading it costs a memory
// round trip, so a poll reads it only every kErrCheckRounds rounds (its own CTA's abort flag, in
// shared memory, every round).
constexpr uint32_t kErrCheckRounds = 64;
__device__ __forceinline__ bool other_cta_failed(const Params& p, uint32_t& rounds) {
    return (++rounds % kErrCheckRounds) == 0 && ld_relaxed_gpu(reinterpret_cast<const uint32_t*>(p.err)) != 0;
}

// The loader's side of a step boundary: before the first copy of KV-cache rows in step s > 0 of a
// multi-step launch (rows the previous step wrote), every CTA has retired that step and the
// writes are acquired, then ordered before this thread's bulk (async-proxy) reads.  Weight pages
// need no wait, so a step's first matvec pages stream in while the consumers are still in the
// previous step.  False: stop, abort or timeout.
__device__ bool loader_boundary(const Params& p, const Shared& sh, int s, int pc) {
    const uint32_t target = (p.epoch + uint32_t(s)) * gridDim.x;
    const uint64_t t0 = globaltimer();
    uint32_t rounds = 0;
    while (int32_t(ld_relaxed_gpu(p.step_bar) - target) < 0) {
        __nanosleep(100);
        if (*reinterpret_cast<volatile int*>(sh.abort) || *reinterpret_cast<volatile int*>(sh.stop)) return false;
        if (other_cta_failed(p, rounds)) {
            *reinterpret_cast<volatile int*>(sh.abort) = 1;
            return false;
        }
        if (globaltimer() - t0 > p.timeout_ns) {
            raise_error(p, sh, MK_ERR_TIMEOUT, ROLE_LOADER, pc, -1, ld_relaxed_gpu(p.step_bar), target);
            return false;
        }
    }
    fence_acquire_gpu();
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

__device__ void loader(const Params& p, const Shared& sh) {
    const int32_t* q = p.queues + size_t(blockIdx.x) * p.Q * kWords;
    const uint64_t pol = evict_first_policy();
    const uint32_t PB = uint32_t(p.page_bytes);
    const uint32_t NP = uint32_t(p.n_pages);
    const int n_chunks = (p.Q + kQWin - 1) / kQWin;
    // The queue is read through a two-buffer shared-memory window, kQWin instructions per bulk
    // copy; a multi-step launch reads it once per step.  Window fetches, instruction slots and
    // completion records are indexed by running counts over all steps.
    int qf = 0;                              // window fetches issued so far
    auto fetch_chunk = [&](int chunk) {
        const int n = min(kQWin, p.Q - chunk * kQWin);
        uint64_t* bar = sh.qfull + (qf & 1);
        mbar_arrive_expect_tx(bar, uint32_t(n * kWords * 4));
        bulk_g2s(sh.qwin + (qf & 1) * kQWin * kWords, q + size_t(chunk) * kQWin * kWords, uint32_t(n * kWords * 4),
                 bar, pol);
        ++qf;
    };
    uint32_t gi = 0;                         // instructions published so far
    uint32_t page_seq = 0;                   // pages issued so far
    uint32_t cur_slot = 0, cur_phase = 0;    // ring slot and phase parity of the next page
    bool stop = false;
    int bar_seen = 0;                        // the last step whose boundary this thread has acquired
    for (int s = 0; s < p.n_steps && !stop; ++s) {
        const int f0 = qf;                   // fetch index of this step's chunk 0
        if (s > 0) fence_proxy_async_smem();   // the previous step's generic reads of both buffers
        fetch_chunk(0);
        if (n_chunks > 1) fetch_chunk(1);
        int chunks_issued = n_chunks > 1 ? 2 : 1;
        int chunks_waited = 0;
        for (int pc = 0; pc < p.Q; ++pc) {
            const uint32_t g = gi++;
            const int slot = int(g % kSlots);
            const int chunk = pc / kQWin;
            const int fi = f0 + chunk;       // this chunk's fetch: buffer fi & 1, phase (fi >> 1) & 1
            if (pc % kQWin == 0) {
                if (!wait_bar(p, sh, sh.qfull + (fi & 1), (fi >> 1) & 1, ROLE_LOADER, pc)) { stop = true; break; }
                chunks_waited = chunk + 1;
            }
            if (g >= uint32_t(kSlots) && !wait_bar(p, sh, sh.ins_empty + slot, ((g / kSlots) - 1) & 1, ROLE_LOADER, pc)) {
                stop = true;
                break;
            }
            SlotInfo& si = sh.slots[slot];
            const int4* src = reinterpret_cast<const int4*>(sh.qwin + ((fi & 1) * kQWin + pc % kQWin) * kWords);
#pragma unroll
            for (int i = 0; i < kWords / 4; ++i) reinterpret_cast<int4*>(si.w)[i] = src[i];
            if (pc % kQWin == kQWin - 1 && chunks_issued < n_chunks) {
                fence_proxy_async_smem();   // generic reads of this buffer before the async refill
                fetch_chunk(chunks_issued++);
            }
            Stream st;
            const int e = stream_of(p, si.w, st, s);
            if (e != MK_OK) {
                raise_error(p, sh, e, ROLE_LOADER, pc, -1, uint32_t(si.w[W_OP]), 0);
                stop = true;
                break;
            }
            if (s > bar_seen && st.pages > 0 && !st.rows) {   // KV rows: after the step boundary
                if (!loader_boundary(p, sh, s, pc)) { stop = true; break; }
                bar_seen = s;
            }
            si.first_page = int32_t(page_seq);
            si.n_pages = st.pages;
            si.kv_off = st.kv_off;
            si.first_slot = int32_t(cur_slot);
            si.first_phase = int32_t(cur_phase);
            if (is_matvec(si.w[W_OP])) {   // shape of the op (bind-time table) and of this tile
                si.rows = int32_t(st.rows);
                si.inter = st.inter;
                si.mv = p.mv[si.w[W_OP]];
            }
            {   // completion words for the publisher, which may lag up to kDone instructions behind
                const uint64_t t0 = globaltimer();
                while (int(g) - *reinterpret_cast<volatile int*>(sh.published) >= kDone) {
                    __nanosleep(200);
                    if (*reinterpret_cast<volatile int*>(sh.abort) || *reinterpret_cast<volatile int*>(sh.stop)) {
                        stop = true;
                        break;
                    }
                    if (globaltimer() - t0 > budget(p, ROLE_LOADER)) {
                        raise_error(p, sh, MK_ERR_TIMEOUT, ROLE_LOADER, pc, -1, 0, 0);
                        stop = true;
                        break;
                    }
                }
                if (stop) break;
                int* pi = sh.pubinfo + (g % kDone) * 8;
                pi[0] = si.w[W_OP];
                pi[1] = si.w[W_NPUB];
#pragma unroll
                for (int i = 0; i < 4; ++i) pi[2 + i] = si.w[W_PUB + i];
                pi[6] = si.w[W_COND];   // 1: completions only if the consumer marks the tile as the group's last
                pi[7] = 0;              // set by the consumer: this tile completed its group
            }
            stamp(p, pc, 0);
            mbar_arrive(sh.ins_full + slot);   // release: the slot's words are visible to the consumers
            if (si.w[W_OP] == OP_END) break;
            for (int pg = 0; pg < st.pages; ++pg) {
                const uint32_t ps = cur_slot;
                if (page_seq >= NP && !wait_bar(p, sh, sh.empty + ps, cur_phase ^ 1u, ROLE_LOADER, pc)) {
                    stop = true;
                    break;
                }
                uint8_t* dst = sh.ring + (size_t(ps) << p.page_shift);
                if (kBatchedKernel && st.rows) {
                    // batch > 1: block q of rows (gate/up: 8 gate rows, then the same pairs' up rows)
                    // over the kp positions of slice sl; pages in the order (range, block, slice)
                    const uint32_t kp = uint32_t(p.mmv_kp), nsr = uint32_t(kMmvRange) / kp;
                    const uint32_t nsl = (st.K + kp - 1u) / kp, per_r = st.nblk * nsr;
                    const uint32_t r = st.r0 + uint32_t(pg) / per_r, rem = uint32_t(pg) % per_r;
                    const uint32_t nsl_r = min(nsr, nsl - r * nsr);
                    const uint32_t q = rem / nsl_r, sl = r * nsr + rem % nsl_r;
                    // one tensor box per page (gate/up: the 8 gate rows, then the same pairs' up
                    // rows); a box counts its full size, positions past K and rows past the matrix
                    // read as zeros
                    const int c1 = int((sl * kp) / st.g0), row = int(st.row0 + q * (st.inter ? 8u : 16u));
                    mbar_arrive_expect_tx(sh.full + ps, uint32_t(p.page_bytes));
                    tma_load_3d(dst, st.tmap, 0, c1, row, sh.full + ps, pol);
                    if (st.inter) tma_load_3d(dst + 8u * kp * 2u, st.tmap, 0, c1, row + int(st.up), sh.full + ps, pol);
                } else if (st.rows) {   // matvec: a group of whole rows (gate/up: gate rows on even pages, up rows on odd)
                    uint32_t bytes;
                    const uint8_t* psrc = mv_page(st, uint32_t(pg), bytes);
                    mbar_arrive_expect_tx(sh.full + ps, bytes);
                    bulk_g2s(dst, psrc, bytes, sh.full + ps, pol);
                } else {
                    const uint32_t lo = uint32_t(pg) * PB;
                    const uint32_t hi = min(lo + PB, st.total);
                    mbar_arrive_expect_tx(sh.full + ps, hi - lo);
#pragma unroll
                    for (int sg = 0; sg < 2; ++sg) {   // (static indexes: the stream stays in registers)
                        if (sg >= st.nseg) break;
                        const uint32_t a = max(lo, st.seg[sg].off);
                        const uint32_t z = min(hi, st.seg[sg].off + st.seg[sg].bytes);
                        if (a < z) bulk_g2s(dst + (a - lo), st.seg[sg].src + (a - st.seg[sg].off), z - a, sh.full + ps, pol);
                    }
                }
                ++page_seq;
                if (++cur_slot == NP) { cur_slot = 0; cur_phase ^= 1u; }
            }
            if (stop) break;
            stamp(p, pc, 1);
            *reinterpret_cast<volatile unsigned long long*>(sh.issued) += st.total;
        }
        // this step's window copies still in flight (prefetched past END, or abandoned): the next
        // step (or the exit) reuses the buffers
        for (int cch = chunks_waited; cch < chunks_issued; ++cch) {
            const int fi = f0 + cch;
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(sh.qfull + (fi & 1), (fi >> 1) & 1))
                if (globaltimer() - t0 > 1000000000ull) break;   // copies always land; 1 s cap
        }
    }
    {   // drain: wait for the last copy issued into every page so no bulk copy outlives the CTA (after
        // an abort, or a stop at a step boundary, the consumers may never take those pages; after a
        // normal end these waits find completed phases)
        const uint32_t first = page_seq > NP ? page_seq - NP : 0;
        for (uint32_t k = first; k < page_seq; ++k) {
            const uint32_t ps = k % NP;
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(sh.full + ps, (k / NP) & 1)) {
                if (globaltimer() - t0 > 1000000000ull) break;   // copies always land; 1 s cap
            }
        }
    }
}

// ------------------------------------------------------------------------- publisher --------
__device__ void publisher(const Params& p, const Shared& sh) {
    // Retires instructions in queue order.  Every instruction the consumer warps have finished is
    // taken into one batch: one release fence, then one add per distinct counter.  The publisher
    // owns its own completion ring (kDone deep), so a slow fence never holds up the loader.
    constexpr int kBatch = 32;
    int pc = 0;     // instructions retired over all steps (the completion ring's index)
    int qpc = 0;    // queue index of instruction pc within its step
    int ends = 0;   // steps retired (an END closes a step)
    while (ends < p.n_steps) {
        if (!wait_bar(p, sh, sh.done + (pc % kDone), (pc / kDone) & 1, ROLE_PUBLISHER, pc)) break;
        int n = 1;
        while (n < kBatch && sh.pubinfo[((pc + n - 1) % kDone) * 8] != OP_END &&
               mbar_test_wait(sh.done + ((pc + n) % kDone), ((pc + n) / kDone) & 1))
            ++n;
        // pass 1: the batch's extent (END closes it), whether it needs the release fence, and
        // whether it adds anything at all
        bool release = p.sync_counters != 0, any = false;
        for (int i = 0; i < n; ++i) {
            const int* pi = sh.pubinfo + ((pc + i) % kDone) * 8;
            if (pi[0] == OP_END) { n = i + 1; break; }
            release |= (p.release_ops >> pi[0]) & 1;   // its output is read after an acquire, untagged
            any |= pi[1] > 0 && !(pi[6] && !pi[7]);
        }
        // counters mode (and outputs read untagged): everything the consumers wrote for these
        // instructions, then the counters.  Otherwise the data is tagged: no fence
        if (any && release) fence_release_gpu();
        // pass 2: the adds, one per run of completions to the same counter (queue order keeps
        // the tiles of one operator together), accumulated in registers
        int run_c = -1;
        uint32_t run_d = 0;
        for (int i = 0; i < n; ++i) {
            const int* pi = sh.pubinfo + ((pc + i) % kDone) * 8;
            if (pi[0] == OP_END) break;
            if (pi[6] && !pi[7]) continue;   // conditional completion not fired by this tile
            for (int k = 0; k < pi[1]; ++k) {
                const int c = pi[2 + 2 * k];
                if (c != run_c) {
                    if (run_c >= 0) red_add_relaxed_gpu(p.counters + run_c, run_d);
                    run_c = c;
                    run_d = 0;
                }
                run_d += uint32_t(pi[3 + 2 * k]);
            }
        }
        if (run_c >= 0) red_add_relaxed_gpu(p.counters + run_c, run_d);
        if (p.trace)
            for (int i = 0; i < n; ++i) stamp(p, qpc + i, 4);
        const bool end = sh.pubinfo[((pc + n - 1) % kDone) * 8] == OP_END;
        if (end) {
            // the step is retired in this CTA: every consumer warp arrived on the END record after its
            // last tile.  A next step in this launch reads what they wrote once the step word shows
            // every CTA, so this CTA's writes are released first (cumulative over the CTA's warps)
            if (ends + 1 < p.n_steps) fence_release_gpu();
            red_add_relaxed_gpu(p.step_bar, 1u);
        }
        pc += n;
        qpc = end ? 0 : qpc + n;
        ends += end ? 1 : 0;
        *reinterpret_cast<volatile int*>(sh.published) = pc;
    }
}

// ------------------------------------------------------------------------- consumer warps ---
// The 16 consumer warps walk the instruction stream independently.  A matvec tile needs one
// consumer barrier per input vector (every warp takes its segment of the input once it is
// complete in shared memory) and none per row: warp w computes segment w mod G of the rows of
// each page group, with its segment of the input in registers; the G segment sums of a row meet
// in shared memory, where the last-arriving warp adds them in segment order and writes the row.
// Attention and argmax cooperate through an mbarrier-based consumer barrier whose waits are
// bounded and give up when the CTA aborts.

struct Cw {
    const Params& p;
    const Shared& sh;
    int warp, lane;
    uint32_t cb_phase;   // consumer-barrier uses so far
    uint32_t xphase;     // input loads so far
    // the step this warp is in: a launch runs p.n_steps steps, step s at epoch p.epoch + s (tag
    // one more) with every position advanced by s
    int32_t step;
    uint32_t epoch, tag;
};

__device__ __forceinline__ const uint8_t* ring_ptr(const Shared& sh, const Params& p, uint32_t first_slot, uint32_t off) {
    uint32_t s = first_slot + (off >> p.page_shift);
    if (s >= uint32_t(p.n_pages)) s -= uint32_t(p.n_pages);
    return sh.ring + (size_t(s) << p.page_shift) + (off & (uint32_t(p.page_bytes) - 1u));
}

// Every warp waits for every page of the instruction before it may release them: an early
// release could otherwise count toward the previous use of the same page slot.
__device__ bool wait_pages(const Cw& c, const SlotInfo& si, int pc) {
    uint32_t slot = uint32_t(si.first_slot), ph = uint32_t(si.first_phase);
    for (int i = 0; i < si.n_pages; ++i) {
        if (!wait_bar(c.p, c.sh, c.sh.full + slot, ph, ROLE_CONSUMER, pc)) return false;
        if (++slot == uint32_t(c.p.n_pages)) { slot = 0; ph ^= 1u; }
    }
    return true;
}
__device__ void release_pages(const Cw& c, const SlotInfo& si) {
    __syncwarp();
    if (c.lane == 0) {
        uint32_t slot = uint32_t(si.first_slot);
        for (int i = 0; i < si.n_pages; ++i) {
            mbar_arrive(c.sh.empty + slot);
            if (++slot == uint32_t(c.p.n_pages)) slot = 0;
        }
    }
}

// barrier over the 8 consumer warps; false when the CTA aborted while waiting
__device__ bool cbar(Cw& c, int pc) {
    __syncwarp();
    if (c.lane == 0) mbar_arrive(c.sh.cbar);
    const bool ok = wait_bar(c.p, c.sh, c.sh.cbar, c.cb_phase & 1u, ROLE_CONSUMER, pc);
    ++c.cb_phase;
    __syncwarp();
    return ok;
}

// Bounded wait on tagged data, by a whole warp: call after a poll in which some lane did not yet
// see this step's tag.  False (warp-uniform) once the CTA aborts, another CTA has recorded an
// error, or the time budget runs out (then the timeout is recorded here).
struct Spin {
    uint64_t t0 = 0;
    bool started = false;
    uint32_t rounds = 0;
};
__device__ bool spin_more(const Params& p, const Shared& sh, int lane, Spin& sp, int pc, uint32_t tag) {
    int stop = 0;
    if (lane == 0) {
        if (*reinterpret_cast<volatile int*>(sh.abort) || other_cta_failed(p, sp.rounds)) {
            *reinterpret_cast<volatile int*>(sh.abort) = 1;
            stop = 1;
        } else {
            const uint64_t now = globaltimer();
            if (!sp.started) {
                sp.t0 = now;
                sp.started = true;
            } else if (now - sp.t0 > p.timeout_ns) {
                raise_error(p, sh, MK_ERR_TIMEOUT, ROLE_DATA, pc, -1, 0, tag);
                stop = 1;
            }
            if (!stop) __nanosleep(kPollBackoffNs);   // (yields the issue slot between polling rounds)
        }
    }
    return __shfl_sync(0xFFFFFFFFu, stop, 0) == 0;
}
__device__ __forceinline__ bool spin_more(const Cw& c, Spin& sp, int pc) { return spin_more(c.p, c.sh, c.lane, sp, pc, c.tag); }
// warp-wide: lanes with `valid` read the tagged words a0 and a1 until both carry this step's tag
__device__ bool wpoll2(const Cw& c, bool valid, const uint64_t* a0, const uint64_t* a1, float& v0, float& v1, int pc) {
    Spin sp;
    while (true) {
        bool ok = true;
        if (valid) {
            const uint64_t w0 = ld_tag(a0), w1 = ld_tag(a1);
            v0 = tag_val(w0);
            v1 = tag_val(w1);
            ok = tag_of(w0) == c.tag && tag_of(w1) == c.tag;
        }
        if (__all_sync(0xFFFFFFFFu, ok)) return true;
        if (!spin_more(c, sp, pc)) return false;
    }
}
// one thread: one tagged element (a thread of a divergent branch).  On abort or timeout the CTA's
// abort flag is set and the value read last is returned; the caller's next wait then gives up.
__device__ float poll1(const Params& p, const Shared& sh, const uint64_t* a, int pc, uint32_t tag) {
    uint64_t w = ld_tag(a);
    if (tag_of(w) == tag) return tag_val(w);
    const uint64_t t0 = globaltimer();
    uint32_t rounds = 0;
    while (true) {
        w = ld_tag(a);
        if (tag_of(w) == tag) break;
        if (*reinterpret_cast<volatile int*>(sh.abort) || other_cta_failed(p, rounds)) {
            *reinterpret_cast<volatile int*>(sh.abort) = 1;
            break;
        }
        if (globaltimer() - t0 > p.timeout_ns) {
            raise_error(p, sh, MK_ERR_TIMEOUT, ROLE_DATA, pc, -1, tag_of(w), tag);
            break;
        }
    }
    return tag_val(w);
}

// the same for a 3-bit-tagged 32-bit word (batch > 1 activations)
__device__ float poll1h(const Params& p, const Shared& sh, const uint32_t* a, int pc, uint32_t tag) {
    const uint32_t ht = htag(tag);
    const uint64_t t0 = globaltimer();
    uint32_t rounds = 0, w;
    while (true) {
        asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(w) : "l"(a));
        if (((w ^ ht) & 7u) == 0) break;
        if (*reinterpret_cast<volatile int*>(sh.abort) || other_cta_failed(p, rounds)) {
            *reinterpret_cast<volatile int*>(sh.abort) = 1;
            break;
        }
        if (globaltimer() - t0 > p.timeout_ns) {
            raise_error(p, sh, MK_ERR_TIMEOUT, ROLE_DATA, pc, -1, w & 7u, ht);
            break;
        }
    }
    return __uint_as_float(w & ~7u);
}

__device__ __forceinline__ void load8_bf16(const uint16_t* src, float* v) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(src));
    v[0] = bf_lo(w.x); v[1] = bf_hi(w.x); v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
    v[4] = bf_lo(w.z); v[5] = bf_hi(w.z); v[6] = bf_lo(w.w); v[7] = bf_hi(w.w);
}
// where a matvec input comes from: epoch-tagged activations (t), the 3-bit tagged SwiGLU output
// (h), or the bf16 embedding row of the step's token (b)
struct XSrc {
    const uint64_t* t;
    const uint32_t* h;
    const uint16_t* b;
};
// eight elements from element e0 on; false when a tagged element does not yet carry this step's tag
__device__ __forceinline__ bool load8x(const XSrc& x, int e0, float* v, uint32_t tag) {
    if (x.t) return ld8_tagged(x.t + e0, v, tag);
    if (x.h) return ld8_htagged(x.h + e0, v, htag(tag));
    load8_bf16(x.b + e0, v);
    return true;
}
// four elements from element e0 on (e0 a multiple of 4); false when a tagged element does not yet
// carry this step's tag
__device__ __forceinline__ bool load4x(const XSrc& x, int e0, float* v, uint32_t tag) {
    if (x.t) {
        uint64_t w0, w1, w2, w3;
        ld_tag2(x.t + e0, w0, w1);
        ld_tag2(x.t + e0 + 2, w2, w3);
        v[0] = tag_val(w0); v[1] = tag_val(w1); v[2] = tag_val(w2); v[3] = tag_val(w3);
        return tag_of(w0) == tag && tag_of(w1) == tag && tag_of(w2) == tag && tag_of(w3) == tag;
    }
    if (x.h) {
        uint32_t w[4];
        asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "l"(x.h + e0));
        const uint32_t ht = htag(tag);
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = __uint_as_float(w[e] & ~7u);
        return (((w[0] ^ ht) | (w[1] ^ ht) | (w[2] ^ ht) | (w[3] ^ ht)) & 7u) == 0;
    }
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(x.b + e0));
    v[0] = bf_lo(w.x); v[1] = bf_hi(w.x); v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
    return true;
}

// the step's input token of sequence b: the first step's from the host (or, in a chained call,
// from the previous launch's greedy tokens in device memory); a later step of a multi-step launch
// takes the previous step's greedy token.  Device tokens are clamped to the vocabulary, since a
// step that failed may have left none (its recorded error is what the host then reports).
__device__ __forceinline__ int step_token(const Cw& c, int b) {
    const Params& p = c.p;
    const int32_t* src = c.step > 0 ? p.next_dev + size_t(c.step - 1) * p.B : p.tok_dev;
    if (!src) return p.tok[b];
    return min(max(__ldcg(src + b), 0), p.V - 1);
}

// where an epilogue's residual comes from: epoch-tagged words, or the bf16 embedding row (layer 0)
struct RSrc {
    const uint32_t* t;   // 3-bit-tagged fp32 words
    const uint16_t* b;
};

// The input vector of a matvec tile (sequence b) into this warp's registers: its segment g of the
// row length, RMS-normalised where the operator has a norm.  Rows up to the shared buffer's length
// take their input cooperatively: thread t polls the 8-element chunks t, t + 256, ... into shared
// memory, all of them before checking a tag, with one sum of squares per warp; after the CTA-wide arrival every warp adds the 16 sums
// in warp order (the same scale everywhere) and takes its segment.  Longer rows (the MLP down
// projection's input) are polled by each warp for its own segment, straight into registers.  In
// the same polling round thread t < nres fetches the residual word of the tile's row t into the
// shared residual buffer (O projection, MLP down).  Every warp runs this for every matvec tile
// (the instruction sequence is the same in all warps); xfree keeps a warp from overwriting a
// buffer another warp still reads: the shared input until every warp has taken its segment, a
// residual buffer (there are two, alternating) until every warp has finished the tile before.
template <int CPL>
__device__ bool load_input(Cw& c, const SlotInfo& si, const XSrc& src, const uint16_t* gain, const RSrc& rs, int nres,
                           float (&xr)[8 * CPL], float*& res, int pc) {
    const Params& p = c.p;
    const MvShape& m = si.mv;
    const int tid = c.warp * 32 + c.lane;
    const int g = c.warp & (m.G - 1);
    const int cg0 = g * m.segch;
    const int nch = min(m.segch, m.chunks - cg0);   // chunks of this warp's segment (the last may be short)
    if (c.xphase > 0 && !wait_bar(p, c.sh, c.sh.xfree, (c.xphase - 1u) & 1u, ROLE_CONSUMER, pc)) return false;
    res = c.sh.res + (c.xphase & 1u) * kResBuf;
    // the residual word of tile row tid: its load is issued before the input poll, so the two round
    // trips overlap (the residual was produced an operator earlier: it is almost always ready)
    const bool rmine = tid < nres;
    uint32_t rw = 0;
    float rb = 0.f;
    if (rmine) {
        if (rs.b) rb = bf16f(rs.b[tid]);
        else asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(rw) : "l"(rs.t + tid));
    }
    // the RMSNorm gain of this warp's segment depends on nothing: it is loaded into registers
    // before the poll, so its round trip overlaps the wait for the input (at 8 chunks per lane
    // the registers are not there: the gain is loaded after the poll)
    constexpr bool kGainEarly = CPL == 4;
    uint4 gw[CPL];
    if (kGainEarly && gain && !m.direct) {
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int ch = c.lane + 32 * i;
            gw[i] = ch < nch ? __ldg(reinterpret_cast<const uint4*>(gain + (cg0 + ch) * 8)) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    Spin sp;
    if (!m.direct) {
        // every chunk of this thread is loaded before any tag is checked: one round trip for a row
        // of up to 8 * kXChunks * 256 elements
        float ss = 0.f;
        for (int base = 0; base < m.chunks; base += kXChunks * kConsumerThreads) {   // warp-uniform
            float v[kXChunks][8];
            uint32_t good = 0;   // chunks already read with this step's tag: not read again
            while (true) {
                bool ok = true;
#pragma unroll
                for (int q = 0; q < kXChunks; ++q) {
                    const int ch = base + q * kConsumerThreads + tid;
                    if (ch < m.chunks && !((good >> q) & 1u)) {
                        const bool gq = load8x(src, ch * 8, v[q], c.tag);
                        good |= uint32_t(gq) << q;
                        ok &= gq;
                    }
                }
                if (__all_sync(0xFFFFFFFFu, ok)) break;
                if (!spin_more(c, sp, pc)) return false;
            }
#pragma unroll
            for (int q = 0; q < kXChunks; ++q) {
                const int ch = base + q * kConsumerThreads + tid;
                if (ch < m.chunks) {
                    *reinterpret_cast<float4*>(c.sh.xbuf + ch * 8) = make_float4(v[q][0], v[q][1], v[q][2], v[q][3]);
                    *reinterpret_cast<float4*>(c.sh.xbuf + ch * 8 + 4) = make_float4(v[q][4], v[q][5], v[q][6], v[q][7]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = fmaf(v[q][e], v[q][e], ss);
                }
            }
        }
        if (gain) {
            ss = warp_sum(ss);
            if (c.lane == 0) c.sh.red[48 + c.warp] = ss;
        }
    } else {
        uint32_t good = 0;   // chunks already read with this step's tag: not read again
        while (true) {
            bool ok = true;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const int ch = c.lane + 32 * i;
                if (ch < nch) {
                    if (!((good >> i) & 1u)) {
                        const bool gi = load8x(src, (cg0 + ch) * 8, &xr[8 * i], c.tag);
                        good |= uint32_t(gi) << i;
                        ok &= gi;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) xr[8 * i + e] = 0.f;
                }
            }
            if (__all_sync(0xFFFFFFFFu, ok)) break;
            if (!spin_more(c, sp, pc)) return false;
        }
    }
    if (rmine)
        res[tid] = rs.b ? rb
                        : (((rw ^ htag(c.tag)) & 7u) == 0 ? __uint_as_float(rw & ~7u) : poll1h(p, c.sh, rs.t + tid, pc, c.tag));
    __syncwarp();
    if (c.lane == 0) mbar_arrive(c.sh.xfull);
    if (!wait_bar(p, c.sh, c.sh.xfull, c.xphase & 1u, ROLE_CONSUMER, pc)) return false;
    if (!m.direct) {
        float scale = 1.0f;
        if (gain) {
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < kNumConsumerWarps; ++w) tot += c.sh.red[48 + w];
            scale = rsqrtf(tot / float(m.K) + p.rms_eps);
        }
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int ch = c.lane + 32 * i;
            float* x = &xr[8 * i];
            if (ch < nch) {
                const int cg = cg0 + ch;
                const float4 a = *reinterpret_cast<const float4*>(c.sh.xbuf + cg * 8);
                const float4 b = *reinterpret_cast<const float4*>(c.sh.xbuf + cg * 8 + 4);
                x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
                if (gain) {
                    if (!kGainEarly) gw[i] = __ldg(reinterpret_cast<const uint4*>(gain + cg * 8));
                    x[0] = (x[0] * scale) * bf_lo(gw[i].x); x[1] = (x[1] * scale) * bf_hi(gw[i].x);
                    x[2] = (x[2] * scale) * bf_lo(gw[i].y); x[3] = (x[3] * scale) * bf_hi(gw[i].y);
                    x[4] = (x[4] * scale) * bf_lo(gw[i].z); x[5] = (x[5] * scale) * bf_hi(gw[i].z);
                    x[6] = (x[6] * scale) * bf_lo(gw[i].w); x[7] = (x[7] * scale) * bf_hi(gw[i].w);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = 0.f;
            }
        }
    }
    __syncwarp();
    if (c.lane == 0) mbar_arrive(c.sh.xfree);
    ++c.xphase;
    return true;
}

// Output of one matvec row (tile row ru, run by one lane).  The LM head keeps this lane's running
// (max, lowest index) in bv / bi.
template <bool RES = true>   // RES: residuals of rows below kResBuf are in res (batch 1)
__device__ __forceinline__ void mv_epilogue(const Cw& c, const SlotInfo& si, int pc, int b, int ru, float s0,
                                            float s1, const float* res, float& bv, int& bi) {
    const Params& p = c.p;
    const int op = si.w[W_OP], l = si.w[W_LAYER];
    const size_t lb = size_t(l) * p.B + b;
    const int row = si.w[W_A0] + ru;
    switch (op) {
        case OP_QKV: st_tag(p.qkv + lb * p.nqkv + row, s0, c.tag); break;
        case OP_OPROJ: {   // (3-bit-tagged 32-bit residual words; res: the tile's residual buffer, or
                           // at batch > 1 the one word read ahead)
            const float r = (RES && ru < kResBuf) ? res[ru]
                          : l == 0            ? bf16f(p.embed[size_t(step_token(c, b)) * p.H + row])
                          : (!RES && res)     ? *res
                                              : poll1h(p, c.sh, reinterpret_cast<const uint32_t*>(p.x_out) + (lb - p.B) * p.H + row,
                                                       pc, c.tag);
            st_htag(reinterpret_cast<uint32_t*>(p.x_attn) + lb * p.H + row, r + s0, htag(c.tag));
            break;
        }
        case OP_UPGATE: st_htag(p.h + lb * p.F + row, __fdividef(s0, 1.0f + __expf(-s0)) * s1, htag(c.tag)); break;
        case OP_DOWN: {
            const float r = (RES && ru < kResBuf) ? res[ru]
                          : (!RES && res)     ? *res
                                              : poll1h(p, c.sh, reinterpret_cast<const uint32_t*>(p.x_attn) + lb * p.H + row, pc, c.tag);
            st_htag(reinterpret_cast<uint32_t*>(p.x_out) + lb * p.H + row, r + s0, htag(c.tag));
            break;
        }
        default:   // LM head: the logit, then this lane's running (max, lowest index)
            p.logits[size_t(b) * p.V + row] = s0;
            if (s0 > bv || (s0 == bv && row < bi)) {
                bv = s0;
                bi = row;
            }
            break;
    }
}

// A page group of a matvec tile: its pages' ring slots and phase parities, and the tile rows of
// each page.
struct GroupRef {
    uint32_t slot, slot1, par, par1;
    int r0, n0, r1, n1;
};

// The rows of one page group, once every consumer warp has left its segment sums, one lane per
// row.  A row's G segment sums are added in segment order (the same order whichever warp runs
// this, so the result does not depend on timing or SM count).  Page 0 holds tile rows
// [r0, r0 + n0), page 1 rows [r1, r1 + n1); for gate/up both pages hold the same n0 rows (gate sums
// in word 0 of a unit's partial, up sums in word 1).  The LM head keeps each lane's running
// (max, lowest index) in bv / bi.
__device__ void group_epilogue(const Cw& c, const SlotInfo& si, int pc, int b, const GroupRef& gr, const float* res,
                               float& bv, int& bi) {
    const Params& p = c.p;
    const int G = si.mv.G, lg = si.mv.logG;
    const bool pair = si.inter != 0;
    const int nrows = pair ? gr.n0 : gr.n0 + gr.n1;
    const float* cb0 = c.sh.comb + (size_t(gr.slot) * 2 + gr.par) * p.comb_stride * 2;
    const float* cb1 = c.sh.comb + (size_t(gr.slot1) * 2 + gr.par1) * p.comb_stride * 2;
    for (int i = c.lane; i < nrows; i += 32) {
        const bool second = !pair && i >= gr.n0;
        const int r = second ? i - gr.n0 : i;
        const float* q = (second ? cb1 : cb0) + (size_t(r) << lg) * 2;
        float s0 = q[0], s1 = q[1];
#pragma unroll 1
        for (int k = 1; k < G; ++k) {
            s0 += q[2 * k];
            s1 += q[2 * k + 1];
        }
        mv_epilogue(c, si, pc, b, (second ? gr.r1 : gr.r0) + r, s0, s1, res, bv, bi);
    }
}

// Writes a page group's rows once all consumer warps have arrived on its counter (a bounded wait:
// the group's other warps are at most a step behind), then resets the counter for the slot's
// next use of this phase.  False when the CTA aborts or the wait runs out.
__device__ bool finish_group(const Cw& c, const SlotInfo& si, int pc, int b, const GroupRef& gr, const float* res,
                             float& bv, int& bi) {
    volatile int* cnt = c.sh.combcnt + gr.slot * 2 + gr.par;
    int ok = 1;
    if (c.lane == 0 && *cnt != kNumConsumerWarps) {
        const uint64_t t0 = globaltimer();
        while (*cnt != kNumConsumerWarps) {
            if (*reinterpret_cast<volatile int*>(c.sh.abort)) { ok = 0; break; }
            if (globaltimer() - t0 > budget(c.p, ROLE_CONSUMER)) {
                raise_error(c.p, c.sh, MK_ERR_TIMEOUT, ROLE_CONSUMER, pc, -1, uint32_t(*cnt), kNumConsumerWarps);
                ok = 0;
                break;
            }
        }
    }
    __threadfence_block();
    if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) return false;
    __syncwarp();
    group_epilogue(c, si, pc, b, gr, res, bv, bi);
    __syncwarp();
    if (c.lane == 0) *cnt = 0;   // (seen by the slot's next use of this phase through the ring's mbarriers)
    return true;
}

// ------------------------------------------------------------------- batch > 1 matvec ------
// A batch > 1 matvec tile is one contraction of the tile's rows with the batch's input vectors on
// the tensor cores: mma.sync m16n8k16, bf16 operands, fp32 accumulation, the sequences as the
// 8 columns.  Each input element is split as hi = bf16(x), lo = bf16(x - hi); the weights are
// bf16 already, so W x = W hi + W lo keeps the input to about 16 mantissa bits.  The row length
// is taken in ranges of up to kMmvRange positions: the inputs of every sequence for one range are
// staged in shared memory once per tile (fp32 as polled, then turned in place into (hi, lo) word
// pairs, normalised for the RMSNorm operators), and the products of the range are added into
// accumulators that persist over the ranges.  The tile's pages hold whole rows and stay leased
// for the tile.  An MMA takes 16 rows -- row r of the first page of a pair of pages and row r of
// the second (for gate/up: the gate row and the up row) -- over 16 positions; one 16-byte load per
// row and lane covers two MMAs, the same positions for every row and for the inputs.  Warp w takes
// the 32-position steps w, w + 8, ... of each range; the 8 warps' sums meet in shared memory and
// are added in warp order.

__device__ __forceinline__ uint32_t bf16x2_rn(float e0, float e1) {   // e0 in the low half
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(e1), "f"(e0));
    return d;
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// where sequence b's input of a matvec operator comes from (and its RMSNorm gain)
__device__ __forceinline__ XSrc mmv_src(const Cw& c, int op, int l, int b, const uint16_t*& gain) {
    const Params& p = c.p;
    XSrc src{nullptr, nullptr, nullptr};
    const size_t lb = size_t(l) * p.B + b;
    gain = nullptr;
    // (the residual streams and the attention output are 3-bit-tagged 32-bit words, like the
    // SwiGLU output: half the bytes every SM polls)
    const uint32_t* xo = reinterpret_cast<const uint32_t*>(p.x_out);
    switch (op) {
        case OP_QKV:
            gain = c.sh.layers[l].attn_norm;
            if (l == 0) src.b = p.embed + size_t(step_token(c, b)) * p.H;
            else src.h = xo + (lb - p.B) * p.H;
            break;
        case OP_OPROJ: src.h = reinterpret_cast<const uint32_t*>(p.o) + lb * p.qd; break;
        case OP_UPGATE: gain = c.sh.layers[l].mlp_norm; src.h = reinterpret_cast<const uint32_t*>(p.x_attn) + lb * p.H; break;
        case OP_DOWN: src.h = p.h + lb * p.F; break;
        default: gain = p.final_norm; src.h = xo + (size_t(p.L - 1) * p.B + b) * p.H; break;
    }
    return src;
}

// The 32-position steps of one 16-row block over the staged range: positions [k0, k0 + kr) of
// the rows, [0, kr) of the staged inputs; the hi and lo products in two accumulator chains.
struct MmvBlk {
    uint32_t a0, a1;   // shared addresses of this lane's rows (g, g + 8) at position 0
    bool v0, v1;
};
__device__ __forceinline__ void mmv_steps(const Cw& c, const MmvBlk& bk, uint32_t xrow, int k0, int kr,
                                          float (&acc)[2][4]) {
    const int t4 = c.lane & 3;
    const int npr = (kr + 31) / 32;
    for (int pr = c.warp; pr < npr; pr += kNumConsumerWarps) {
        const int kl = pr * 32 + 8 * t4;   // position within the range
        const bool kv = kl < kr;           // (only a range's last 32-step can be short: zeros past it;
                                           // every lane still takes part in the MMAs)
        const uint32_t ka = uint32_t(k0 + kl) * 2u;
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        const uint4 x0 = kv ? lds128(xrow + uint32_t(kl) * 4u) : z, x1 = kv ? lds128(xrow + uint32_t(kl) * 4u + 16u) : z;
        const uint4 A0 = (kv && bk.v0) ? lds128(bk.a0 + ka) : z;
        const uint4 A1 = (kv && bk.v1) ? lds128(bk.a1 + ka) : z;
        // staged words: hi in the low half, lo in the high half
        mma16816(acc[0], A0.x, A1.x, A0.y, A1.y, __byte_perm(x0.x, x0.y, 0x5410), __byte_perm(x0.z, x0.w, 0x5410));
        mma16816(acc[1], A0.x, A1.x, A0.y, A1.y, __byte_perm(x0.x, x0.y, 0x7632), __byte_perm(x0.z, x0.w, 0x7632));
        mma16816(acc[0], A0.z, A1.z, A0.w, A1.w, __byte_perm(x1.x, x1.y, 0x5410), __byte_perm(x1.z, x1.w, 0x5410));
        mma16816(acc[1], A0.z, A1.z, A0.w, A1.w, __byte_perm(x1.x, x1.y, 0x7632), __byte_perm(x1.z, x1.w, 0x7632));
    }
}
// the slot and phase of page pg of a tile
__device__ __forceinline__ void tile_page(const Params& p, const SlotInfo& si, int pg, uint32_t& slot, uint32_t& ph) {
    const uint32_t idx = uint32_t(si.first_slot) + uint32_t(pg);
    slot = idx % uint32_t(p.n_pages);
    ph = uint32_t(si.first_phase) ^ ((idx / uint32_t(p.n_pages)) & 1u);
}

// A down-projection tile of one staging range (batch > 1, rows longer than kMmvRange): the tile
// of a lower range r stores its sum s of row `row` for sequence b as a 3-bit-tagged partial
// ([L][ranges - 1][B][H]) and returns s; the tile of the last range reads the other ranges'
// partials as they land (the loads of up to four issued before any tag is checked), adds them in
// range order and its own sum last, and returns the row's sum.
__device__ float down_partials(const Cw& c, int pc, int l, int b, int row, int r, int nrg, float s) {
    const Params& p = c.p;
    const size_t rstride = size_t(p.B) * p.H;
    uint32_t* base = p.dpart + size_t(l) * (nrg - 1) * rstride + size_t(b) * p.H + row;
    const uint32_t ht = htag(c.tag);
    if (r + 1 < nrg) {
        st_htag(base + r * rstride, s, ht);
        return s;
    }
    float t = 0.f;
    for (int r0 = 0; r0 < nrg - 1; r0 += 4) {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (r0 + i < nrg - 1)
                asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(w[i]) : "l"(base + (r0 + i) * rstride));
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (r0 + i < nrg - 1)
                t += ((w[i] ^ ht) & 7u) == 0 ? __uint_as_float(w[i] & ~7u)
                                             : poll1h(p, c.sh, base + (r0 + i) * rstride, pc, c.tag);
    }
    return t + s;
}

__device__ bool mmv_tile(Cw& c, const SlotInfo& si, int pc) {
    const Params& p = c.p;
    const MvShape& m = si.mv;
    const int op = si.w[W_OP], l = si.w[W_LAYER];
    const bool pair = si.inter != 0;
    const int K = m.K, R = si.rows, B = p.B, kp = p.mmv_kp;
    const int tid = c.warp * 32 + c.lane, g = c.lane >> 2, t4 = c.lane & 3;
    // a page is one 16-row block (gate/up: 8 pairs, gate rows then up rows) over kp positions, the
    // pages in the order (staging range, block, slice).  Rows longer than a staging range keep the
    // sums of every block of the tile over the ranges (at most 4 blocks: 64 rows, scheduled so)
    const int KR = min(K, kMmvRange), RS = int(mmv_row_stride(KR));
    const bool multi = K > KR;
    // the down projection of such rows runs one staging range per tile (range a2); the tile of the
    // last range adds the other ranges' partial sums and alone writes the rows
    const int nrg = (K + KR - 1) / KR;
    const bool dsplit = op == OP_DOWN && mmv_down_ranges(B, p.F) > 1;
    const int rr0 = dsplit ? si.w[W_A2] : 0, rr1 = dsplit ? rr0 + 1 : nrg;
    const bool dred = rr1 == nrg;   // this tile writes the rows
    uint8_t* stage = reinterpret_cast<uint8_t*>(c.sh.xbuf);
    float* part = reinterpret_cast<float*>(stage + uint32_t(p.xbuf_floats) * 4u - kMmvPartBytes);
    const uint32_t stage_s = smem_u32(stage), ring_base = smem_u32(c.sh.ring);
    const int rb = pair ? 8 : 16;   // tile rows (pairs) of a block
    const int nblk = (R + rb - 1) / rb;
    const int nsl = (K + kp - 1) / kp;
    const uint32_t pstride = uint32_t(kp) * 2u;   // bytes between a page's rows
    const int gs = min(g, B - 1);   // (columns past the batch read a valid row; unused)
    const uint16_t* gain;
    mmv_src(c, op, l, 0, gain);
    float bv = -INFINITY;   // LM head: this lane's running (max, lowest index) for sequence lane % 8
    int bi = 0x7FFFFFFF;
    if (multi && nblk > 4) {   // (not scheduled: such tiles take at most 64 rows)
        raise_error(p, c.sh, MK_ERR_CAPACITY, ROLE_CONSUMER, pc, -1, uint32_t(nblk), 4u);
        return false;
    }
    float acc[4][2][4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[q][h][e] = 0.f;
    int pg = 0;   // the tile's next page
    // rows of 8 x 256 positions (one range): a thread's items all take gain chunk tid, read ahead
    // of the input poll so that its round trip overlaps the poll
    const bool gpre = gain && K == 8 * kConsumerThreads;
    const uint4 gw_pre = gpre ? __ldg(reinterpret_cast<const uint4*>(gain + tid * 8)) : make_uint4(0u, 0u, 0u, 0u);
    // the residual of this thread's output in the first round of outputs, read ahead of the input
    // poll (produced an operator or more earlier: almost always ready), so the two round trips
    // overlap; a stale tag leaves it to the epilogue's poll
    float rres = 0.f;
    bool rok = false;
    {
        const int oq = tid >> 7, orr = (tid >> 3) & 15, ocol = tid & 7, orow = oq * rb + orr;
        if (((op == OP_DOWN && dred) || (op == OP_OPROJ && l > 0)) && !pair && oq < nblk && ocol < B && orow < R) {
            const size_t lb = size_t(l) * B + ocol;
            const uint32_t* a = op == OP_DOWN ? reinterpret_cast<const uint32_t*>(p.x_attn) + lb * p.H + si.w[W_A0] + orow
                                              : reinterpret_cast<const uint32_t*>(p.x_out) + (lb - B) * p.H + si.w[W_A0] + orow;
            uint32_t w;
            asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(w) : "l"(a));
            rok = ((w ^ htag(c.tag)) & 7u) == 0;
            rres = __uint_as_float(w & ~7u);
        }
    }
    // block q over the slices [s0, s1) of the staged range (positions from k0): MMA rows g and
    // g + 8 are page rows g and g + 8; each page is waited for, used and given back in turn
    auto block = [&](int q, int s0, int s1, int k0, uint32_t xrow, float (&a)[2][4]) -> bool {
        const bool v0 = pair ? q * 8 + g < R : q * 16 + g < R;
        const bool v1 = pair ? v0 : q * 16 + g + 8 < R;
        for (int sl = s0; sl < s1; ++sl, ++pg) {
            uint32_t slot, ph;
            tile_page(p, si, pg, slot, ph);
            if (!wait_bar(p, c.sh, c.sh.full + slot, ph, ROLE_CONSUMER, pc)) return false;
            MmvBlk bk;
            bk.v0 = v0;
            bk.v1 = v1;
            bk.a0 = ring_base + (slot << p.page_shift) + uint32_t(g) * pstride;
            bk.a1 = bk.a0 + 8u * pstride;
            mmv_steps(c, bk, xrow + uint32_t(sl * kp - k0) * 4u, 0, min(kp, K - sl * kp), a);
            __syncwarp();
            if (c.lane == 0) mbar_arrive(c.sh.empty + slot);
        }
        return true;
    };
    // the outputs of blocks blk0 and blk0 + 1 from their sums: the 8 warps' partials meet in shared
    // memory and are added in warp order
    auto outputs = [&](int blk0, float (&a0)[2][4], float (&a1)[2][4]) -> bool {
        const int nb = min(2, nblk - blk0);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float (&a)[2][4] = q == 0 ? a0 : a1;
            float* pw = part + (q * kNumConsumerWarps + c.warp) * 128;
            pw[g * 8 + 2 * t4] = a[0][0] + a[1][0];
            pw[g * 8 + 2 * t4 + 1] = a[0][1] + a[1][1];
            pw[(g + 8) * 8 + 2 * t4] = a[0][2] + a[1][2];
            pw[(g + 8) * 8 + 2 * t4 + 1] = a[0][3] + a[1][3];
        }
        if (!cbar(c, pc)) return false;
        {   // thread (block q, MMA row rr, column = sequence col)
            const int q = tid >> 7, rr = (tid >> 3) & 15, col = tid & 7;
            const int blk = blk0 + q;
            if (q < nb && col < B && (!pair || rr < 8)) {
                const int row = blk * rb + rr;   // (gate/up: pair rr, its up row at MMA row rr + 8)
                if (row < R) {
                    float s0 = 0.f, s1 = 0.f;
                    for (int w = 0; w < kNumConsumerWarps; ++w) {
                        s0 += part[(q * kNumConsumerWarps + w) * 128 + rr * 8 + col];
                        if (pair) s1 += part[(q * kNumConsumerWarps + w) * 128 + (rr + 8) * 8 + col];
                    }
                    if (gain) {   // RMSNorm: the sequence's 1 / rms
                        const float sc = c.sh.red[48 + col];
                        s0 *= sc;
                        s1 *= sc;
                    }
                    if (dsplit) s0 = down_partials(c, pc, l, col, si.w[W_A0] + row, rr0, nrg, s0);
                    if (dred) mv_epilogue<false>(c, si, pc, col, row, s0, s1, (blk0 == 0 && rok) ? &rres : nullptr, bv, bi);
                }
            }
        }
        return cbar(c, pc);   // the partial area is reused
    };
    for (int rr = rr0; rr < rr1; ++rr) {
        const int k0 = rr * KR;
        const int kr = min(KR, K - k0), csr = kr / 8, items = B * csr;
        // 1. the range's inputs, every element polled until it carries this step's tag and stored
        //    into the stage (rewritten on every round) as the (high, remainder) words the
        //    contraction reads; with a norm they hold x * gain, each item's sum of squares of x is
        //    kept, and the sequence's 1 / rms scales the row sums in the outputs (a pass rescaling
        //    the staged inputs cost about 2 us a tile).  (Every SM reads the inputs in the same
        //    order: spreading the SMs over different parts of the inputs at a time was measured
        //    slower.)
        {
            Spin spn;
            uint32_t good = 0;   // items already read with this step's tag: not read again
            while (true) {
                bool ok = true;
                // (two items per unrolled step: the kernel carries every operator body and its
                // instruction cache is short; measured at batch 8, full unrolling 1455 us a step,
                // two items 1438, one item 1471)
#pragma unroll 2
                for (int j = 0; j < kMmvItems; ++j) {
                    const int i = tid + j * kConsumerThreads;
                    if (i >= items) break;
                    if ((good >> j) & 1u) continue;
                    const int s = i / csr, ci = i % csr;
                    const uint16_t* gn;
                    const XSrc src = mmv_src(c, op, l, s, gn);
                    float v[8];
                    const bool gj = load8x(src, k0 + ci * 8, v, c.tag);
                    good |= uint32_t(gj) << j;
                    ok &= gj;
                    float y[8];
                    if (gain) {
                        const uint4 gw = gpre ? gw_pre : __ldg(reinterpret_cast<const uint4*>(gain + k0 + ci * 8));
                        y[0] = v[0] * bf_lo(gw.x); y[1] = v[1] * bf_hi(gw.x); y[2] = v[2] * bf_lo(gw.y); y[3] = v[3] * bf_hi(gw.y);
                        y[4] = v[4] * bf_lo(gw.z); y[5] = v[5] * bf_hi(gw.z); y[6] = v[6] * bf_lo(gw.w); y[7] = v[7] * bf_hi(gw.w);
                        part[i] = ((v[0] * v[0] + v[1] * v[1]) + (v[2] * v[2] + v[3] * v[3])) +
                                  ((v[4] * v[4] + v[5] * v[5]) + (v[6] * v[6] + v[7] * v[7]));
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) y[e] = v[e];
                    }
                    uint32_t o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const uint32_t hb = bf16x2_rn(y[e], 0.f) & 0xFFFFu;
                        o[e] = hb | (bf16x2_rn(y[e] - __uint_as_float(hb << 16), 0.f) << 16);
                    }
                    uint4* dst = reinterpret_cast<uint4*>(stage + s * RS + ci * 32);
                    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
                }
                if (__all_sync(0xFFFFFFFFu, ok)) break;
                if (!spin_more(c, spn, pc)) return false;
            }
        }
        if (rr == rr0 && c.warp == 0 && c.lane == 0) stamp(p, pc, 6);   // (trace: this warp's inputs polled)
        if (gain) {   // RMSNorm (one range: the row length is at most kMmvRange): 1 / rms per sequence,
                      // read by the outputs after their barrier
            if (!cbar(c, pc)) return false;   // every item's sum of squares (and staged words)
            if (c.warp < B) {   // warp s: sequence s's chunk sums, lane-strided, then a butterfly
                float q = 0.f;
                for (int ci = c.lane; ci < csr; ci += 32) q += part[c.warp * csr + ci];
                q = warp_sum(q);
                if (c.lane == 0) c.sh.red[48 + c.warp] = rsqrtf(q / float(K) + p.rms_eps);
            }
        }
        if (!cbar(c, pc)) return false;   // staged words visible; the partial area and the scales are free again
        // 3. the contraction of the range
        const uint32_t xrow = stage_s + uint32_t(gs * RS);
        const int s0 = k0 / kp, s1 = min(nsl, s0 + (KR + kp - 1) / kp);   // the range's slices (rows shorter than a page: one)
        if (multi) {   // every block into its sums over the ranges
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (q >= nblk) break;
                if (!block(q, s0, s1, k0, xrow, acc[q])) return false;
            }
            if (rr + 1 < rr1) {
                if (!cbar(c, pc)) return false;   // the next range restages the inputs
                continue;
            }
            if (!outputs(0, acc[0], acc[1])) return false;
            if (nblk > 2 && !outputs(2, acc[2], acc[3])) return false;
        } else {   // two blocks at a time
            for (int blk0 = 0; blk0 < nblk; blk0 += 2) {
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[q][h][e] = 0.f;
                if (!block(blk0, s0, s1, k0, xrow, acc[0])) return false;
                if (blk0 + 1 < nblk && !block(blk0 + 1, s0, s1, k0, xrow, acc[1])) return false;
                if (!outputs(blk0, acc[0], acc[1])) return false;
            }
        }
    }
    if (op == OP_LMHEAD) {   // per sequence: this warp's running best (lanes col, col + 8, col + 16, col + 24)
#pragma unroll
        for (int o = 8; o <= 16; o <<= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (c.lane < B) {
            const int b = c.lane;
            float2& run = c.sh.lmbest[c.warp * kMaxBatch + b];
            if (bv > run.x || (bv == run.x && bi < __float_as_int(run.y))) run = make_float2(bv, __int_as_float(bi));
            p.lm_part[(size_t(b) * gridDim.x + blockIdx.x) * kNumConsumerWarps + c.warp] =
                make_int4(__float_as_int(run.x), __float_as_int(run.y), int(c.epoch), 0);
        }
    }
    return true;
}

// Matvec tile (QKV / O / gate-up / down / LM-head rows).  Pages hold whole rows; the tile is
// walked in groups of two pages: two row pages, or for gate/up the gate page and the up page of
// the same row group.  A page holds units (row, segment) in row-major order; warp w takes units
// j = w, w + 16, ... of the group, always its own segment, two row dots at a time (the unit in the
// first page and the unit in the second), and leaves each sum in the page slot's partial area.
// The warp that arrives last on the group's counter writes the group's rows.  At batch 1 the tile
// streams: a warp waits only for the pages of its current group and gives them back when done with
// them, so a tile may be far larger than the page ring.  At batch > 1 every sequence reads every
// page: the tile's pages are held until it is done.
template <int CPL>
__device__ bool matvec_tile(Cw& c, const SlotInfo& si, int pc) {
    const Params& p = c.p;
    const int op = si.w[W_OP], l = si.w[W_LAYER], a0 = si.w[W_A0];
    const bool pair = si.inter != 0;
    const MvShape& m = si.mv;
    const int R = si.rows, rpp = m.rpp, lg = m.logG;
    const int g = c.warp & (m.G - 1);
    const int nch = min(m.segch, m.chunks - g * m.segch);
    const uint32_t rowbytes = m.rowbytes, NP = uint32_t(p.n_pages);
    const int npg = si.n_pages;
    const bool stream = p.B == 1;
    if (!stream && !wait_pages(c, si, pc)) return false;
    float xr[8 * CPL];
    const uint32_t lane_off = uint32_t(g * m.segch + c.lane) * 16u;   // this lane's first chunk within a row
    const uint32_t ring_base = smem_u32(c.sh.ring);
    // this lane's partial word within a unit: lane 0 the first sum (word 0), lane 16 the second
    // (gate/up: word 1 of the same unit; otherwise word 0 of the second page's unit)
    const int pword = (pair && c.lane == 16) ? 1 : 0;
    // (the residual streams and the attention output: 3-bit-tagged 32-bit words)
    const uint32_t* xo = reinterpret_cast<const uint32_t*>(p.x_out);
    const uint32_t* xa = reinterpret_cast<const uint32_t*>(p.x_attn);
    for (int b = 0; b < p.B; ++b) {
        XSrc src{nullptr, nullptr, nullptr};
        RSrc rs{nullptr, nullptr};
        const uint16_t* gain = nullptr;
        int nres = 0;
        const size_t lb = size_t(l) * p.B + b;
        switch (op) {
            case OP_QKV:
                gain = c.sh.layers[l].attn_norm;
                if (l == 0) src.b = p.embed + size_t(step_token(c, b)) * p.H;
                else src.h = xo + (lb - p.B) * p.H;
                break;
            case OP_OPROJ:
                src.h = reinterpret_cast<const uint32_t*>(p.o) + lb * p.qd;
                if (l == 0) rs.b = p.embed + size_t(step_token(c, b)) * p.H + a0;
                else rs.t = xo + (lb - p.B) * p.H + a0;
                nres = min(R, kResBuf);
                break;
            case OP_UPGATE: gain = c.sh.layers[l].mlp_norm; src.h = xa + lb * p.H; break;
            case OP_DOWN:
                src.h = p.h + lb * p.F;
                rs.t = xa + lb * p.H + a0;
                nres = min(R, kResBuf);
                break;
            default: gain = p.final_norm; src.h = xo + (size_t(p.L - 1) * p.B + b) * p.H; break;
        }
        float* res;
        if (!load_input<CPL>(c, si, src, gain, rs, nres, xr, res, pc)) return false;
        if (b == 0 && c.warp == 0 && c.lane == 0) stamp(p, pc, 6);
        uint32_t slot = uint32_t(si.first_slot), ph = uint32_t(si.first_phase);
        GroupRef prev{};
        float bv = -INFINITY;   // LM head: the running (max, lowest index) of the rows this lane wrote
        int bi = 0x7FFFFFFF;
        const int ngroups = (npg + 1) / 2;
        for (int k = 0; k < ngroups; ++k) {
            const bool two = 2 * k + 1 < npg;
            const uint32_t slot1 = slot + 1u == NP ? 0u : slot + 1u;
            const uint32_t ph1 = slot + 1u == NP ? ph ^ 1u : ph;
            if (stream) {
                if (!wait_bar(p, c.sh, c.sh.full + slot, ph, ROLE_CONSUMER, pc)) return false;
                if (two && !wait_bar(p, c.sh, c.sh.full + slot1, ph1, ROLE_CONSUMER, pc)) return false;
            }
            int r0, n0, r1, n1;   // first tile row and rows of each page of the group
            if (pair) {
                r0 = r1 = k * rpp;
                n0 = n1 = min(rpp, R - r0);
            } else {
                r0 = 2 * k * rpp;
                n0 = min(rpp, R - r0);
                r1 = r0 + rpp;
                n1 = two ? min(rpp, R - r1) : 0;
            }
            {
                const int u0 = n0 << lg, u1 = n1 << lg, U = max(u0, u1);
                const uint32_t base0 = ring_base + (slot << p.page_shift) + lane_off;
                const uint32_t base1 = ring_base + (slot1 << p.page_shift) + lane_off;
                float* cb0 = c.sh.comb + (size_t(slot) * 2 + (ph & 1u)) * p.comb_stride * 2;
                float* cb1 = pair ? cb0 + 1 : c.sh.comb + (size_t(slot1) * 2 + (ph1 & 1u)) * p.comb_stride * 2;
                bool released = !stream;
                // RPI row units per step: units j and j + 8 of each page (CPL 4), or unit j of each page
                constexpr int RPI = CPL == 4 ? 4 : 2;
                constexpr int JSTEP = (RPI / 2) * kNumConsumerWarps;
                for (int jb = c.warp; jb < U; jb += JSTEP) {   // warp-uniform
                    bool val[RPI];
                    uint32_t addr[RPI];
#pragma unroll
                    for (int r = 0; r < RPI; ++r) {
                        const int j = jb + (r % (RPI / 2)) * kNumConsumerWarps;
                        const bool second = r >= RPI / 2;
                        val[r] = j < (second ? u1 : u0);
                        addr[r] = (second ? base1 : base0) + uint32_t(j >> lg) * rowbytes;
                    }
                    uint4 w[RPI][CPL];
#pragma unroll
                    for (int r = 0; r < RPI; ++r)
#pragma unroll
                        for (int i = 0; i < CPL; ++i)
                            w[r][i] = (val[r] && c.lane + 32 * i < nch) ? lds128(addr[r] + i * 512) : make_uint4(0u, 0u, 0u, 0u);
                    float sr[RPI];
#pragma unroll
                    for (int r = 0; r < RPI; ++r) {
                        float acc[CPL];
#pragma unroll
                        for (int i = 0; i < CPL; ++i) acc[i] = dot8(w[r][i], &xr[8 * i], 0.f);
                        float t = acc[0];
#pragma unroll
                        for (int h = 1; h < CPL; h *= 2)   // pairwise: ((a0 + a1) + (a2 + a3)) + ...
#pragma unroll
                            for (int i = 0; i + h < CPL; i += 2 * h) acc[i] += acc[i + h];
                        t = acc[0];
                        sr[r] = t;
                    }
                    // The group's pages go back to the loader once the warp's last step has consumed
                    // every value it loaded from them (the dot products above): an arrival right
                    // after the loads were issued let the loader's refill overwrite a page before
                    // all of them had read it (measured: runs no longer bit-identical).  The
                    // reduction, the partial sums and the rows need no page.
                    if (!released && jb + JSTEP >= U) {
                        __syncwarp();
                        if (c.lane == 0) {
                            mbar_arrive(c.sh.empty + slot);
                            if (two) mbar_arrive(c.sh.empty + slot1);
                        }
                        released = true;
                    }
                    // transposed butterfly: every row's 32-lane sum, row r ending in lanes
                    // [r * 32 / RPI, (r + 1) * 32 / RPI)
                    const bool b4 = c.lane & 16;
                    float v;
                    if (RPI == 4) {
                        const bool b3 = c.lane & 8;
                        const float a0 = (b4 ? sr[2 % RPI] : sr[0]) + __shfl_xor_sync(0xFFFFFFFFu, b4 ? sr[0] : sr[2 % RPI], 16);
                        const float a1 = (b4 ? sr[3 % RPI] : sr[1]) + __shfl_xor_sync(0xFFFFFFFFu, b4 ? sr[1] : sr[3 % RPI], 16);
                        v = (b3 ? a1 : a0) + __shfl_xor_sync(0xFFFFFFFFu, b3 ? a0 : a1, 8);
#pragma unroll
                        for (int o = 4; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                    } else {
                        v = (b4 ? sr[1] : sr[0]) + __shfl_xor_sync(0xFFFFFFFFu, b4 ? sr[0] : sr[1], 16);
#pragma unroll
                        for (int o = 8; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                    }
                    // the first lane of each row's lane group leaves the row's segment sum
                    const int lr = c.lane / (32 / RPI);   // this lane's row of the step
                    if ((c.lane & (32 / RPI - 1)) == 0) {
                        bool ok = false;
#pragma unroll
                        for (int r = 0; r < RPI; ++r) ok |= (lr == r) && val[r];
                        if (ok) {
                            const int j = jb + (lr % (RPI / 2)) * kNumConsumerWarps;
                            (lr >= RPI / 2 ? cb1 : cb0)[size_t(j) * 2] = v;
                        }
                    }
                }
                if (!released) {   // (a warp without units in this group)
                    __syncwarp();
                    if (c.lane == 0) {
                        mbar_arrive(c.sh.empty + slot);
                        if (two) mbar_arrive(c.sh.empty + slot1);
                    }
                }
            }
            // The group's pages went back to the loader after the warp's dot products: the rows
            // are written from the partial area, not from the pages.  The partial area and counter
            // of a page slot alternate with its phase: a slot's next use (the other phase) may
            // start before this group's rows are written, and the use after it (this phase again)
            // cannot start before every warp -- the writing one included -- has given the slot
            // back once more, which the writing warp does only after these rows.
            // Every warp arrives on the group's counter.  The group's rows are written one group
            // later by warp k mod 8: the writing rotates over the warps, so no warp carries it on
            // every group (the warp that arrives last would, and so arrive last again).
            __syncwarp();
            if (c.lane == 0) {
                __threadfence_block();
                atomicAdd(c.sh.combcnt + slot * 2 + (ph & 1u), 1);
            }
            if (k >= 1 && ((k - 1) & (kNumConsumerWarps - 1)) == c.warp &&
                !finish_group(c, si, pc, b, prev, res, bv, bi))
                return false;
            prev = GroupRef{slot, slot1, ph & 1u, ph1 & 1u, r0, n0, r1, n1};
            if (two) {
                slot = slot1 + 1u == NP ? 0u : slot1 + 1u;
                ph = slot1 + 1u == NP ? ph1 ^ 1u : ph1;
            } else {
                slot = slot1;
                ph = ph1;
            }
        }
        if (ngroups >= 1 && ((ngroups - 1) & (kNumConsumerWarps - 1)) == c.warp &&
            !finish_group(c, si, pc, b, prev, res, bv, bi))
            return false;
        if (op == OP_LMHEAD) {   // this warp's running best over the CTA's LM-head rows so far
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
                const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (c.lane == 0) {
                float2& run = c.sh.lmbest[c.warp * kMaxBatch + b];
                if (bv > run.x || (bv == run.x && bi < __float_as_int(run.y))) run = make_float2(bv, __int_as_float(bi));
                p.lm_part[(size_t(b) * gridDim.x + blockIdx.x) * kNumConsumerWarps + c.warp] =
                    make_int4(__float_as_int(run.x), __float_as_int(run.y), int(c.epoch), 0);
            }
        }
        // batch > 1: the page slots' partials and counters serve the next sequence
        if (!stream && !cbar(c, pc)) return false;
    }
    if (c.warp == 0 && c.lane == 0) stamp(p, pc, 7);
    if (!stream) release_pages(c, si);
    return true;
}

// bf16x2 of (a, b) (a in the low half), or of their rounding remainders
__device__ __forceinline__ uint32_t bf_part2(float a, float b, bool lo) {
    const uint32_t h = bf16x2_rn(a, b);
    return lo ? bf16x2_rn(a - bf_lo(h), b - bf_hi(h)) : h;
}
// Scores of one attention chunk on the tensor cores: sc[h][t] = (q_h . k_t) * scale for t < n
// (row n_old is the new key).  An MMA (m16n8k16) takes 16 positions (rows) over 16 elements of
// head_dim against 8 columns: the bf16 high parts of four heads' rotated q, then their remainders,
// so the two column halves add up to the fp32 q.  A lane's 16-byte load of a K row covers two MMAs:
// within each 32 elements, lane quad t4 takes elements 8 t4 .. 8 t4 + 7 (the same order for the q
// columns -- the contraction does not depend on it).  Warp w takes the 16-row blocks w, w + 8, ...,
// two of them a round (every load of both blocks issued before their MMAs).
template <int NP>   // head_dim / 32
__device__ __forceinline__ void attn_scores_mma(const Cw& c, int n, int n_old, int hpg, int C, const uint8_t* kbase,
                                                bool k1p, uint32_t first_slot, float* sc) {
    const Params& p = c.p;
    constexpr int d = NP * 32;
    constexpr uint32_t rowb = uint32_t(d) * 2u;
    const int g = c.lane >> 2, t4 = c.lane & 3;
    const int nmt = (n + 15) >> 4;
    const uint8_t* knew = reinterpret_cast<const uint8_t*>(c.sh.knew);
    for (int h0 = 0; h0 < hpg; h0 += 4) {
        uint32_t bq[NP][4];   // column g: head h0 + g % 4, high part (g < 4) or remainder
        {
            const float* qh = c.sh.qrot + min(h0 + (g & 3), hpg - 1) * d + 8 * t4;
            const bool lo = g >= 4;
#pragma unroll
            for (int pp = 0; pp < NP; ++pp) {
                const float4 qa = *reinterpret_cast<const float4*>(qh + 32 * pp);
                const float4 qb = *reinterpret_cast<const float4*>(qh + 32 * pp + 4);
                bq[pp][0] = bf_part2(qa.x, qa.y, lo);
                bq[pp][1] = bf_part2(qa.z, qa.w, lo);
                bq[pp][2] = bf_part2(qb.x, qb.y, lo);
                bq[pp][3] = bf_part2(qb.z, qb.w, lo);
            }
        }
        auto row = [&](int r) -> const uint8_t* {   // (rows past n read the new key; not stored)
            if (r < n_old) return k1p ? kbase + uint32_t(r) * rowb : ring_ptr(c.sh, p, first_slot, uint32_t(r) * rowb);
            return knew;
        };
        // two 16-row blocks (mt, mt + 8) a round: every load of both first, then their MMAs
        for (int mt = c.warp; mt < nmt; mt += 2 * kNumConsumerWarps) {
            const bool two = mt + kNumConsumerWarps < nmt;
            const int ra = mt * 16 + g, rb = ra + kNumConsumerWarps * 16;
            const uint32_t p0 = smem_u32(row(ra)) + 16u * t4;   // (shared-window addresses: plain ld.shared)
            const uint32_t p1 = smem_u32(row(ra + 8)) + 16u * t4;
            const uint32_t p2 = smem_u32(row(two ? rb : ra)) + 16u * t4;
            const uint32_t p3 = smem_u32(row(two ? rb + 8 : ra + 8)) + 16u * t4;
            uint4 A[NP][4];
#pragma unroll
            for (int pp = 0; pp < NP; ++pp) {
                A[pp][0] = lds128(p0 + 64u * pp);
                A[pp][1] = lds128(p1 + 64u * pp);
                A[pp][2] = lds128(p2 + 64u * pp);
                A[pp][3] = lds128(p3 + 64u * pp);
            }
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int pp = 0; pp < NP; ++pp)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint4 X = A[pp][2 * q], Y = A[pp][2 * q + 1];
                    mma16816(acc[q], X.x, Y.x, X.y, Y.y, bq[pp][0], bq[pp][1]);
                    mma16816(acc[q], X.z, Y.z, X.w, Y.w, bq[pp][2], bq[pp][3]);
                }
            // D (row, column 2 t4 + {0, 1}): quads t4 and t4 ^ 2 hold the two parts of the same heads
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[q][e] += __shfl_xor_sync(0xFFFFFFFFu, acc[q][e], 2);
            if (t4 < 2) {
                const int h = h0 + 2 * t4;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    if (q == 1 && !two) break;
                    const int r0 = q == 0 ? ra : rb, r1 = r0 + 8;
                    if (r0 < n) {
                        if (h < hpg) sc[h * C + r0] = acc[q][0] * p.attn_scale;
                        if (h + 1 < hpg) sc[(h + 1) * C + r0] = acc[q][1] * p.attn_scale;
                    }
                    if (r1 < n) {
                        if (h < hpg) sc[h * C + r1] = acc[q][2] * p.attn_scale;
                        if (h + 1 < hpg) sc[(h + 1) * C + r1] = acc[q][3] * p.attn_scale;
                    }
                }
            }
        }
    }
}
// Softmax pieces and o partial of one consumer warp over its own positions -- the 16-row blocks
// mt = warp, warp + 8, ... whose scores it computed: m_w[h] = max_t s[h][t], w[t][h] =
// exp(s[h][t] - m_w[h]), l_w[h] = sum_t w[t][h], o_w[h][e] = sum_t w[t][h] v_t[e] (row n_old is the
// new value); lane the EPL elements EPL lane .. EPL lane + EPL - 1 of every head.  Written to
// pw[warp][h][e] and mlw[warp][h] = (m_w, l_w); nothing is shared with the other warps until then.
template <int EPL, int HP>   // head_dim / 32; heads padded to HP
__device__ __forceinline__ void attn_softmax_pv_warp(const Cw& c, int n, int n_old, int hpg, int C, const float* sc,
                                                     const uint8_t* vbase, bool v1p, uint32_t first_slot, uint32_t voff,
                                                     float* wT, float* pw, float* mlw) {
    const Params& p = c.p;
    constexpr int d = EPL * 32;
    constexpr uint32_t rowb = uint32_t(d) * 2u;
    const int nmt = (n + 15) >> 4;
    const int nw = nmt > c.warp ? ((nmt - 1 - c.warp) / kNumConsumerWarps + 1) * 16 : 0;   // this warp's slots
    auto pos = [&](int j) { return (c.warp + (j >> 4) * kNumConsumerWarps) * 16 + (j & 15); };
    __syncwarp();   // this warp's scores
    float mh[HP], lh[HP];
#pragma unroll
    for (int h = 0; h < HP; ++h) { mh[h] = -INFINITY; lh[h] = 0.f; }
    for (int j = c.lane; j < nw; j += 32) {
        const int t = pos(j);
        if (t < n)
#pragma unroll
            for (int h = 0; h < HP; ++h)
                if (h < hpg) mh[h] = fmaxf(mh[h], sc[h * C + t]);
    }
#pragma unroll
    for (int h = 0; h < HP; ++h) mh[h] = warp_max(mh[h]);
    for (int j = c.lane; j < nw; j += 32) {
        const int t = pos(j);
        if (t < n) {
            float e[HP];
#pragma unroll
            for (int h = 0; h < HP; ++h) {
                e[h] = h < hpg ? expf(sc[h * C + t] - mh[h]) : 0.f;
                lh[h] += e[h];
            }
#pragma unroll
            for (int h4 = 0; h4 < HP; h4 += 4)
                *reinterpret_cast<float4*>(wT + t * HP + h4) = make_float4(e[h4], e[h4 + 1], e[h4 + 2], e[h4 + 3]);
        }
    }
#pragma unroll
    for (int h = 0; h < HP; ++h) lh[h] = warp_sum(lh[h]);
    __syncwarp();   // the weights
    float acc[HP][EPL];
#pragma unroll
    for (int h = 0; h < HP; ++h)
#pragma unroll
        for (int i = 0; i < EPL; ++i) acc[h][i] = 0.f;
    const uint8_t* vnew = reinterpret_cast<const uint8_t*>(c.sh.vnew);
    for (int mt = c.warp; mt < nmt; mt += kNumConsumerWarps) {
        if (v1p && mt * 16 + 16 <= n_old) {   // a block of cached rows: eight rows' loads, then their products
#pragma unroll
            for (int r8 = 0; r8 < 16; r8 += 8) {
                const int t0 = mt * 16 + r8;
                float v[8][EPL], w[8][HP];
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const uint8_t* vr = vbase + uint32_t(t0 + r) * rowb;
                    if constexpr (EPL == 1) {
                        v[r][0] = bf16f(*reinterpret_cast<const uint16_t*>(vr + c.lane * 2));
                    } else if constexpr (EPL == 2) {
                        const uint32_t u = *reinterpret_cast<const uint32_t*>(vr + c.lane * 4);
                        v[r][0] = bf_lo(u); v[r][1] = bf_hi(u);
                    } else {
                        const uint2 u = *reinterpret_cast<const uint2*>(vr + c.lane * 8);
                        v[r][0] = bf_lo(u.x); v[r][1] = bf_hi(u.x); v[r][2] = bf_lo(u.y); v[r][3] = bf_hi(u.y);
                    }
#pragma unroll
                    for (int h4 = 0; h4 < HP; h4 += 4) {
                        const float4 w4 = *reinterpret_cast<const float4*>(wT + (t0 + r) * HP + h4);
                        w[r][h4] = w4.x; w[r][h4 + 1] = w4.y; w[r][h4 + 2] = w4.z; w[r][h4 + 3] = w4.w;
                    }
                }
#pragma unroll
                for (int r = 0; r < 8; ++r)
#pragma unroll
                    for (int h = 0; h < HP; ++h)
#pragma unroll
                        for (int i = 0; i < EPL; ++i) acc[h][i] = fmaf(w[r][h], v[r][i], acc[h][i]);
            }
            continue;
        }
        for (int r = 0; r < 16; ++r) {   // (the block with the new row, or a ragged one)
            const int t = mt * 16 + r;
            if (t >= n) break;
            const uint8_t* vr = t < n_old ? (v1p ? vbase + uint32_t(t) * rowb : ring_ptr(c.sh, p, first_slot, voff + uint32_t(t) * rowb))
                                          : vnew;
            float v[EPL];
            if constexpr (EPL == 1) {
                v[0] = bf16f(*reinterpret_cast<const uint16_t*>(vr + c.lane * 2));
            } else if constexpr (EPL == 2) {
                const uint32_t u = *reinterpret_cast<const uint32_t*>(vr + c.lane * 4);
                v[0] = bf_lo(u); v[1] = bf_hi(u);
            } else {
                const uint2 u = *reinterpret_cast<const uint2*>(vr + c.lane * 8);
                v[0] = bf_lo(u.x); v[1] = bf_hi(u.x); v[2] = bf_lo(u.y); v[3] = bf_hi(u.y);
            }
            float w[HP];
#pragma unroll
            for (int h4 = 0; h4 < HP; h4 += 4) {
                const float4 w4 = *reinterpret_cast<const float4*>(wT + t * HP + h4);
                w[h4] = w4.x; w[h4 + 1] = w4.y; w[h4 + 2] = w4.z; w[h4 + 3] = w4.w;
            }
#pragma unroll
            for (int h = 0; h < HP; ++h)
#pragma unroll
                for (int i = 0; i < EPL; ++i) acc[h][i] = fmaf(w[h], v[i], acc[h][i]);
        }
    }
#pragma unroll
    for (int h = 0; h < HP; ++h)
        if (h < hpg) {
#pragma unroll
            for (int i = 0; i < EPL; ++i) pw[(c.warp * HP + h) * d + c.lane * EPL + i] = acc[h][i];
            if (c.lane == 0) { mlw[(c.warp * HP + h) * 2] = mh[h]; mlw[(c.warp * HP + h) * 2 + 1] = lh[h]; }
        }
}
// Combine of one (sequence, KV group)'s chunk partials (chunks 0 .. nact - 1) in chunk order:
// M = max_c m_c, f_c = exp(m_c - M), L = sum_c f_c l_c, o = sum_c f_c o_c / L.  The partials are
// tagged, so the combining tile polls them straight from the chunk tiles' writes (no arrival
// counter, no second round trip).  lb = layer * B + sequence.
__device__ __forceinline__ bool attn_combine(Cw& c, int pc, size_t lb, int g, int nact) {
    const Params& p = c.p;
    const int d = p.d, hpg = p.hpg;
    const int tid = c.warp * 32 + c.lane;
    const int per = hpg * (d + 2);   // words of one chunk's partial
    const uint64_t* pbase = p.part + (lb * p.nkv + g) * size_t(p.n_chunk) * per;
    // chunks staged at a time in the shared-x buffer (free: every warp is past its last input);
    // with more active chunks the combine runs over groups of them, rescaling the running sums by
    // exp(M_old - M_new) (0 before the first group)
    const int kg = (kCombWords * kConsumerThreads) / per;
    float* stage = c.sh.xbuf;
    constexpr int kOut = kMaxHpg * kMaxHeadDim / kConsumerThreads;   // outputs per thread at most
    float Mr[kOut], Lr[kOut], Ar[kOut];
#pragma unroll
    for (int j = 0; j < kOut; ++j) { Mr[j] = -INFINITY; Lr[j] = 0.f; Ar[j] = 0.f; }
    for (int k0 = 0; k0 < nact; k0 += kg) {
        const int items = min(kg, nact - k0) * per;
        const uint64_t* src = pbase + size_t(k0) * per;
        Spin sp;
        while (true) {   // every word of this thread loaded before any tag is checked
            bool ok = true;
#pragma unroll
            for (int j = 0; j < kCombWords; ++j) {
                const int i = tid + j * kConsumerThreads;
                if (i < items) {
                    const uint64_t w = ld_tag(src + i);
                    stage[i] = tag_val(w);   // (rewritten by the next round if a tag was stale)
                    ok &= tag_of(w) == c.tag;
                }
            }
            if (__all_sync(0xFFFFFFFFu, ok)) break;
            if (!spin_more(c, sp, pc)) return false;
        }
        if (!cbar(c, pc)) return false;
        const int kn = items / per;
#pragma unroll
        for (int j = 0; j < kOut; ++j) {
            const int idx = tid + j * kConsumerThreads;
            if (idx >= hpg * d) break;
            const int h = idx / d, e = idx % d;
            const float* ph = stage + h * (d + 2);
            float M = Mr[j];
            for (int k = 0; k < kn; ++k) M = fmaxf(M, ph[k * per + d]);
            const float r = expf(Mr[j] - M);
            float Ls = Lr[j] * r, A = Ar[j] * r;
            for (int k = 0; k < kn; ++k) {
                const float f = expf(ph[k * per + d] - M);
                Ls = fmaf(f, ph[k * per + d + 1], Ls);
                A = fmaf(f, ph[k * per + e], A);
            }
            Mr[j] = M;
            Lr[j] = Ls;
            Ar[j] = A;
        }
        if (!cbar(c, pc)) return false;   // the stage is refilled next (next group, next input)
    }
    uint32_t* out = reinterpret_cast<uint32_t*>(p.o) + lb * p.qd + size_t(g) * hpg * d;   // 3-bit-tagged words
#pragma unroll
    for (int j = 0; j < kOut; ++j) {
        const int idx = tid + j * kConsumerThreads;
        if (idx >= hpg * d) continue;
        st_htag(out + idx, Ar[j] / Lr[j], htag(c.tag));
    }
    return true;
}

// Split-K decode attention over one chunk of KV positions for one (sequence, KV group); the
// chunk that holds pos also applies RoPE to the new k, rounds k and v to bf16 and appends them
// to the cache.  Writes the chunk partial (o[d] unnormalised, m, l) for each query head, then
// arrives on the group's arrival counter; the tile that arrives last combines the group's
// partials (fixed chunk order) into o and alone fires the completion the O projection waits on.
__device__ bool attn_tile(Cw& c, const SlotInfo& si, int pc) {
    const Params& p = c.p;
    const int l = si.w[W_LAYER], b = si.w[W_B], g = si.w[W_A0], ch = si.w[W_A1], C = si.w[W_A2];
    const int d = p.d, half = d / 2, hpg = p.hpg;
    const int tid = c.warp * 32 + c.lane;
    const int n_old = attn_old_rows(p, b, ch, C, c.step);
    const size_t lb = size_t(l) * p.B + b;
    const uint64_t* qkv = p.qkv + lb * p.nqkv;
    // [hpg][C] scores in the shared-x buffer: no warp reads a matvec input while the tile runs
    // (every warp passed its previous instruction at the first barrier, and the next
    // instruction's input is written only after the barrier that ends the chunk's work below)
    float* sc = c.sh.xbuf;
    if (n_old >= 0) {
        const int pos = p.pos[b] + c.step;
        const bool has_new = pos < ch * C + C;
        const int n = n_old + (has_new ? 1 : 0);
        const float2* rp = p.rope + size_t(pos) * half;
        // 1. rotate q of the group's heads; RoPE k, round k and v, append them.  q, k and v are
        //    read until they carry this step's tag, in one pass whose items (q pairs, then k pairs,
        //    then v elements) are spread over all warps, so no warp waits on two round trips.  No
        //    barrier first: what this phase writes (rotated q, new k and v) is read only by
        //    attention phases 2-4, and every warp left those of an earlier attention tile before
        //    that tile's arrival barrier; a warp still finishing another kind of instruction
        //    touches none of it (the scores, which reuse the shared-x buffer, wait for the barrier
        //    after this phase)
        {
            const size_t cache = size_t(si.kv_off) + size_t(pos - ch * C) * d;   // row pos (this chunk holds it)
            const uint64_t* kh = qkv + p.qd + size_t(g) * d;
            const uint64_t* vh = qkv + p.qd + p.kvd + size_t(g) * d;
            const int nq = hpg * half, nk = has_new ? half : 0, nitems = nq + nk + (has_new ? d : 0);
            for (int base = c.warp * 32; base < nitems; base += kConsumerThreads) {   // warp-uniform
                const int it = base + c.lane;
                const bool valid = it < nitems;
                const int kind = it < nq ? 0 : it < nq + nk ? 1 : 2;
                const int i = kind == 0 ? it % half : kind == 1 ? it - nq : it - nq - nk;
                const int h = kind == 0 ? it / half : 0;
                const uint64_t* a0 = kind == 0 ? qkv + size_t(g * hpg + h) * d + i : kind == 1 ? kh + i : vh + i;
                const uint64_t* a1 = kind == 2 ? a0 : a0 + half;
                float v0 = 0.f, v1 = 0.f;
                if (!wpoll2(c, valid, a0, a1, v0, v1, pc)) return false;
                if (valid) {
                    if (kind == 0) {
                        const float2 cs = rp[i];
                        c.sh.qrot[h * d + i] = v0 * cs.x - v1 * cs.y;
                        c.sh.qrot[h * d + i + half] = v0 * cs.y + v1 * cs.x;
                    } else if (kind == 1) {
                        const float2 cs = rp[i];
                        const uint16_t r0 = f2bf_rn(v0 * cs.x - v1 * cs.y), r1 = f2bf_rn(v0 * cs.y + v1 * cs.x);
                        c.sh.knew[i] = r0;
                        c.sh.knew[i + half] = r1;
                        p.kc[cache + i] = r0;
                        p.kc[cache + i + half] = r1;
                    } else {
                        const uint16_t r = f2bf_rn(v0);
                        c.sh.vnew[i] = r;
                        p.vc[cache + i] = r;
                    }
                }
            }
        }
        if (!wait_pages(c, si, pc)) return false;
        if (!cbar(c, pc)) return false;
        const uint32_t first_slot = uint32_t(si.first_slot);
        const uint32_t rowb = uint32_t(d) * 2u;
        const uint32_t voff = uint32_t(n_old) * rowb;
        const uint32_t kbytes = voff;
        // the K block and the V block each sit inside one page (the common case): direct pointers
        const bool k1p = n_old == 0 || (0u >> p.page_shift) == ((kbytes - 1u) >> p.page_shift);
        const bool v1p = n_old == 0 || (voff >> p.page_shift) == ((voff + kbytes - 1u) >> p.page_shift);
        const uint8_t* kbase = ring_ptr(c.sh, p, first_slot, 0u);
        const uint8_t* vbase = ring_ptr(c.sh, p, first_slot, voff);
        // 2. scores on the tensor cores; 3. each warp's softmax pieces and o partial over its own
        //    positions; 4. the 8 warps' partials merged in warp order (rescaled to the largest m)
        const int hp = hpg <= 4 ? 4 : kMaxHpg;
        float* wT = sc + ((hpg * C + 3) & ~3);       // [C][hp] (16-byte aligned rows)
        float* pw = wT + C * hp;                     // [8][hp][d]
        float* mlw = pw + kNumConsumerWarps * hp * d;   // [8][hp][2]
        if (d == 64) attn_scores_mma<2>(c, n, n_old, hpg, C, kbase, k1p, first_slot, sc);
        else if (d == 128) attn_scores_mma<4>(c, n, n_old, hpg, C, kbase, k1p, first_slot, sc);
        else attn_scores_mma<1>(c, n, n_old, hpg, C, kbase, k1p, first_slot, sc);
        if (hp == 4) {
            if (d == 64) attn_softmax_pv_warp<2, 4>(c, n, n_old, hpg, C, sc, vbase, v1p, first_slot, voff, wT, pw, mlw);
            else if (d == 128) attn_softmax_pv_warp<4, 4>(c, n, n_old, hpg, C, sc, vbase, v1p, first_slot, voff, wT, pw, mlw);
            else attn_softmax_pv_warp<1, 4>(c, n, n_old, hpg, C, sc, vbase, v1p, first_slot, voff, wT, pw, mlw);
        } else {
            if (d == 64) attn_softmax_pv_warp<2, kMaxHpg>(c, n, n_old, hpg, C, sc, vbase, v1p, first_slot, voff, wT, pw, mlw);
            else if (d == 128) attn_softmax_pv_warp<4, kMaxHpg>(c, n, n_old, hpg, C, sc, vbase, v1p, first_slot, voff, wT, pw, mlw);
            else attn_softmax_pv_warp<1, kMaxHpg>(c, n, n_old, hpg, C, sc, vbase, v1p, first_slot, voff, wT, pw, mlw);
        }
        release_pages(c, si);
        if (!cbar(c, pc)) return false;
        uint64_t* dst = p.part + ((lb * p.nkv + g) * p.n_chunk + ch) * size_t(hpg) * (d + 2);
        for (int idx = tid; idx < hpg * d; idx += kConsumerThreads) {
            const int h = idx / d, e = idx % d;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kNumConsumerWarps; ++w) M = fmaxf(M, mlw[(w * hp + h) * 2]);
            float acc = 0.f, L = 0.f;
#pragma unroll
            for (int w = 0; w < kNumConsumerWarps; ++w) {   // (a warp without positions: m = -inf, f = 0)
                const float f = expf(mlw[(w * hp + h) * 2] - M);
                acc = fmaf(f, pw[(w * hp + h) * d + e], acc);
                L = fmaf(f, mlw[(w * hp + h) * 2 + 1], L);
            }
            uint64_t* dh = dst + size_t(h) * (d + 2);
            st_tag(dh + e, acc, c.tag);
            if (e == 0) {
                st_tag(dh + d, M, c.tag);
                st_tag(dh + d + 1, L, c.tag);
            }
        }
    }
    // 5. the tile of the chunk that holds pos combines the group's partials (at batch > 1 the
    //    group's COMB tile does); the barrier first also frees the scores buffer and the new k/v
    //    for what follows.
    if (!cbar(c, pc)) return false;
    if (kBatchedKernel && si.w[W_COND] == 0) return true;
    const int nact = min(p.n_chunk, (p.pos[b] + c.step) / C + 1);
    if (ch != nact - 1) return true;
    if (tid == 0) c.sh.pubinfo[(pc % kDone) * 8 + 7] = 1;   // this tile alone fires the completion
    return attn_combine(c, pc, lb, g, nact);
}

// Combine tile (batch > 1) of (sequence, KV group): combines the chunk partials of the group's
// active chunks once they land.  The barrier first: the previous instruction's warps may still
// read the shared-x buffer the combine stages into.
__device__ bool comb_tile(Cw& c, const SlotInfo& si, int pc) {
    const int l = si.w[W_LAYER], b = si.w[W_B], g = si.w[W_A0], C = si.w[W_A2];
    const int nact = min(c.p.n_chunk, (c.p.pos[b] + c.step) / C + 1);
    if (!cbar(c, pc)) return false;
    return attn_combine(c, pc, size_t(l) * c.p.B + b, g, nact);
}

// Greedy token: argmax over the LM-head tile partials (largest value, lowest index on ties).
__device__ bool argmax_tile(Cw& c, const SlotInfo& si, int pc) {
    const Params& p = c.p;
    const int b = si.w[W_B];
    const int tid = c.warp * 32 + c.lane;
    const int n = int(gridDim.x) * kNumConsumerWarps;   // one running partial per (CTA, warp)
    const int4* parts = p.lm_part + size_t(b) * n;
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int i = tid; i < n; i += kConsumerThreads) {
        const int4 v = __ldcg(parts + i);
        if (uint32_t(v.z) != c.epoch) continue;   // written in an earlier step: this warp had no LM rows
        const float val = __int_as_float(v.x);
        if (val > bv || (val == bv && v.y < bi)) { bv = val; bi = v.y; }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if (!cbar(c, pc)) return false;   // the previous user of the scratch is done
    if (c.lane == 0) { c.sh.red[2 * c.warp] = bv; c.sh.red[2 * c.warp + 1] = __int_as_float(bi); }
    if (!cbar(c, pc)) return false;
    if (tid == 0) {
        for (int w = 0; w < kNumConsumerWarps; ++w) {
            const float ov = c.sh.red[2 * w];
            const int oi = __float_as_int(c.sh.red[2 * w + 1]);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        p.tokens_out[b] = bi;
        if (p.next_dev) p.next_dev[size_t(c.step) * p.B + b] = bi;
        if (b == 0 && p.ctl) {
            // a multi-step launch: the host's stop request, read once here, decides for every CTA
            // whether a next step runs (each reads this step's word at the next step boundary; the
            // words alternate, so a CTA slow to read it never sees the following step's decision);
            // the steps done so far go back to the host
            p.err[8 + (c.step & 1)] = ld_sys(p.ctl);
            st_sys(p.ctl + 1, c.step + 1);
        }
    }
    return true;
}

// The counter wait this warp saw satisfied last: counters only grow within a launch, so the same
// wait again (consecutive tiles of one operator) needs neither a poll nor another acquire fence.
// One entry only: the cache stays in registers live across the matvec loop, where every register
// counts.
struct CounterCache {
    int32_t id, need;
};

__device__ bool wait_counters(const Params& p, const Shared& sh, const int32_t* w, int pc, CounterCache& cc,
                              uint32_t epoch) {
    const int nw = w[W_NWAIT];
    bool polled = false;
    for (int i = 0; i < nw; ++i) {
        const int cid = w[W_WAIT + 2 * i], need = w[W_WAIT + 2 * i + 1];
        if (cc.id == cid && cc.need == need) continue;
        polled = true;
        const uint32_t target = epoch * __ldg(p.totals + cid) + uint32_t(need);
        uint32_t v = ld_relaxed_gpu(p.counters + cid);
        if (int32_t(v - target) < 0) {
            const uint64_t t0 = globaltimer();
            uint32_t rounds = 0;
            while (true) {
                v = ld_relaxed_gpu(p.counters + cid);
                if (int32_t(v - target) >= 0) break;
                if (*reinterpret_cast<volatile int*>(sh.abort) || other_cta_failed(p, rounds)) {
                    *reinterpret_cast<volatile int*>(sh.abort) = 1;
                    return false;
                }
                if (globaltimer() - t0 > p.timeout_ns) {
                    raise_error(p, sh, MK_ERR_TIMEOUT, ROLE_COUNTER, pc, cid, v, target);
                    return false;
                }
            }
        }
        cc.id = cid;
        cc.need = need;
    }
    if (polled) fence_acquire_gpu();   // acquire: producers' data is visible before this warp reads it
    return true;
}

// The boundary into step c.step (> 0) of a multi-step launch: every CTA has retired the previous
// step (each added 1 to the step word after a release fence), so its greedy tokens -- this step's
// inputs -- and everything else it wrote are visible after the acquire.  The previous step's stop
// word, written by its first argmax, decides for every CTA alike.  False: stop, or the CTA aborts.
__device__ bool step_boundary(Cw& c, int pc) {
    const Params& p = c.p;
    int ok = 1;
    if (c.lane == 0) {
        const uint32_t target = c.epoch * gridDim.x;
        const uint64_t t0 = globaltimer();
        uint32_t rounds = 0;
        while (int32_t(ld_relaxed_gpu(p.step_bar) - target) < 0) {
            if (*reinterpret_cast<volatile int*>(c.sh.abort) || other_cta_failed(p, rounds)) {
                *reinterpret_cast<volatile int*>(c.sh.abort) = 1;
                ok = 0;
                break;
            }
            if (globaltimer() - t0 > p.timeout_ns) {
                raise_error(p, c.sh, MK_ERR_TIMEOUT, ROLE_COUNTER, pc, -1, ld_relaxed_gpu(p.step_bar), target);
                ok = 0;
                break;
            }
        }
        if (ok) {
            fence_acquire_gpu();
            if (*reinterpret_cast<volatile const int32_t*>(p.err + 8 + ((c.step - 1) & 1)) != 0) {
                *reinterpret_cast<volatile int*>(c.sh.stop) = 1;
                ok = 0;
            } else {
                // this warp's LM-head running bests start over
                for (int b = 0; b < p.B; ++b)
                    c.sh.lmbest[c.warp * kMaxBatch + b] = make_float2(-INFINITY, __int_as_float(0x7FFFFFFF));
            }
        }
    }
    return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// CPL: 16-byte chunks a lane holds of its row segment (batch 1); BAT: the batch > 1 kernel, whose
// matvec tiles run on the tensor cores (its own instance: no register allocation is shared with
// the batch-1 matvec path)
template <int CPL, bool BAT>
__device__ void consumer_warp(const Params& p, const Shared& sh) {
    Cw c{p, sh, int(threadIdx.x) >> 5, int(threadIdx.x) & 31, 0u, 0u, 0, p.epoch, p.tag};
    // slots and completion records are indexed by g, the instructions taken over all steps
    uint32_t g = 0;
    for (int s = 0; s < p.n_steps; ++s) {
        c.step = s;
        c.epoch = p.epoch + uint32_t(s);
        c.tag = c.epoch + 1u;
        if (s > 0 && !step_boundary(c, int(g))) return;
        CounterCache cc{-1, -1};
        for (;; ++g) {
            const int slot = int(g % kSlots);
            const int pc = int(g);
            if (!wait_bar(p, sh, sh.ins_full + slot, (g / kSlots) & 1, ROLE_CONSUMER, pc)) return;
            const SlotInfo& si = sh.slots[slot];
            const int op = si.w[W_OP];
            if (op != OP_END) {
                // counters (with acquire semantics) in the counters mode and for the one consumer
                // that reads its inputs without tags (the argmax over the LM-head partials); every
                // other consumer polls the tagged words it reads until they carry this step's tag,
                // with no counter in between: a counter poll before the data read would add a round trip
                int ok = 1;
                if (c.lane == 0 && (p.sync_counters || ((p.acquire_ops >> op) & 1)))
                    ok = wait_counters(p, sh, si.w, pc, cc, c.epoch);
                if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) return;
                if (threadIdx.x == 0) stamp(p, pc, 2);
                bool good;
                switch (op) {
                    case OP_ATTN: good = attn_tile(c, si, pc); break;
                    case OP_ARGMAX: good = argmax_tile(c, si, pc); break;
                    default:
                        if constexpr (BAT) good = op == OP_COMB ? comb_tile(c, si, pc) : mmv_tile(c, si, pc);
                        else good = matvec_tile<CPL>(c, si, pc);
                        break;
                }
                if (!good) return;
                if (threadIdx.x == 0) stamp(p, pc, 3);
            }
            __syncwarp();
            if (c.lane == 0) {
                mbar_arrive(sh.ins_empty + slot);
                mbar_arrive(sh.done + (g % kDone));
            }
            if (op == OP_END) { ++g; break; }
        }
    }
}

template <int CPL, bool BAT>
__global__ void __launch_bounds__(kThreads, 1) megakernel(const Params p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const Shared sh = carve(smem, p);
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.n_pages; ++i) {
            mbar_init(sh.full + i, 1);
            mbar_init(sh.empty + i, kNumConsumerWarps);
        }
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(sh.ins_full + i, 1);
            mbar_init(sh.ins_empty + i, kNumConsumerWarps);
        }
        for (int i = 0; i < kDone; ++i) mbar_init(sh.done + i, kNumConsumerWarps);
        *sh.published = 0;
        mbar_init(sh.qfull + 0, 1);
        mbar_init(sh.qfull + 1, 1);
        mbar_init(sh.cbar, kNumConsumerWarps);
        mbar_init(sh.xfull, kNumConsumerWarps);
        mbar_init(sh.xfree, kNumConsumerWarps);
        *sh.abort = 0;
        *sh.stop = 0;
        *sh.issued = 0ull;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = threadIdx.x; i < 2 * p.n_pages; i += blockDim.x) sh.combcnt[i] = 0;
    for (int i = threadIdx.x; i < kNumConsumerWarps * kMaxBatch; i += blockDim.x)
        sh.lmbest[i] = make_float2(-INFINITY, __int_as_float(0x7FFFFFFF));
    for (int i = threadIdx.x; i < p.L; i += blockDim.x) sh.layers[i] = p.layers[i];
    if (threadIdx.x == 0) stamp(p, 0, 5);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < kNumConsumerWarps) consumer_warp<CPL, BAT>(p, sh);
    else if (warp == kLoaderWarp) { if (lane == 0) loader(p, sh); }
    else if (lane == 0) publisher(p, sh);
    cta_sync_divergent();
}

#ifdef MK_BATCHED_TU
// This translation unit holds the batch > 1 kernel alone (the same device code compiled apart, so
// the batch-1 kernels keep their own inlining and register allocation).
const void* megakernel_fn_batched() { return reinterpret_cast<const void*>(&megakernel<4, true>); }
#else
// RoPE table: rope[p][i] = (cos, sin)(p * theta^(-2i/d)), angles in double
__global__ void rope_table_kernel(float2* out, int max_seq, int d, double theta) {
    const int half = d / 2;
    const int n = max_seq * half;
    for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += gridDim.x * blockDim.x) {
        const int pos = idx / half, i = idx % half;
        const double a = double(pos) * pow(theta, -2.0 * double(i) / double(d));
        out[idx] = make_float2(float(cos(a)), float(sin(a)));
    }
}

// the batch-1 kernel instance for a binding, by CPL (4 or 8)
const void* megakernel_fn(int cpl) {
    return cpl == 4 ? reinterpret_cast<const void*>(&megakernel<4, false>)
                    : reinterpret_cast<const void*>(&megakernel<kMaxCpl, false>);
}

cudaError_t launch_rope_table(float2* out, int max_seq, int d, double theta, cudaStream_t st) {
    const int n = max_seq * (d / 2);
    const int blocks = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
    rope_table_kernel<<<blocks, 256, 0, st>>>(out, max_seq, d, theta);
    return cudaGetLastError();
}
#endif

}  // namespace mk
