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
//  * 8 consumer warps: wait the instruction's counters (one thread spins with relaxed loads,
//     then an acquire fence), run the body on the leased pages, release the pages (mbarrier
//     arrive), write outputs, and hand the instruction to the publisher.
//  * publisher warp (one thread): fence.acq_rel.gpu, then adds the completions to the global
//     counters -- data first, then the fence, then the counter (the page's data-visibility
//     contract), without stalling the consumers on the fence.
// Every wait (counter spin, page / slot barrier) has a time budget; when it runs out the CTA
// records the error, all roles leave their loops, the loader drains its copies in flight and
// the kernel returns (no trap, no endless spin).
#include <cuda_runtime.h>
#include <stdint.h>

#include "mk_internal.h"

namespace mk {

enum Role : int { ROLE_LOADER = 1, ROLE_CONSUMER = 2, ROLE_PUBLISHER = 3, ROLE_COUNTER = 4 };

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
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void red_add_relaxed_gpu(uint32_t* p, uint32_t v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// named barrier 1 over the 256 consumer threads (non-.aligned form: lanes may arrive apart)
__device__ __forceinline__ void cons_sync() { asm volatile("barrier.sync 1, 256;" ::: "memory"); }
// whole-CTA barrier reached by warps whose lanes diverged (loader / publisher lane 0 arrives late)
__device__ __forceinline__ void cta_sync_divergent() { asm volatile("barrier.sync 0;" ::: "memory"); }
// same barrier, returning the OR of every consumer thread's predicate (uniform result)
__device__ __forceinline__ bool cons_sync_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbarrier.red.or.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(pred))
        : "memory");
    return r != 0;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
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

// ------------------------------------------------------------------------- shared memory ----
struct Shared {
    uint8_t* ring;
    SlotInfo* slots;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* ins_full;
    uint64_t* ins_empty;
    uint64_t* done;
    float* red;      // [2][8 warps][8 rows]
    float* normred;  // [8]
    int* abort;      // [1]
    float* qrot;     // [8][128]
    float* ascr;     // [attn_scratch_floats]
    uint16_t* knew;  // [128]
    uint16_t* vnew;  // [128]
    float* ml;       // [8][2]
    float* cml;      // [8]
};

__device__ __forceinline__ Shared carve(uint8_t* base, const Params& p) {
    Shared s;
    s.ring = base;
    uint8_t* m = base + p.smem_misc_off;
    s.slots = reinterpret_cast<SlotInfo*>(m);
    m += sizeof(SlotInfo) * kSlots;
    s.full = reinterpret_cast<uint64_t*>(m);
    s.empty = s.full + p.n_pages;
    s.ins_full = s.empty + p.n_pages;
    s.ins_empty = s.ins_full + kSlots;
    s.done = s.ins_empty + kSlots;
    m = reinterpret_cast<uint8_t*>(s.done + kSlots);
    s.red = reinterpret_cast<float*>(m);
    s.normred = s.red + 2 * kNumConsumerWarps * kMaxRows;
    s.abort = reinterpret_cast<int*>(s.normred + 8);
    s.qrot = reinterpret_cast<float*>(s.abort + 56);
    s.ascr = s.qrot + kMaxHpg * kMaxHeadDim;
    s.ml = s.ascr + p.attn_scratch_floats;
    s.cml = s.ml + 2 * kMaxHpg;
    s.knew = reinterpret_cast<uint16_t*>(s.cml + 2 * kMaxHpg);
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

// bounded mbarrier wait: false when the CTA aborts or the budget runs out (error recorded)
__device__ bool wait_bar(const Params& p, const Shared& sh, uint64_t* bar, uint32_t parity, int role, int pc) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int*>(sh.abort)) return false;
        if (globaltimer() - t0 > p.timeout_ns) {
            raise_error(p, sh, MK_ERR_TIMEOUT, role, pc, -1, 0, 0);
            return false;
        }
    }
}

// ------------------------------------------------------------------------- streams ----------
struct Seg {
    const uint8_t* src;
    uint32_t off, bytes;   // offset of the segment inside the tile's stream
};
struct Stream {
    Seg seg[2];
    int nseg;
    uint32_t total;
    int pages;
};

__device__ __forceinline__ int attn_old_rows(const Params& p, int b, int c, int chunk) {
    const int pos = p.pos[b];
    const int c0 = c * chunk;
    if (c0 > pos) return -1;                 // chunk past pos: inactive
    return min(c0 + chunk, pos) - c0;        // cached positions strictly before pos
}

// validates an instruction and describes the bytes its body streams; returns an mk_status
__device__ int describe(const Params& p, const int32_t* w, Stream& st) {
    st.nseg = 0;
    st.total = 0;
    st.pages = 0;
    const int op = w[W_OP];
    if (op == OP_END) return MK_OK;
    if (op <= 0 || op >= OP_COUNT) return MK_ERR_OPCODE;
    const int l = w[W_LAYER], b = w[W_B], a0 = w[W_A0], a1 = w[W_A1], a2 = w[W_A2];
    if (w[W_NWAIT] < 0 || w[W_NWAIT] > kMaxWait || w[W_NPUB] < 0 || w[W_NPUB] > kMaxPub) return MK_ERR_BOUNDS;
    for (int i = 0; i < w[W_NWAIT]; ++i)
        if (unsigned(w[W_WAIT + 2 * i]) >= unsigned(p.n_counters)) return MK_ERR_BOUNDS;
    for (int i = 0; i < w[W_NPUB]; ++i)
        if (unsigned(w[W_PUB + 2 * i]) >= unsigned(p.n_counters)) return MK_ERR_BOUNDS;
    const bool head = (op == OP_LMHEAD || op == OP_ARGMAX);
    if (head ? (l != p.L) : (unsigned(l) >= unsigned(p.L))) return MK_ERR_BOUNDS;
    if (unsigned(b) >= unsigned(p.B)) return MK_ERR_BOUNDS;
    auto rows = [&](int nrows_total, int maxn) { return a0 >= 0 && a1 >= 1 && a1 <= maxn && a0 + a1 <= nrows_total; };
    const LayerPtrs* lp = head ? nullptr : &p.layers[l];
    switch (op) {
        case OP_QKV:
            if (!rows(p.nqkv, kMaxRows)) return MK_ERR_BOUNDS;
            st.seg[0] = {reinterpret_cast<const uint8_t*>(lp->wqkv) + size_t(a0) * p.H * 2, 0, uint32_t(a1 * p.H * 2)};
            st.nseg = 1;
            break;
        case OP_OPROJ:
            if (!rows(p.H, kMaxRows)) return MK_ERR_BOUNDS;
            st.seg[0] = {reinterpret_cast<const uint8_t*>(lp->wo) + size_t(a0) * p.qd * 2, 0, uint32_t(a1 * p.qd * 2)};
            st.nseg = 1;
            break;
        case OP_UPGATE: {
            if (!rows(p.F, kMaxRows / 2)) return MK_ERR_BOUNDS;
            const uint32_t nb = uint32_t(a1 * p.H * 2);
            st.seg[0] = {reinterpret_cast<const uint8_t*>(lp->wgate_up) + size_t(a0) * p.H * 2, 0, nb};
            st.seg[1] = {reinterpret_cast<const uint8_t*>(lp->wgate_up) + size_t(p.F + a0) * p.H * 2, nb, nb};
            st.nseg = 2;
            break;
        }
        case OP_DOWN:
            if (!rows(p.H, kMaxRows)) return MK_ERR_BOUNDS;
            st.seg[0] = {reinterpret_cast<const uint8_t*>(lp->wdown) + size_t(a0) * p.F * 2, 0, uint32_t(a1 * p.F * 2)};
            st.nseg = 1;
            break;
        case OP_LMHEAD:
            if (!rows(p.V, kMaxRows) || unsigned(a2) >= unsigned(p.n_lm)) return MK_ERR_BOUNDS;
            st.seg[0] = {reinterpret_cast<const uint8_t*>(p.lm_head) + size_t(a0) * p.H * 2, 0, uint32_t(a1 * p.H * 2)};
            st.nseg = 1;
            break;
        case OP_ATTN: {
            if (unsigned(a0) >= unsigned(p.nkv) || unsigned(a1) >= unsigned(p.n_chunk) || a2 != p.attn_chunk)
                return MK_ERR_BOUNDS;
            const int n_old = attn_old_rows(p, b, a1, a2);
            if (n_old > 0) {
                const size_t base = size_t(b) * p.kv_bstride + size_t(l) * p.kv_lstride + size_t(a0) * p.kv_hstride +
                                    size_t(a1) * a2 * p.d;
                const uint32_t nb = uint32_t(n_old * p.d * 2);
                st.seg[0] = {reinterpret_cast<const uint8_t*>(p.kc + base), 0, nb};
                st.seg[1] = {reinterpret_cast<const uint8_t*>(p.vc + base), nb, nb};
                st.nseg = 2;
            }
            break;
        }
        case OP_COMB:
            if (unsigned(a0) >= unsigned(p.nkv) || a1 != p.n_chunk || a2 != p.attn_chunk) return MK_ERR_BOUNDS;
            break;
        case OP_ARGMAX:
            if (a1 != p.n_lm) return MK_ERR_BOUNDS;
            break;
        default:
            return MK_ERR_OPCODE;
    }
    for (int i = 0; i < st.nseg; ++i) st.total += st.seg[i].bytes;
    st.pages = int((st.total + uint32_t(p.page_bytes) - 1) / uint32_t(p.page_bytes));
    if (st.pages > w[W_NPAGES] || st.pages > p.n_pages) return MK_ERR_CAPACITY;
    return MK_OK;
}

// ------------------------------------------------------------------------- loader -----------
__device__ void loader(const Params& p, const Shared& sh) {
    const int32_t* q = p.queues + size_t(blockIdx.x) * p.Q * kWords;
    const uint64_t pol = evict_first_policy();
    const uint32_t PB = uint32_t(p.page_bytes);
    const uint32_t NP = uint32_t(p.n_pages);
    uint32_t page_seq = 0;
    for (int pc = 0; pc < p.Q; ++pc) {
        const int slot = pc % kSlots;
        if (pc >= kSlots && !wait_bar(p, sh, sh.ins_empty + slot, ((pc / kSlots) - 1) & 1, ROLE_LOADER, pc)) break;
        SlotInfo& si = sh.slots[slot];
        const int4* src = reinterpret_cast<const int4*>(q + size_t(pc) * kWords);
#pragma unroll
        for (int i = 0; i < kWords / 4; ++i) reinterpret_cast<int4*>(si.w)[i] = __ldg(src + i);
        Stream st;
        const int e = describe(p, si.w, st);
        if (e != MK_OK) {
            raise_error(p, sh, e, ROLE_LOADER, pc, -1, uint32_t(si.w[W_OP]), 0);
            break;
        }
        si.first_page = int32_t(page_seq);
        si.n_pages = st.pages;
        mbar_arrive(sh.ins_full + slot);   // release: the slot's words are visible to the consumers
        if (si.w[W_OP] == OP_END) break;
        bool stop = false;
        for (int pg = 0; pg < st.pages; ++pg) {
            const uint32_t k = page_seq + uint32_t(pg);
            const uint32_t ps = k % NP;
            if (k >= NP && !wait_bar(p, sh, sh.empty + ps, ((k / NP) - 1) & 1, ROLE_LOADER, pc)) {
                stop = true;
                page_seq = k;   // pages before k were issued
                break;
            }
            const uint32_t lo = uint32_t(pg) * PB;
            const uint32_t hi = min(lo + PB, st.total);
            mbar_arrive_expect_tx(sh.full + ps, hi - lo);
            uint8_t* dst = sh.ring + size_t(ps) * PB;
            for (int s = 0; s < st.nseg; ++s) {
                const uint32_t a = max(lo, st.seg[s].off);
                const uint32_t z = min(hi, st.seg[s].off + st.seg[s].bytes);
                if (a < z) bulk_g2s(dst + (a - lo), st.seg[s].src + (a - st.seg[s].off), z - a, sh.full + ps, pol);
            }
        }
        if (stop) break;
        page_seq += uint32_t(st.pages);
    }
    if (*reinterpret_cast<volatile int*>(sh.abort)) {
        // drain: wait for the last copy issued into every page so no bulk copy outlives the CTA
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
    for (int pc = 0;; ++pc) {
        const int slot = pc % kSlots;
        if (!wait_bar(p, sh, sh.done + slot, (pc / kSlots) & 1, ROLE_PUBLISHER, pc)) break;
        const SlotInfo& si = sh.slots[slot];
        if (si.w[W_OP] == OP_END) break;
        const int np = si.w[W_NPUB];
        fence_acq_rel_gpu();   // everything the consumers wrote for this instruction, then the counters
        for (int i = 0; i < np; ++i) red_add_relaxed_gpu(p.counters + si.w[W_PUB + 2 * i], uint32_t(si.w[W_PUB + 2 * i + 1]));
        mbar_arrive(sh.ins_empty + slot);
    }
}

// ------------------------------------------------------------------------- consumer bodies --
struct Cons {
    const Params& p;
    const Shared& sh;
    int tid, warp, lane;
    int rbuf;
};

__device__ __forceinline__ const uint8_t* ring_ptr(const Shared& sh, const Params& p, uint32_t first_slot, uint32_t off) {
    uint32_t s = first_slot + (off >> p.page_shift);
    if (s >= uint32_t(p.n_pages)) s -= uint32_t(p.n_pages);
    return sh.ring + (size_t(s) << p.page_shift) + (off & (uint32_t(p.page_bytes) - 1u));
}

// waits every page of the instruction; a failed wait only marks the thread (uniform exit later)
__device__ bool wait_pages(const Cons& c, const SlotInfo& si, int pc) {
    bool ok = true;
    for (int i = 0; i < si.n_pages && ok; ++i) {
        const uint32_t k = uint32_t(si.first_page) + uint32_t(i);
        ok = wait_bar(c.p, c.sh, c.sh.full + (k % uint32_t(c.p.n_pages)), (k / uint32_t(c.p.n_pages)) & 1,
                      ROLE_CONSUMER, pc);
    }
    return ok;
}
__device__ void release_pages(const Cons& c, const SlotInfo& si) {
    __syncwarp();
    if (c.lane == 0)
        for (int i = 0; i < si.n_pages; ++i)
            mbar_arrive(c.sh.empty + ((uint32_t(si.first_page) + uint32_t(i)) % uint32_t(c.p.n_pages)));
}

// block sum over the 256 consumer threads, same fixed order in every thread
__device__ float cons_block_sum(const Cons& c, float v) {
    v = warp_sum(v);
    if (c.lane == 0) c.sh.normred[c.warp] = v;
    cons_sync();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kNumConsumerWarps; ++w) s += c.sh.normred[w];
    return s;
}

// loads this thread's x chunks (tid + 256 j) of a length-K input, optionally RMS-normalised
template <int NCH>
__device__ void load_x(const Cons& c, float (&xr)[64], int K, const float* srcf, const uint16_t* srcb,
                       const uint16_t* gain) {
    const int rowchunks = K / 8;
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
        const int ch = c.tid + 256 * j;
        if (ch < rowchunks) {
            if (srcf) {
                const float4 a = __ldcg(reinterpret_cast<const float4*>(srcf) + 2 * ch);
                const float4 b = __ldcg(reinterpret_cast<const float4*>(srcf) + 2 * ch + 1);
                xr[j * 8 + 0] = a.x; xr[j * 8 + 1] = a.y; xr[j * 8 + 2] = a.z; xr[j * 8 + 3] = a.w;
                xr[j * 8 + 4] = b.x; xr[j * 8 + 5] = b.y; xr[j * 8 + 6] = b.z; xr[j * 8 + 7] = b.w;
            } else {
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(srcb) + ch);
                xr[j * 8 + 0] = bf_lo(v.x); xr[j * 8 + 1] = bf_hi(v.x);
                xr[j * 8 + 2] = bf_lo(v.y); xr[j * 8 + 3] = bf_hi(v.y);
                xr[j * 8 + 4] = bf_lo(v.z); xr[j * 8 + 5] = bf_hi(v.z);
                xr[j * 8 + 6] = bf_lo(v.w); xr[j * 8 + 7] = bf_hi(v.w);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(xr[j * 8 + e], xr[j * 8 + e], ss);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) xr[j * 8 + e] = 0.f;
        }
    }
    if (gain) {
        const float tot = cons_block_sum(c, ss);
        const float scale = rsqrtf(tot / float(K) + c.p.rms_eps);
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
            const int ch = c.tid + 256 * j;
            if (ch < rowchunks) {
                const uint4 g = __ldg(reinterpret_cast<const uint4*>(gain) + ch);
                xr[j * 8 + 0] = (xr[j * 8 + 0] * scale) * bf_lo(g.x);
                xr[j * 8 + 1] = (xr[j * 8 + 1] * scale) * bf_hi(g.x);
                xr[j * 8 + 2] = (xr[j * 8 + 2] * scale) * bf_lo(g.y);
                xr[j * 8 + 3] = (xr[j * 8 + 3] * scale) * bf_hi(g.y);
                xr[j * 8 + 4] = (xr[j * 8 + 4] * scale) * bf_lo(g.z);
                xr[j * 8 + 5] = (xr[j * 8 + 5] * scale) * bf_hi(g.z);
                xr[j * 8 + 6] = (xr[j * 8 + 6] * scale) * bf_lo(g.w);
                xr[j * 8 + 7] = (xr[j * 8 + 7] * scale) * bf_hi(g.w);
            }
        }
    }
}

// Matvec tile: rows of a row-major bf16 matrix (the stream in the leased pages) times the
// thread-distributed input x.  Thread t owns the 16-byte column chunks t, t+256, ... of every
// row, so x stays in registers across rows and across consecutive tiles with the same input.
// Row sums: per-thread partials -> an 8-row butterfly inside the warp -> fixed-order sum over
// the 8 warps.  The order depends only on K, never on the tile or the SM.
template <int NCH>
__device__ void matvec_tile(Cons& c, const SlotInfo& si, int pc, float (&xr)[64], int& xkey) {
    const Params& p = c.p;
    const int op = si.w[W_OP], l = si.w[W_LAYER], a0 = si.w[W_A0], n = si.w[W_A1];
    int K, nrows;
    switch (op) {
        case OP_QKV: K = p.H; nrows = n; break;
        case OP_OPROJ: K = p.qd; nrows = n; break;
        case OP_UPGATE: K = p.H; nrows = 2 * n; break;
        case OP_DOWN: K = p.F; nrows = n; break;
        default: K = p.H; nrows = n; break;   // LM head
    }
    const int rowchunks = K / 8;
    const uint32_t rowbytes = uint32_t(K) * 2u;
    const uint32_t first_slot = uint32_t(si.first_page) % uint32_t(p.n_pages);
    const bool pages_ok = wait_pages(c, si, pc);
    (void)pages_ok;   // a failed wait already set the abort flag; the loop exits at the next barrier
    for (int b = 0; b < p.B; ++b) {
        // ---- input vector (cached across tiles with the same key) ----
        const float* srcf = nullptr;
        const uint16_t* srcb = nullptr;
        const uint16_t* gain = nullptr;
        const size_t lb = size_t(l) * p.B + b;
        switch (op) {
            case OP_QKV:
                gain = p.layers[l].attn_norm;
                if (l == 0) srcb = p.embed + size_t(p.tok[b]) * p.H;
                else srcf = p.x_out + (lb - p.B) * p.H;
                break;
            case OP_OPROJ: srcf = p.o + lb * p.qd; break;
            case OP_UPGATE: gain = p.layers[l].mlp_norm; srcf = p.x_attn + lb * p.H; break;
            case OP_DOWN: srcf = p.h + lb * p.F; break;
            default: gain = p.final_norm; srcf = p.x_out + (size_t(p.L - 1) * p.B + b) * p.H; break;
        }
        const int key = ((op * 64 + (l & 63)) * kMaxBatch + b) + 1;
        if (key != xkey) {
            load_x<NCH>(c, xr, K, srcf, srcb, gain);
            xkey = key;
        }
        // ---- accumulate ----
        float acc[kMaxRows];
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
            acc[r] = 0.f;
            if (r < nrows) {
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                    const int ch = c.tid + 256 * j;
                    if (ch < rowchunks) {
                        const uint4 v = *reinterpret_cast<const uint4*>(
                            ring_ptr(c.sh, p, first_slot, uint32_t(r) * rowbytes + uint32_t(ch) * 16u));
                        acc[r] = dot8(v, &xr[j * 8], acc[r]);
                    }
                }
            }
        }
        if (b == p.B - 1) release_pages(c, si);
        // ---- 8-row butterfly: lane ends with the warp sum of row (lane >> 2) & 7 ----
        {
            const bool b4 = (c.lane >> 4) & 1, b3 = (c.lane >> 3) & 1, b2 = (c.lane >> 2) & 1;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float send = b4 ? acc[i] : acc[i + 4];
                const float keep = b4 ? acc[i + 4] : acc[i];
                acc[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float send = b3 ? acc[i] : acc[i + 2];
                const float keep = b3 ? acc[i + 2] : acc[i];
                acc[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
            }
            {
                const float send = b2 ? acc[0] : acc[1];
                const float keep = b2 ? acc[1] : acc[0];
                acc[0] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 4);
            }
            acc[0] += __shfl_xor_sync(0xFFFFFFFFu, acc[0], 2);
            acc[0] += __shfl_xor_sync(0xFFFFFFFFu, acc[0], 1);
        }
        float* red = c.sh.red + c.rbuf * (kNumConsumerWarps * kMaxRows);
        if ((c.lane & 3) == 0) red[c.warp * kMaxRows + ((c.lane >> 2) & 7)] = acc[0];
        cons_sync();
        c.rbuf ^= 1;
        auto rowsum = [&](int r) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kNumConsumerWarps; ++w) s += red[w * kMaxRows + r];
            return s;
        };
        // ---- epilogue (warp 0) ----
        if (c.warp == 0) {
            const int r = c.lane;
            switch (op) {
                case OP_QKV:
                    if (r < n) p.qkv[lb * p.nqkv + a0 + r] = rowsum(r);
                    break;
                case OP_OPROJ:
                    if (r < n) {
                        const int row = a0 + r;
                        const float res = (l == 0) ? bf16f(p.embed[size_t(p.tok[b]) * p.H + row])
                                                   : __ldcg(p.x_out + (lb - p.B) * p.H + row);
                        p.x_attn[lb * p.H + row] = res + rowsum(r);
                    }
                    break;
                case OP_UPGATE:
                    if (r < n) {
                        const float gt = rowsum(r), up = rowsum(n + r);
                        p.h[lb * p.F + a0 + r] = gt / (1.0f + expf(-gt)) * up;
                    }
                    break;
                case OP_DOWN:
                    if (r < n) {
                        const int row = a0 + r;
                        p.x_out[lb * p.H + row] = __ldcg(p.x_attn + lb * p.H + row) + rowsum(r);
                    }
                    break;
                default: {   // LM head
                    if (r < n) p.logits[size_t(b) * p.V + a0 + r] = rowsum(r);
                    if (r == 0) {
                        float best = rowsum(0);
                        int bi = 0;
                        for (int k = 1; k < n; ++k) {
                            const float v = rowsum(k);
                            if (v > best) { best = v; bi = k; }
                        }
                        p.lm_part[size_t(b) * p.n_lm + si.w[W_A2]] = make_float2(best, __int_as_float(a0 + bi));
                    }
                    break;
                }
            }
        }
    }
}

// Split-K decode attention over one chunk of KV positions for one (sequence, KV group); the
// chunk that holds pos also applies RoPE to the new k, rounds k and v to bf16 and appends them
// to the cache.  Writes the chunk partial (o[d] unnormalised, m, l) for each query head.
__device__ void attn_tile(Cons& c, const SlotInfo& si, int pc) {
    const Params& p = c.p;
    const int l = si.w[W_LAYER], b = si.w[W_B], g = si.w[W_A0], ch = si.w[W_A1], C = si.w[W_A2];
    const int d = p.d, half = d / 2, hpg = p.hpg;
    const int n_old = attn_old_rows(p, b, ch, C);
    if (n_old < 0) return;   // chunk past pos: no work, no pages
    const int pos = p.pos[b];
    const bool has_new = pos < ch * C + C;
    const int n = n_old + (has_new ? 1 : 0);
    const size_t lb = size_t(l) * p.B + b;
    const float* qkv = p.qkv + lb * p.nqkv;
    const float2* rp = p.rope + size_t(pos) * half;
    // 1. rotate q of the group's heads; RoPE k, round k and v, append them
    for (int idx = c.tid; idx < hpg * half; idx += kConsumerThreads) {
        const int h = idx / half, i = idx % half;
        const float* qh = qkv + size_t(g * hpg + h) * d;
        const float q0 = __ldcg(qh + i), q1 = __ldcg(qh + i + half);
        const float2 cs = rp[i];
        c.sh.qrot[h * d + i] = q0 * cs.x - q1 * cs.y;
        c.sh.qrot[h * d + i + half] = q0 * cs.y + q1 * cs.x;
    }
    if (has_new) {
        const size_t cache = size_t(b) * p.kv_bstride + size_t(l) * p.kv_lstride + size_t(g) * p.kv_hstride +
                             size_t(pos) * d;
        for (int i = c.tid; i < half; i += kConsumerThreads) {
            const float* kh = qkv + p.qd + size_t(g) * d;
            const float k0 = __ldcg(kh + i), k1 = __ldcg(kh + i + half);
            const float2 cs = rp[i];
            const uint16_t r0 = f2bf_rn(k0 * cs.x - k1 * cs.y), r1 = f2bf_rn(k0 * cs.y + k1 * cs.x);
            c.sh.knew[i] = r0;
            c.sh.knew[i + half] = r1;
            p.kc[cache + i] = r0;
            p.kc[cache + i + half] = r1;
        }
        for (int i = c.tid; i < d; i += kConsumerThreads) {
            const uint16_t r = f2bf_rn(__ldcg(qkv + p.qd + p.kvd + size_t(g) * d + i));
            c.sh.vnew[i] = r;
            p.vc[cache + i] = r;
        }
    }
    cons_sync();
    wait_pages(c, si, pc);
    const uint32_t first_slot = uint32_t(si.first_page) % uint32_t(p.n_pages);
    const uint32_t rowb = uint32_t(d) * 2u;
    const uint32_t voff = uint32_t(n_old) * rowb;
    float* sc = c.sh.ascr;   // [hpg][C]
    // 2. scores s[h][t] = (q_h . k_t) * scale; d/8 consecutive lanes share a position
    const int cpr = d / 8;
    for (int base = 0; base < n * cpr; base += kConsumerThreads) {
        const int idx = base + c.tid;
        const bool valid = idx < n * cpr;
        const int t = idx / cpr, j = idx % cpr;
        float part[kMaxHpg];
#pragma unroll
        for (int h = 0; h < kMaxHpg; ++h) part[h] = 0.f;
        if (valid) {
            const uint4 kv = (t < n_old) ? *reinterpret_cast<const uint4*>(ring_ptr(c.sh, p, first_slot, uint32_t(t) * rowb + uint32_t(j) * 16u))
                                         : *reinterpret_cast<const uint4*>(c.sh.knew + j * 8);
#pragma unroll
            for (int h = 0; h < kMaxHpg; ++h)
                if (h < hpg) part[h] = dot8(kv, c.sh.qrot + h * d + j * 8, 0.f);
        }
        for (int o = 1; o < cpr; o <<= 1)
#pragma unroll
            for (int h = 0; h < kMaxHpg; ++h) part[h] += __shfl_xor_sync(0xFFFFFFFFu, part[h], o);
        if (valid && j == 0)
#pragma unroll
            for (int h = 0; h < kMaxHpg; ++h)
                if (h < hpg) sc[h * C + t] = part[h] * p.attn_scale;
    }
    cons_sync();
    // 3. softmax pieces per head (warp h): m, w_t = exp(s_t - m), l = sum w_t
    if (c.warp < hpg) {
        const int h = c.warp;
        float m = -INFINITY;
        for (int t = c.lane; t < n; t += 32) m = fmaxf(m, sc[h * C + t]);
        m = warp_max(m);
        float s = 0.f;
        for (int t = c.lane; t < n; t += 32) {
            const float e = expf(sc[h * C + t] - m);
            sc[h * C + t] = e;
            s += e;
        }
        s = warp_sum(s);
        if (c.lane == 0) { c.sh.ml[2 * h] = m; c.sh.ml[2 * h + 1] = s; }
    }
    cons_sync();
    // 4. o[h][e] = sum_t w_t v_t[e]
    float* dst = p.part + ((lb * p.nkv + g) * p.n_chunk + ch) * size_t(hpg) * (d + 2);
    for (int idx = c.tid; idx < hpg * d; idx += kConsumerThreads) {
        const int h = idx / d, e = idx % d;
        float acc = 0.f;
        for (int t = 0; t < n; ++t) {
            const float v = (t < n_old) ? bf16f(*reinterpret_cast<const uint16_t*>(ring_ptr(c.sh, p, first_slot, voff + uint32_t(t) * rowb + uint32_t(e) * 2u)))
                                        : bf16f(c.sh.vnew[e]);
            acc = fmaf(sc[h * C + t], v, acc);
        }
        float* dh = dst + size_t(h) * (d + 2);
        dh[e] = acc;
        if (e == 0) { dh[d] = c.sh.ml[2 * h]; dh[d + 1] = c.sh.ml[2 * h + 1]; }
    }
    release_pages(c, si);
}

// Fixed-order log-sum-exp combine of the active chunks of one (sequence, group):
// M = max_c m_c, f_c = exp(m_c - M), L = sum_c f_c l_c, o = sum_c f_c o_c / L.
__device__ void comb_tile(Cons& c, const SlotInfo& si) {
    const Params& p = c.p;
    const int l = si.w[W_LAYER], b = si.w[W_B], g = si.w[W_A0], nch = si.w[W_A1], C = si.w[W_A2];
    const int d = p.d, hpg = p.hpg;
    const int nact = min(nch, p.pos[b] / C + 1);
    const size_t lb = size_t(l) * p.B + b;
    const float* base = p.part + (lb * p.nkv + g) * size_t(p.n_chunk) * hpg * (d + 2);
    float* fac = c.sh.ascr;   // [hpg][n_chunk]
    if (c.warp < hpg) {
        const int h = c.warp;
        float M = -INFINITY;
        for (int k = c.lane; k < nact; k += 32) M = fmaxf(M, __ldcg(base + (size_t(k) * hpg + h) * (d + 2) + d));
        M = warp_max(M);
        float Ls = 0.f;
        for (int k = c.lane; k < nact; k += 32) {
            const float* ph = base + (size_t(k) * hpg + h) * (d + 2);
            const float f = expf(__ldcg(ph + d) - M);
            fac[h * p.n_chunk + k] = f;
            Ls = fmaf(f, __ldcg(ph + d + 1), Ls);
        }
        Ls = warp_sum(Ls);
        if (c.lane == 0) c.sh.cml[h] = Ls;
    }
    cons_sync();
    float* out = p.o + lb * p.qd + size_t(g) * hpg * d;
    for (int idx = c.tid; idx < hpg * d; idx += kConsumerThreads) {
        const int h = idx / d, e = idx % d;
        float acc = 0.f;
        for (int k = 0; k < nact; ++k) acc = fmaf(fac[h * p.n_chunk + k], __ldcg(base + (size_t(k) * hpg + h) * (d + 2) + e), acc);
        out[idx] = acc / c.sh.cml[h];
    }
}

// Greedy token: argmax over the LM-head tile partials (largest value, lowest index on ties).
__device__ void argmax_tile(Cons& c, const SlotInfo& si) {
    const Params& p = c.p;
    const int b = si.w[W_B], n = si.w[W_A1];
    const float2* parts = p.lm_part + size_t(b) * p.n_lm;
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int i = c.tid; i < n; i += kConsumerThreads) {
        const float2 v = __ldcg(parts + i);
        const int idx = __float_as_int(v.y);
        if (v.x > bv || (v.x == bv && idx < bi)) { bv = v.x; bi = idx; }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    float* red = c.sh.red + c.rbuf * (kNumConsumerWarps * kMaxRows);
    if (c.lane == 0) { red[2 * c.warp] = bv; red[2 * c.warp + 1] = __int_as_float(bi); }
    cons_sync();
    c.rbuf ^= 1;
    if (c.tid == 0) {
        for (int w = 0; w < kNumConsumerWarps; ++w) {
            const float ov = red[2 * w];
            const int oi = __float_as_int(red[2 * w + 1]);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        p.tokens_out[b] = bi;
        if (p.next_dev) p.next_dev[b] = bi;
    }
}

__device__ bool wait_counters(const Params& p, const Shared& sh, const int32_t* w, int pc) {
    const int nw = w[W_NWAIT];
    for (int i = 0; i < nw; ++i) {
        const int cid = w[W_WAIT + 2 * i];
        const uint32_t target = p.epoch * __ldg(p.totals + cid) + uint32_t(w[W_WAIT + 2 * i + 1]);
        uint32_t v = ld_relaxed_gpu(p.counters + cid);
        if (int32_t(v - target) >= 0) continue;
        const uint64_t t0 = globaltimer();
        while (true) {
            v = ld_relaxed_gpu(p.counters + cid);
            if (int32_t(v - target) >= 0) break;
            if (*reinterpret_cast<volatile int*>(sh.abort) || ld_relaxed_gpu(reinterpret_cast<const uint32_t*>(p.err))) {
                *reinterpret_cast<volatile int*>(sh.abort) = 1;
                return false;
            }
            if (globaltimer() - t0 > p.timeout_ns) {
                raise_error(p, sh, MK_ERR_TIMEOUT, ROLE_COUNTER, pc, cid, v, target);
                return false;
            }
        }
    }
    fence_acq_rel_gpu();   // acquire: producers' data is visible before any consumer reads it
    return true;
}

template <int NCH>
__device__ void consumer_loop(const Params& p, const Shared& sh) {
    Cons c{p, sh, int(threadIdx.x), int(threadIdx.x) >> 5, int(threadIdx.x) & 31, 0};
    float xr[64];
    int xkey = -1;
    for (int pc = 0;; ++pc) {
        const int slot = pc % kSlots;
        bool ok = wait_bar(p, sh, sh.ins_full + slot, (pc / kSlots) & 1, ROLE_CONSUMER, pc);
        const SlotInfo& si = sh.slots[slot];
        const int op = ok ? si.w[W_OP] : OP_END;
        if (ok && op != OP_END && c.tid == 0) ok = wait_counters(p, sh, si.w, pc);
        const bool stop = cons_sync_or(!ok || *reinterpret_cast<volatile int*>(sh.abort) != 0);
        if (stop) break;
        switch (op) {
            case OP_QKV:
            case OP_OPROJ:
            case OP_UPGATE:
            case OP_DOWN:
            case OP_LMHEAD: matvec_tile<NCH>(c, si, pc, xr, xkey); break;
            case OP_ATTN: attn_tile(c, si, pc); break;
            case OP_COMB: comb_tile(c, si); break;
            case OP_ARGMAX: argmax_tile(c, si); break;
            default: break;   // END
        }
        __syncwarp();
        if (c.lane == 0) mbar_arrive(sh.done + slot);
        if (op == OP_END) break;
    }
}

template <int NCH>
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
            mbar_init(sh.ins_empty + i, 1);
            mbar_init(sh.done + i, kNumConsumerWarps);
        }
        *sh.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < kNumConsumerWarps) consumer_loop<NCH>(p, sh);
    else if (warp == kLoaderWarp) { if (lane == 0) loader(p, sh); }
    else if (lane == 0) publisher(p, sh);
    cta_sync_divergent();
}

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

// x chunks per thread: ceil(K / 8 / 256) for the longest matvec row of the model
static const void* kernel_for(int nch) {
    switch (nch) {
        case 1: return reinterpret_cast<const void*>(&megakernel<1>);
        case 2: return reinterpret_cast<const void*>(&megakernel<2>);
        case 3: return reinterpret_cast<const void*>(&megakernel<3>);
        case 4: return reinterpret_cast<const void*>(&megakernel<4>);
        case 5: return reinterpret_cast<const void*>(&megakernel<5>);
        case 6: return reinterpret_cast<const void*>(&megakernel<6>);
        case 7: return reinterpret_cast<const void*>(&megakernel<7>);
        case 8: return reinterpret_cast<const void*>(&megakernel<8>);
        default: return nullptr;
    }
}

const void* megakernel_fn(int nch) { return kernel_for(nch); }

cudaError_t launch_rope_table(float2* out, int max_seq, int d, double theta, cudaStream_t st) {
    const int n = max_seq * (d / 2);
    const int blocks = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
    rope_table_kernel<<<blocks, 256, 0, st>>>(out, max_seq, d, theta);
    return cudaGetLastError();
}

}  // namespace mk
