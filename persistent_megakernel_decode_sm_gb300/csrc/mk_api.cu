// C ABI: bind a schedule to one model instance, launch the resident grid, read back status.
//
// Binding follows the page "Inference MegaKernel" (section "Hand-written whole-model
// MegaKernel": one model-specific binding passes weights, KV cache, activations and counters
// as objects of the resident execution) and checks two of its four device-protocol contracts
// (section "Unified framework") before any launch:
//   capacity  -- the largest tile's stream fits the shared-memory page ring, every pos < max_seq;
//   resources -- one CTA with the kernel's registers and shared memory is resident on each of
//                the S SMs (the launch is cooperative, so an oversubscribed grid fails instead of
//                deadlocking: the forward-progress contract).
#include <cuda.h>   // tensor-map types (the encoder itself is fetched through the runtime)
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <type_traits>

#include <atomic>

#include "mk_internal.h"

namespace mk {
const void* megakernel_fn(int cpl);
cudaError_t launch_rope_table(float2* out, int max_seq, int d, double theta, cudaStream_t st);
}  // namespace mk
namespace mk_bat {
const void* megakernel_fn_batched();   // (mk_kernel_batch.cu: the same kernel source, batch > 1)
}

using namespace mk;

struct mk_ctx {
    Params base;
    const void* fn;
    int grid, smem;
    cudaStream_t stream;
    int device;
    int32_t* d_queues;
    uint32_t* d_totals;
    LayerPtrs* d_layers;
    int32_t* h_result;   // pinned: err[16] then tokens[8]
    uint32_t epoch;
    bool poisoned;
    // a step ran on the static scratch: the bound scratch's activation words did not advance with
    // the epoch (the 3-bit SwiGLU tag repeats every 7 steps), so it is cleared before its next use
    bool bound_stale;
    const int32_t* last_err;   // error word of the last launched step (bound or static scratch)
    uint8_t* d_tmaps;          // batch > 1: the weights' TMA tensor maps
    uint32_t* d_step_bar;      // grid-wide step word: each CTA adds 1 per step it retires
    volatile int32_t* h_ctl;   // mapped pinned words: [0] stop request (host), [1] steps done (device)
    int32_t* d_ctl;            // their device address
    // a persistent launch in flight: its step budget and token buffer (the epoch advances by the
    // steps it ran, known only once it has ended)
    bool run_active;
    int32_t run_steps;
    const int32_t* run_tokens;
    mk_model_cfg cfg;
    // what a schedule switch (mk_rebind_schedule) needs: the bound weights (pointer tables copied),
    // the geometry and counter totals of the bound schedule, its KV windows per sequence
    mk_weights w;
    std::vector<const void*> wtab;   // the per-layer pointer tables behind w
    Geometry geo;
    int32_t S;
    std::vector<uint32_t> totals;
    size_t queue_words;               // capacity of d_queues in words
};

static mk_status cuda_fail(cudaError_t e, const char* what) {
    return fail(MK_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// batch > 1: TMA tensor maps over the matvec weights.  A [R][K] bf16 matrix is described as the
// 3-d tensor [R][K / g0][g0] (mmv_g0) with a box of (g0, kp / g0, rows): one box is one page of
// the ring, a block of rows over kp positions, rows 2 kp bytes apart; rows past R read as zeros
static_assert(sizeof(CUtensorMap) == 128, "tensor maps are indexed in 128-byte records");
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static mk_status weight_map(EncodeTiledFn enc, CUtensorMap* out, const void* base, int64_t R, int64_t K, int kp,
                            int rows) {
    const int g0 = mmv_g0(int(K), kp);
    if (reinterpret_cast<uintptr_t>(base) % 16 || K % 8)
        return fail(MK_ERR_ARG, "batch > 1 needs 16-byte aligned weight matrices with rows of a multiple of 8");
    const cuuint64_t dim[3] = {cuuint64_t(g0), cuuint64_t(K / g0), cuuint64_t(R)};
    const cuuint64_t stride[2] = {cuuint64_t(g0) * 2u, cuuint64_t(K) * 2u};
    const cuuint32_t box[3] = {cuuint32_t(g0), cuuint32_t(kp / g0), cuuint32_t(rows)};
    const cuuint32_t es[3] = {1u, 1u, 1u};
    const CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3u, const_cast<void*>(base), dim, stride, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled: error %d", int(r));
    return MK_OK;
}
#define CK(call)                                    \
    do {                                            \
        cudaError_t e_ = (call);                    \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
    } while (0)

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static void free_ctx(mk_ctx* c) {
    if (!c) return;
    if (c->d_queues) cudaFree(c->d_queues);
    if (c->d_totals) cudaFree(c->d_totals);
    if (c->d_layers) cudaFree(c->d_layers);
    if (c->h_result) cudaFreeHost(c->h_result);
    if (c->d_step_bar) cudaFree(c->d_step_bar);
    if (c->d_tmaps) cudaFree(c->d_tmaps);
    if (c->h_ctl) cudaFreeHost(const_cast<int32_t*>(c->h_ctl));
    delete c;
}

extern "C" mk_status mk_device_sm_count(int32_t* out) {
    if (!out) return fail(MK_ERR_ARG, "null argument");
    int dev = 0, n = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev));
    *out = n;
    return MK_OK;
}

// Device copy of the queues: validates every instruction of a known opcode against the model (the
// device then trusts those fields) and writes the resolved weight stream of each matvec tile into
// words 26..31 (source addresses and byte counts), so the loader on the device does no decoding.
// Unknown opcodes are copied as they are: the device rejects them (MK_ERR_OPCODE).
static mk_status resolve_queues(const mk_schedule* s, const mk_weights* w, const MvShape* mv, int kp,
                                std::vector<int32_t>& dq) {
    const mk_model_cfg& c = s->cfg;
    const Geometry& g = s->geo;
    const int L = c.n_layers, H = c.hidden, F = c.ffn, V = c.vocab, B = c.batch, nkv = c.n_kv_heads;
    const int qd = c.n_q_heads * c.head_dim, nqkv = qd + 2 * nkv * c.head_dim;
    dq = s->queues;
    auto put64 = [](int32_t* w2, const void* ptr) {
        const uint64_t v = reinterpret_cast<uint64_t>(ptr);
        w2[0] = int32_t(uint32_t(v));
        w2[1] = int32_t(uint32_t(v >> 32));
    };
    for (size_t i = 0; i < dq.size(); i += kWords) {
        int32_t* x = &dq[i];
        const int op = x[W_OP];
        if (op == OP_END || op < 0 || op >= OP_COUNT) continue;
        const int l = x[W_LAYER], b = x[W_B], a0 = x[W_A0], a1 = x[W_A1], a2 = x[W_A2];
        const long slot = long(i / kWords);
        auto bad = [&](const char* what) {
            return fail(MK_ERR_BOUNDS, "queue %ld slot %ld: %s", slot / s->Q, slot % s->Q, what);
        };
        if (x[W_NWAIT] < 0 || x[W_NWAIT] > kMaxWait || x[W_NPUB] < 0 || x[W_NPUB] > kMaxPub) return bad("wait/completion count");
        for (int k = 0; k < x[W_NWAIT]; ++k)
            if (unsigned(x[W_WAIT + 2 * k]) >= unsigned(g.n_counters)) return bad("counter id");
        for (int k = 0; k < x[W_NPUB]; ++k)
            if (unsigned(x[W_PUB + 2 * k]) >= unsigned(g.n_counters)) return bad("counter id");
        const bool head = op == OP_LMHEAD || op == OP_ARGMAX;
        if (head ? l != L : unsigned(l) >= unsigned(L)) return bad("layer");
        if (unsigned(b) >= unsigned(B)) return bad("sequence");
        auto rows = [&](int total, int maxn) { return a0 >= 0 && a1 >= 1 && a1 <= maxn && int64_t(a0) + a1 <= total; };
        const void* src0 = nullptr;
        const void* src1 = nullptr;
        int64_t b0 = 0, b1 = 0;
        switch (op) {
            case OP_QKV:
                if (!rows(nqkv, c.head_dim)) return bad("rows");
                src0 = static_cast<const uint8_t*>(w->wqkv[l]) + int64_t(a0) * H * 2;
                b0 = int64_t(a1) * H * 2;
                break;
            case OP_OPROJ:
                if (!rows(H, H)) return bad("rows");
                src0 = static_cast<const uint8_t*>(w->wo[l]) + int64_t(a0) * qd * 2;
                b0 = int64_t(a1) * qd * 2;
                break;
            case OP_UPGATE:
                if (!rows(F, F)) return bad("rows");
                src0 = static_cast<const uint8_t*>(w->wgate_up[l]) + int64_t(a0) * H * 2;
                src1 = static_cast<const uint8_t*>(w->wgate_up[l]) + int64_t(F + a0) * H * 2;
                b0 = b1 = int64_t(a1) * H * 2;
                break;
            case OP_DOWN:   // (batch > 1, rows longer than kMmvRange: a2 = the tile's staging range)
                if (!rows(H, H) || unsigned(a2) >= unsigned(mmv_down_ranges(B, F))) return bad("rows");
                src0 = static_cast<const uint8_t*>(w->wdown[l]) + int64_t(a0) * F * 2;
                b0 = int64_t(a1) * F * 2;
                break;
            case OP_LMHEAD:
                if (!rows(V, V) || unsigned(a2) >= unsigned(g.n_lm)) return bad("rows");
                src0 = static_cast<const uint8_t*>(w->lm_head) + int64_t(a0) * H * 2;
                b0 = int64_t(a1) * H * 2;
                break;
            case OP_ATTN:   // (batch 1: the chunk holding pos combines; batch > 1: COMB tiles do)
                if (unsigned(a0) >= unsigned(nkv) || unsigned(a1) >= unsigned(g.n_chunk) || a2 != g.attn_chunk ||
                    x[W_COND] != (B == 1 ? 1 : 0))
                    return bad("attention fields");
                break;
            case OP_COMB:
                if (B == 1 || unsigned(a0) >= unsigned(nkv) || a1 != 0 || a2 != g.attn_chunk || x[W_COND] != 0 ||
                    x[W_NPAGES] != 0)
                    return bad("combine fields");
                break;
            case OP_ARGMAX:
                if (a1 != g.n_lm) return bad("argmax fields");
                break;
            default: break;
        }
        if (src0) {   // whole rows (or row slices) per page; gate/up: gate and up row groups alternate
            if (mv[op].rpp < 1) return bad("a page holds no row");
            if (kp && mv[op].K > kMmvRange && a1 > 64) return bad("rows of a tile over several ranges");   // (<= 4 blocks)
            const int64_t pages = (op == OP_DOWN && mmv_down_ranges(B, F) > 1)
                                      ? mmv_range_pages(F, kp, a1, a2) : mv_tile_pages(mv[op], kp, a1, op == OP_UPGATE);
            if (pages != x[W_NPAGES] || b0 + b1 > (int64_t(1) << 31) - 1) return bad("page count");
            put64(x + W_SRC0, src0);
            put64(x + W_SRC1, src1);
            x[W_BYTES0] = int32_t(b0);
            x[W_BYTES1] = int32_t(b1);
        }
    }
    return MK_OK;
}

extern "C" mk_status mk_bind(const mk_schedule* s, const mk_weights* w, const mk_kv* kv, uint32_t* counters,
                             void* scratch, void* stream, mk_ctx** out) {
    return mk_bind_paged(s, w, kv, nullptr, counters, scratch, stream, out);
}

extern "C" mk_status mk_bind_paged(const mk_schedule* s, const mk_weights* w, const mk_kv* kv,
                                   const mk_kv_pages* pages, uint32_t* counters, void* scratch, void* stream,
                                   mk_ctx** out) {
    if (!s || !w || !kv || !counters || !scratch || !out) return fail(MK_ERR_ARG, "null argument");
    *out = nullptr;
    const mk_model_cfg& c = s->cfg;
    const Geometry& g = s->geo;
    const int L = c.n_layers, H = c.hidden, d = c.head_dim, hpg = c.n_q_heads / c.n_kv_heads;
    const int qd = c.n_q_heads * d;

    // ---- arguments ----
    if (!w->embed || !w->lm_head || !w->final_norm || !w->attn_norm || !w->wqkv || !w->wo || !w->mlp_norm ||
        !w->wgate_up || !w->wdown)
        return fail(MK_ERR_ARG, "mk_weights has a null field");
    const void* ptrs[3] = {w->embed, w->lm_head, w->final_norm};
    for (const void* p : ptrs)
        if (!aligned16(p)) return fail(MK_ERR_ARG, "weight pointer not 16-byte aligned");
    for (int l = 0; l < L; ++l) {
        const void* lp[6] = {w->attn_norm[l], w->wqkv[l], w->wo[l], w->mlp_norm[l], w->wgate_up[l], w->wdown[l]};
        for (const void* p : lp)
            if (!p || !aligned16(p)) return fail(MK_ERR_ARG, "layer %d weight pointer null or not 16-byte aligned", l);
    }
    if (!kv->k || !kv->v || !aligned16(kv->k) || !aligned16(kv->v))
        return fail(MK_ERR_ARG, "KV pointers null or not 16-byte aligned");
    if (pages) {   // a pool of blocks per (layer, KV head), reached through the block table
        if (!pages->block_table || (reinterpret_cast<uintptr_t>(pages->block_table) & 3u))
            return fail(MK_ERR_ARG, "block table null or not 4-byte aligned");
        if (pages->block_size != g.attn_chunk)
            return fail(MK_ERR_ARG, "block_size %d must equal the schedule's attention chunk %d", pages->block_size,
                        g.attn_chunk);
        if (pages->n_blocks < 1 || int64_t(pages->max_blocks) * pages->block_size < c.max_seq)
            return fail(MK_ERR_ARG, "the block table must cover max_seq positions and the pool hold a block");
        if (kv->layer_stride % 8 || kv->head_stride % 8 ||
            kv->head_stride < int64_t(pages->n_blocks) * pages->block_size * d ||
            kv->layer_stride < kv->head_stride * c.n_kv_heads)
            return fail(MK_ERR_ARG, "KV strides must be multiples of 8 elements and cover the pool per head");
    } else if (kv->batch_stride % 8 || kv->layer_stride % 8 || kv->head_stride % 8 ||
               kv->head_stride < int64_t(c.max_seq) * d || kv->layer_stride < kv->head_stride * c.n_kv_heads ||
               (c.batch > 1 && kv->batch_stride < kv->layer_stride * L)) {
        return fail(MK_ERR_ARG, "KV strides must be multiples of 8 elements and cover [max_seq, head_dim] per head");
    }
    if (reinterpret_cast<uintptr_t>(scratch) & 255u) return fail(MK_ERR_ARG, "scratch must be 256-byte aligned");
    if (reinterpret_cast<uintptr_t>(counters) & 3u) return fail(MK_ERR_ARG, "counters must be 4-byte aligned");
    if (g.page_bytes & (g.page_bytes - 1)) return fail(MK_ERR_ARG, "page_bytes must be a power of two");
    if (L > kMaxLayersSmem) return fail(MK_ERR_ARG, "more than %d layers", kMaxLayersSmem);

    // ---- device and resources ----
    int dev = 0, sms = 0, optin = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    CK(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
    if (s->S > sms) return fail(MK_ERR_RESOURCES, "schedule has %d queues but the device has %d SMs", s->S, sms);
    // shared input buffer: the hidden size (the normed inputs) and at least kMinXBuf floats (the
    // attention's scores and combine); matvec inputs longer than it are polled per warp
    int xbuf = std::max(kMinXBuf, H);
    if (c.batch > 1) {   // every sequence's staged inputs for one range of positions, then the partials
        if (H > kMmvRange)
            return fail(MK_ERR_ARG, "batch > 1 needs hidden <= %d (the RMSNorm inputs are staged in one range)", kMmvRange);
        const int kmx = std::max(H, std::max(qd, c.ffn));
        const uint32_t stage = uint32_t(c.batch) * mmv_row_stride(std::min(kmx, kMmvRange));
        xbuf = std::max(xbuf, int((stage + kMmvPartBytes) / 4u));
    }
    {   // attention: scores [hpg][C], weights [C][hp], per consumer warp an output partial [hp][d]
        // and its (m, l) per head
        const int hp = hpg <= 4 ? 4 : kMaxHpg;
        xbuf = std::max(xbuf, ((hpg * g.attn_chunk + 3) & ~3) + g.attn_chunk * hp + kNumConsumerWarps * hp * (d + 2));
    }
    if (hpg * g.attn_chunk > xbuf)
        return fail(MK_ERR_ARG, "attn_chunk %d: the scores of %d heads do not fit %d floats", g.attn_chunk, hpg, xbuf);
    // matvec shapes: whole rows per page, segments per row (a property of the row length only)
    // chunks per lane: 4 when every row fits kMaxSeg segments of 128 chunks, else 8
    const int kmax = std::max(H, std::max(qd, c.ffn));
    const int cpl = (kmax / 8 + kMaxSeg - 1) / kMaxSeg <= 128 ? 4 : kMaxCpl;
    MvShape mv[OP_COUNT] = {};
    // batch > 1: a page holds a 16-row block over kp positions (kp divides kMmvRange, MMA steps of 32)
    const int kp = c.batch > 1 ? g.page_bytes / 32 : 0;
    if (c.batch > 1 && (kp < 32 || kp > kMmvRange))
        return fail(MK_ERR_ARG, "batch > 1 needs page_bytes in [1024, %d]", 32 * kMmvRange);
    int comb_stride = 1;
    for (int op : {int(OP_QKV), int(OP_OPROJ), int(OP_UPGATE), int(OP_DOWN), int(OP_LMHEAD)}) {
        const int K = op == OP_OPROJ ? qd : (op == OP_DOWN ? c.ffn : H);
        mv[op] = mv_shape(K, cpl, g.page_bytes, xbuf);
        if (mv[op].segch > 32 * cpl)
            return fail(MK_ERR_ARG, "matvec row length %d cannot be cut into %d segments", K, kMaxSeg);
        if (c.batch == 1)
            comb_stride = std::max(comb_stride, mv[op].rpp * mv[op].G);   // (row, segment) units of a page
        else
            mv[op].rpp = 16;   // (a block of rows over kp positions)
        if (mv[op].rpp < 1)
            return fail(MK_ERR_CAPACITY, "a %d-byte page holds no %d-element row", g.page_bytes, K);
    }
    const void* fn = c.batch > 1 ? mk_bat::megakernel_fn_batched() : megakernel_fn(cpl);
    const int qrf = (hpg * d + 3) & ~3;
    int n_pages = 0;
    while (n_pages < kMaxRingPages &&
           int64_t(n_pages + 1) * g.page_bytes + smem_misc_bytes(n_pages + 1, qrf, xbuf, comb_stride) <= optin)
        ++n_pages;
    if (n_pages < 1) return fail(MK_ERR_CAPACITY, "no room for a page ring");
    const int misc = smem_misc_bytes(n_pages, qrf, xbuf, comb_stride);
    // capacity: a matvec tile streams through the ring one group of two pages at a time; an
    // attention tile holds its K and V rows
    const int need_pages = std::max<int>(2, int((2ll * g.attn_chunk * d * 2 + g.page_bytes - 1) / g.page_bytes));
    if (n_pages < need_pages)
        return fail(MK_ERR_CAPACITY, "page ring of %d pages cannot hold the %d pages a step needs", n_pages, need_pages);
    const int smem = n_pages * g.page_bytes + misc;
    CK(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    int per_sm = 0;
    CK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem));
    if (per_sm < 1) return fail(MK_ERR_RESOURCES, "the kernel cannot be resident (%d B shared memory)", smem);

    // ---- context ----
    mk_ctx* x = new mk_ctx();   // (value-initialised: every scalar field zero)
    x->cfg = c;
    x->fn = fn;
    x->grid = s->S;
    x->smem = smem;
    x->stream = static_cast<cudaStream_t>(stream);
    x->device = dev;
    x->geo = g;
    x->S = s->S;
    x->totals = s->totals;
    x->queue_words = s->queues.size();
    {   // the weights' pointer tables, for resolving another schedule's queues later
        x->wtab.reserve(size_t(6) * L);
        const void* const* tabs[6] = {w->attn_norm, w->wqkv, w->wo, w->mlp_norm, w->wgate_up, w->wdown};
        for (auto* t : tabs) x->wtab.insert(x->wtab.end(), t, t + L);
        x->w = *w;
        x->w.attn_norm = &x->wtab[0];
        x->w.wqkv = &x->wtab[size_t(L)];
        x->w.wo = &x->wtab[size_t(2) * L];
        x->w.mlp_norm = &x->wtab[size_t(3) * L];
        x->w.wgate_up = &x->wtab[size_t(4) * L];
        x->w.wdown = &x->wtab[size_t(5) * L];
    }
    auto bail = [&](mk_status st) { free_ctx(x); return st; };
    cudaError_t e;
    const size_t qbytes = s->queues.size() * sizeof(int32_t);
    if ((e = cudaMalloc(&x->d_queues, qbytes)) != cudaSuccess) return bail(cuda_fail(e, "cudaMalloc(queues)"));
    if ((e = cudaMalloc(&x->d_totals, s->totals.size() * 4)) != cudaSuccess) return bail(cuda_fail(e, "cudaMalloc(totals)"));
    if ((e = cudaMalloc(&x->d_layers, sizeof(LayerPtrs) * L)) != cudaSuccess) return bail(cuda_fail(e, "cudaMalloc(layers)"));
    if ((e = cudaMallocHost(&x->h_result, 256)) != cudaSuccess) return bail(cuda_fail(e, "cudaMallocHost"));
    if ((e = cudaMalloc(&x->d_step_bar, 4)) != cudaSuccess) return bail(cuda_fail(e, "cudaMalloc(step word)"));
    {
        int32_t* ctl = nullptr;
        if ((e = cudaHostAlloc(&ctl, 64, cudaHostAllocMapped)) != cudaSuccess)
            return bail(cuda_fail(e, "cudaHostAlloc(control words)"));
        x->h_ctl = ctl;
        ctl[0] = ctl[1] = 0;
        if ((e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&x->d_ctl), ctl, 0)) != cudaSuccess)
            return bail(cuda_fail(e, "cudaHostGetDevicePointer(control words)"));
    }
    if (c.batch > 1) {   // tensor maps over every matvec weight matrix
        cudaDriverEntryPointQueryResult q{};
        void* fnp = nullptr;
        if ((e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fnp, 12000, cudaEnableDefault, &q)) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess || !fnp)
            return bail(fail(MK_ERR_CUDA, "cuTensorMapEncodeTiled is not available"));
        const EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(fnp);
        std::vector<CUtensorMap> maps(size_t(4) * L + 1);
        for (int l = 0; l < L; ++l) {
            mk_status st = weight_map(enc, &maps[4 * l + 0], w->wqkv[l], qd + 2 * c.n_kv_heads * d, H, kp, 16);
            if (st == MK_OK) st = weight_map(enc, &maps[4 * l + 1], w->wo[l], H, qd, kp, 16);
            if (st == MK_OK) st = weight_map(enc, &maps[4 * l + 2], w->wgate_up[l], 2 * int64_t(c.ffn), H, kp, 8);
            if (st == MK_OK) st = weight_map(enc, &maps[4 * l + 3], w->wdown[l], H, c.ffn, kp, 16);
            if (st != MK_OK) return bail(st);
        }
        {
            const mk_status st = weight_map(enc, &maps[4 * L], w->lm_head, c.vocab, H, kp, 16);
            if (st != MK_OK) return bail(st);
        }
        const size_t mb = maps.size() * sizeof(CUtensorMap);
        if ((e = cudaMalloc(&x->d_tmaps, mb)) != cudaSuccess) return bail(cuda_fail(e, "cudaMalloc(tensor maps)"));
        if ((e = cudaMemcpy(x->d_tmaps, maps.data(), mb, cudaMemcpyHostToDevice)) != cudaSuccess)
            return bail(cuda_fail(e, "cudaMemcpy(tensor maps)"));
    }
    std::vector<LayerPtrs> lp(L);
    for (int l = 0; l < L; ++l)
        lp[l] = {static_cast<const uint16_t*>(w->attn_norm[l]), static_cast<const uint16_t*>(w->wqkv[l]),
                 static_cast<const uint16_t*>(w->wo[l]), static_cast<const uint16_t*>(w->mlp_norm[l]),
                 static_cast<const uint16_t*>(w->wgate_up[l]), static_cast<const uint16_t*>(w->wdown[l])};
    std::vector<int32_t> dq;
    {
        const mk_status rs = resolve_queues(s, w, mv, kp, dq);
        if (rs != MK_OK) return bail(rs);
    }
    if ((e = cudaMemcpy(x->d_queues, dq.data(), qbytes, cudaMemcpyHostToDevice)) != cudaSuccess ||
        (e = cudaMemcpy(x->d_totals, s->totals.data(), s->totals.size() * 4, cudaMemcpyHostToDevice)) != cudaSuccess ||
        (e = cudaMemcpy(x->d_layers, lp.data(), sizeof(LayerPtrs) * L, cudaMemcpyHostToDevice)) != cudaSuccess)
        return bail(cuda_fail(e, "cudaMemcpy(bind tables)"));

    const ScratchLayout sl = scratch_layout(c, g, s->S);
    uint8_t* sb = static_cast<uint8_t*>(scratch);
    Params& p = x->base;
    for (int op = 0; op < OP_COUNT; ++op) p.mv[op] = mv[op];
    p.mmv_kp = kp;
    p.tmaps = x->d_tmaps;
    p.L = L; p.H = H; p.nq = c.n_q_heads; p.nkv = c.n_kv_heads; p.d = d; p.F = c.ffn; p.V = c.vocab;
    p.B = c.batch; p.max_seq = c.max_seq; p.hpg = hpg; p.qd = qd; p.kvd = c.n_kv_heads * d;
    p.nqkv = qd + 2 * p.kvd;
    p.rms_eps = float(c.rms_eps);
    p.attn_scale = float(1.0 / std::sqrt(double(d)));
    p.page_bytes = g.page_bytes;
    p.page_shift = 0;
    while ((1 << p.page_shift) < g.page_bytes) ++p.page_shift;
    p.n_pages = n_pages;
    p.attn_chunk = g.attn_chunk;
    p.n_chunk = g.n_chunk;
    p.n_lm = g.n_lm;
    p.queues = x->d_queues;
    p.Q = s->Q;
    p.n_counters = g.n_counters;
    p.totals = x->d_totals;
    p.counters = counters;
    p.embed = static_cast<const uint16_t*>(w->embed);
    p.lm_head = static_cast<const uint16_t*>(w->lm_head);
    p.final_norm = static_cast<const uint16_t*>(w->final_norm);
    p.layers = x->d_layers;
    p.kc = static_cast<uint16_t*>(kv->k);
    p.vc = static_cast<uint16_t*>(kv->v);
    p.kv_bstride = kv->batch_stride;
    p.kv_lstride = kv->layer_stride;
    p.kv_hstride = kv->head_stride;
    p.kv_table = pages ? pages->block_table : nullptr;
    p.kv_max_blocks = pages ? pages->max_blocks : 0;
    p.kv_n_blocks = pages ? pages->n_blocks : 0;
    p.err = reinterpret_cast<int32_t*>(sb + sl.err);
    p.tokens_out = reinterpret_cast<int32_t*>(sb + sl.tokens);
    p.x_attn = reinterpret_cast<uint64_t*>(sb + sl.x_attn);
    p.x_out = reinterpret_cast<uint64_t*>(sb + sl.x_out);
    p.qkv = reinterpret_cast<uint64_t*>(sb + sl.qkv);
    p.part = reinterpret_cast<uint64_t*>(sb + sl.part);
    p.o = reinterpret_cast<uint64_t*>(sb + sl.o);
    p.h = reinterpret_cast<uint32_t*>(sb + sl.h);
    p.dpart = reinterpret_cast<uint32_t*>(sb + sl.dpart);
    p.lm_part = reinterpret_cast<int4*>(sb + sl.lm_part);
    p.rope = reinterpret_cast<const float2*>(sb + sl.rope);
    // The one reader without tags: the argmax over the LM-head partials, after an acquiring wait
    // on the counter the LM-head tiles publish after a release fence.
    p.acquire_ops = 1u << OP_ARGMAX;
    p.release_ops = 1u << OP_LMHEAD;
    p.timeout_ns = 2000000000ull;
    p.n_steps = 1;
    p.step_bar = x->d_step_bar;
    p.ctl = nullptr;
    x->last_err = p.err;
    p.smem_misc_off = n_pages * g.page_bytes;
    p.qrot_floats = qrf;
    p.xbuf_floats = xbuf;
    p.comb_stride = comb_stride;

    // tags start at 0 (never a step's tag): words left in the scratch by an earlier binding must
    // not pass for this context's first steps
    if ((e = cudaMemsetAsync(counters, 0, s->totals.size() * 4, x->stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(x->d_step_bar, 0, 4, x->stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(sb + sl.err, 0, 256, x->stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(sb + sl.x_attn, 0, sl.lm_part - sl.x_attn, x->stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(sb + sl.lm_part, 0xFF, sl.rope - sl.lm_part, x->stream)) != cudaSuccess)
        return bail(cuda_fail(e, "cudaMemsetAsync"));
    if ((e = launch_rope_table(reinterpret_cast<float2*>(sb + sl.rope), c.max_seq, d, c.rope_theta, x->stream)) !=
        cudaSuccess)
        return bail(cuda_fail(e, "rope table kernel"));
    if ((e = cudaStreamSynchronize(x->stream)) != cudaSuccess) return bail(cuda_fail(e, "bind synchronize"));
    *out = x;
    return MK_OK;
}

extern "C" mk_status mk_rebind_schedule(mk_ctx* c, const mk_schedule* s) {
    if (!c || !s) return fail(MK_ERR_ARG, "null argument");
    if (c->run_active) return fail(MK_ERR_ARG, "a persistent launch is in flight (mk_decode_persistent_wait first)");
    if (c->poisoned) return fail(MK_ERR_POISONED, "context poisoned by an earlier device error");
    // the same model, SM count and shapes: only the tiles' placement and the KV windows may differ
    const Geometry& a = c->geo;
    const Geometry& b = s->geo;
    if (std::memcmp(&s->cfg, &c->cfg, sizeof(mk_model_cfg)) != 0 || s->S != c->S || b.page_bytes != a.page_bytes ||
        b.attn_chunk != a.attn_chunk || b.n_chunk != a.n_chunk || b.r_qkv != a.r_qkv || b.r_o != a.r_o ||
        b.r_up != a.r_up || b.r_dn != a.r_dn || b.r_lm != a.r_lm || b.n_counters != a.n_counters ||
        s->totals != c->totals)
        return fail(MK_ERR_ARG, "the schedule differs from the bound one in more than placement and KV windows");
    std::vector<int32_t> dq;
    const mk_status rs = resolve_queues(s, &c->w, c->base.mv, c->base.mmv_kp, dq);
    if (rs != MK_OK) return rs;
    CK(cudaStreamSynchronize(c->stream));   // no launch reads the queues any more
    if (dq.size() > c->queue_words) {
        int32_t* nq = nullptr;
        CK(cudaMalloc(&nq, dq.size() * sizeof(int32_t)));
        cudaFree(c->d_queues);
        c->d_queues = nq;
        c->queue_words = dq.size();
    }
    CK(cudaMemcpy(c->d_queues, dq.data(), dq.size() * sizeof(int32_t), cudaMemcpyHostToDevice));
    c->base.queues = c->d_queues;
    c->base.Q = s->Q;
    c->geo = b;
    return MK_OK;
}

extern "C" mk_status mk_set_timeout(mk_ctx* c, uint64_t ns) {
    if (!c || ns == 0) return fail(MK_ERR_ARG, "bad argument");
    c->base.timeout_ns = ns;
    return MK_OK;
}

extern "C" mk_status mk_set_sync(mk_ctx* c, int32_t mode) {
    if (!c) return fail(MK_ERR_ARG, "null context");
    if (mode != MK_SYNC_TAGS && mode != MK_SYNC_COUNTERS) return fail(MK_ERR_ARG, "unknown sync mode %d", mode);
    c->base.sync_counters = mode == MK_SYNC_COUNTERS ? 1 : 0;
    return MK_OK;
}

extern "C" mk_status mk_set_trace(mk_ctx* c, uint64_t* buf) {
    if (!c) return fail(MK_ERR_ARG, "null context");
    if (reinterpret_cast<uintptr_t>(buf) & 7u) return fail(MK_ERR_ARG, "trace buffer not 8-byte aligned");
    c->base.trace = buf;
    return MK_OK;
}

// Clears the activation words, attention partials and LM-head partials of a scratch (tag 0 is
// never a step's tag; LM-head partial epochs 0xFFFFFFFF are never a step's epoch).
static cudaError_t clear_scratch(const Params& p, cudaStream_t st) {
    const size_t act = size_t(reinterpret_cast<const uint8_t*>(p.lm_part) - reinterpret_cast<const uint8_t*>(p.x_attn));
    const size_t lm = size_t(reinterpret_cast<const uint8_t*>(p.rope) - reinterpret_cast<const uint8_t*>(p.lm_part));
    cudaError_t e = cudaMemsetAsync(p.x_attn, 0, act, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(p.lm_part, 0xFF, lm, st);
    return e;
}

// Launches the resident grid with fully prepared parameters (scratch pointers, tokens,
// positions) at the context's epoch, then advances the epoch.
static mk_status launch_params(mk_ctx* c, Params& p) {
    p.epoch = c->epoch;
    p.tag = c->epoch + 1u;
    void* args[] = {&p};
    cudaError_t e = cudaLaunchCooperativeKernel(c->fn, dim3(c->grid), dim3(kThreads), args, size_t(c->smem), c->stream);
    if (e == cudaErrorCooperativeLaunchTooLarge)
        return fail(MK_ERR_RESOURCES, "cooperative launch of %d CTAs does not fit the device", c->grid);
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchCooperativeKernel");
    c->last_err = p.err;
    c->epoch += 1;
    return MK_OK;
}

// One step on the bound stream.  Its tokens come from the host (tokens) or, when tok_dev is set,
// from device memory (a chained step: the previous step's greedy tokens); pos[b] + dpos is its
// position.  The caller has checked the arguments.
static mk_status launch(mk_ctx* c, const int32_t* tokens, const int32_t* pos, int32_t dpos, float* logits,
                        int32_t* next_tokens_dev, const int32_t* tok_dev) {
    Params p = c->base;
    if (c->bound_stale) {   // steps ran on the static scratch since this scratch was last used
        const cudaError_t e = clear_scratch(p, c->stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(bound scratch)");
        c->bound_stale = false;
    }
    for (int b = 0; b < c->cfg.batch; ++b) {
        p.tok[b] = tok_dev ? 0 : tokens[b];
        p.pos[b] = pos[b] + dpos;
    }
    p.tok_dev = tok_dev;
    p.logits = logits;
    p.next_dev = next_tokens_dev;
    return launch_params(c, p);
}

static mk_status check_step_args(mk_ctx* c, const int32_t* tokens, const int32_t* pos, int32_t n_steps,
                                 const float* logits) {
    if (!c || !tokens || !pos || !logits) return fail(MK_ERR_ARG, "null argument");
    if (c->run_active) return fail(MK_ERR_ARG, "a persistent launch is in flight (mk_decode_persistent_wait first)");
    if (c->poisoned) return fail(MK_ERR_POISONED, "context poisoned by an earlier device error");
    if (reinterpret_cast<uintptr_t>(logits) & 3u) return fail(MK_ERR_ARG, "logits not 4-byte aligned");
    for (int b = 0; b < c->cfg.batch; ++b) {
        if (tokens[b] < 0 || tokens[b] >= c->cfg.vocab) return fail(MK_ERR_ARG, "token %d out of range", tokens[b]);
        if (pos[b] < 0 || int64_t(pos[b]) + n_steps > c->cfg.max_seq)
            return fail(MK_ERR_ARG, "positions %d..%d outside the KV capacity [0, %d)", pos[b], pos[b] + n_steps - 1,
                        c->cfg.max_seq);
        if (int64_t(pos[b]) + n_steps > c->geo.kv_limit[b])
            return fail(MK_ERR_ARG, "sequence %d: positions up to %d outside the schedule's window [0, %d) (re-plan: "
                        "mk_rebind_schedule)", b, pos[b] + n_steps - 1, c->geo.kv_limit[b]);
    }
    return MK_OK;
}

extern "C" mk_status mk_launch_step(mk_ctx* c, const int32_t* tokens, const int32_t* pos, float* logits,
                                    int32_t* next_tokens_dev) {
    const mk_status st = check_step_args(c, tokens, pos, 1, logits);
    if (st != MK_OK) return st;
    return launch(c, tokens, pos, 0, logits, next_tokens_dev, nullptr);
}

// Reads back the error word (and output tokens) of the context's last step -- from the scratch
// that step used -- and poisons the context on a device error.
static mk_status read_status(mk_ctx* c, int32_t* info) {
    cudaError_t e = cudaMemcpyAsync(c->h_result, c->last_err, 96, cudaMemcpyDeviceToHost, c->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) {
        c->poisoned = true;
        return cuda_fail(e, "step readback");
    }
    if (info)
        for (int i = 0; i < 8; ++i) info[i] = c->h_result[i];
    const int code = c->h_result[0];
    if (code != 0) {
        c->poisoned = true;
        return fail(mk_status(code), "device error %d (CTA %d, queue slot %d, counter %d, seen %d, wanted %d, role %d)",
                    code, c->h_result[1], c->h_result[2], c->h_result[3], c->h_result[4], c->h_result[5],
                    c->h_result[6]);
    }
    return MK_OK;
}

extern "C" mk_status mk_decode_step(mk_ctx* c, const int32_t* tokens, const int32_t* pos, float* logits,
                                    int32_t* next_tokens) {
    if (!next_tokens) return fail(MK_ERR_ARG, "null next_tokens");
    mk_status st = mk_launch_step(c, tokens, pos, logits, nullptr);
    if (st != MK_OK) return st;
    st = read_status(c, nullptr);
    if (st != MK_OK) return st;
    for (int b = 0; b < c->cfg.batch; ++b) next_tokens[b] = c->h_result[16 + b];
    return MK_OK;
}

extern "C" mk_status mk_decode_steps(mk_ctx* c, const int32_t* tokens, const int32_t* pos, int32_t n_steps,
                                     float* logits, int32_t* tokens_dev, int32_t* tokens_out) {
    if (n_steps < 1) return fail(MK_ERR_ARG, "n_steps %d < 1", n_steps);
    if (!tokens_dev || !tokens_out) return fail(MK_ERR_ARG, "null argument");
    if (reinterpret_cast<uintptr_t>(tokens_dev) & 3u) return fail(MK_ERR_ARG, "tokens_dev not 4-byte aligned");
    mk_status st = check_step_args(c, tokens, pos, n_steps, logits);
    if (st != MK_OK) return st;
    const int B = c->cfg.batch;
    for (int i = 0; i < n_steps; ++i) {   // back to back on the stream: no host round trip in between
        st = launch(c, tokens, pos, i, logits, tokens_dev + size_t(i) * B, i ? tokens_dev + size_t(i - 1) * B : nullptr);
        if (st != MK_OK) {
            c->poisoned = true;   // steps already enqueued have advanced the counters
            return st;
        }
    }
    const cudaError_t e =
        cudaMemcpyAsync(tokens_out, tokens_dev, size_t(n_steps) * B * sizeof(int32_t), cudaMemcpyDeviceToHost, c->stream);
    if (e != cudaSuccess) {
        c->poisoned = true;
        return cuda_fail(e, "token readback");
    }
    return read_status(c, nullptr);
}

// ---- persistent multi-step decode: one launch, up to n_steps steps, a host stop request ----
extern "C" mk_status mk_decode_persistent_start(mk_ctx* c, const int32_t* tokens, const int32_t* pos,
                                                int32_t n_steps, float* logits, int32_t* tokens_dev) {
    if (!c) return fail(MK_ERR_ARG, "null context");
    if (n_steps < 1) return fail(MK_ERR_ARG, "n_steps %d < 1", n_steps);
    if (!tokens_dev || (reinterpret_cast<uintptr_t>(tokens_dev) & 3u))
        return fail(MK_ERR_ARG, "tokens_dev null or not 4-byte aligned");
    mk_status st = check_step_args(c, tokens, pos, n_steps, logits);
    if (st != MK_OK) return st;
    Params p = c->base;
    if (c->bound_stale) {
        const cudaError_t e = clear_scratch(p, c->stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(bound scratch)");
        c->bound_stale = false;
    }
    for (int b = 0; b < c->cfg.batch; ++b) {
        p.tok[b] = tokens[b];
        p.pos[b] = pos[b];
    }
    p.tok_dev = nullptr;
    p.logits = logits;
    p.next_dev = tokens_dev;
    p.n_steps = n_steps;
    p.ctl = c->d_ctl;
    p.trace = nullptr;   // the trace holds one step's stamps
    // the control words are written before the launch is enqueued: the device sees them
    c->h_ctl[0] = 0;
    c->h_ctl[1] = 0;
    std::atomic_thread_fence(std::memory_order_seq_cst);
    p.epoch = c->epoch;
    p.tag = c->epoch + 1u;
    void* args[] = {&p};
    const cudaError_t e =
        cudaLaunchCooperativeKernel(c->fn, dim3(c->grid), dim3(kThreads), args, size_t(c->smem), c->stream);
    if (e == cudaErrorCooperativeLaunchTooLarge)
        return fail(MK_ERR_RESOURCES, "cooperative launch of %d CTAs does not fit the device", c->grid);
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchCooperativeKernel");
    c->last_err = p.err;
    c->run_active = true;
    c->run_steps = n_steps;
    c->run_tokens = tokens_dev;
    return MK_OK;
}

extern "C" mk_status mk_decode_persistent_stop(mk_ctx* c) {
    if (!c) return fail(MK_ERR_ARG, "null context");
    if (!c->run_active) return fail(MK_ERR_ARG, "no persistent launch in flight");
    c->h_ctl[0] = 1;
    std::atomic_thread_fence(std::memory_order_seq_cst);
    return MK_OK;
}

extern "C" mk_status mk_decode_persistent_progress(mk_ctx* c, int32_t* steps_done) {
    if (!c || !steps_done) return fail(MK_ERR_ARG, "null argument");
    std::atomic_thread_fence(std::memory_order_seq_cst);
    *steps_done = c->h_ctl[1];
    return MK_OK;
}

extern "C" mk_status mk_decode_persistent_wait(mk_ctx* c, int32_t* steps_done, int32_t* tokens_out) {
    if (!c) return fail(MK_ERR_ARG, "null context");
    if (!c->run_active) return fail(MK_ERR_ARG, "no persistent launch in flight");
    c->run_active = false;
    cudaError_t e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) {
        c->poisoned = true;
        return cuda_fail(e, "persistent launch");
    }
    const int32_t ran = c->h_ctl[1];
    // the steps run advanced the counters, the step word and the tags by that many epochs
    c->epoch += uint32_t(ran > 0 ? ran : 0);
    const mk_status st = read_status(c, nullptr);
    if (st != MK_OK) return st;
    if (ran < 1 || ran > c->run_steps) {
        c->poisoned = true;
        return fail(MK_ERR_CUDA, "persistent launch reported %d steps of %d", ran, c->run_steps);
    }
    if (steps_done) *steps_done = ran;
    if (tokens_out) {
        e = cudaMemcpy(tokens_out, c->run_tokens, size_t(ran) * c->cfg.batch * sizeof(int32_t), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(e, "token readback");
    }
    return MK_OK;
}

extern "C" mk_status mk_ctx_status(mk_ctx* c, int32_t* info) {
    if (!c) return fail(MK_ERR_ARG, "null context");
    if (c->run_active) return fail(MK_ERR_ARG, "a persistent launch is in flight (mk_decode_persistent_wait first)");
    if (c->poisoned && !info) return fail(MK_ERR_POISONED, "context poisoned by an earlier device error");
    return read_status(c, info);
}

extern "C" void mk_unbind(mk_ctx* c) {
    if (!c) return;
    if (c->run_active) c->h_ctl[0] = 1;   // a persistent launch ends at its next step boundary
    cudaStreamSynchronize(c->stream);
    free_ctx(c);
}

// ------------------------------------------------------------------------------------------------
// Decode step without caller scratch.  Some callers cannot allocate device memory themselves:
// code that runs under a framework whose caching allocator owns the GPU's memory (a direct
// cudaMalloc bypasses its accounting and can fail once the pool has reserved the device), or a
// latency-critical serving loop where a cudaMalloc / cudaFree may synchronise the whole device.
// For them this entry point keeps the step's scratch in a library-owned array of fixed size that
// every GPU loading the library holds until the process exits.  Calls share the array: two calls
// that overlap on the GPU (different streams, or different contexts at once) race on it.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;   // MK_STATIC_SCRATCH_BYTES
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];
static uint8_t* g_static_scratch_dev[64];                    // device address, per device
static std::mutex g_static_mutex;

extern "C" mk_status mk_decode_step_static(mk_ctx* c, const int32_t* tokens, const int32_t* pos, float* logits,
                                           int32_t* next_tokens) {
    if (!c || !tokens || !pos || !logits || !next_tokens) return fail(MK_ERR_ARG, "null argument");
    if (c->run_active) return fail(MK_ERR_ARG, "a persistent launch is in flight (mk_decode_persistent_wait first)");
    if (c->poisoned) return fail(MK_ERR_POISONED, "context poisoned by an earlier device error");
    int dev = -1;
    CK(cudaGetDevice(&dev));
    if (dev != c->device) return fail(MK_ERR_ARG, "the context is bound to device %d, device %d is current", c->device, dev);
    if (dev < 0 || dev >= 64) return fail(MK_ERR_ARG, "device ordinal %d out of range", dev);
    uint8_t* base;
    {   // set-up, once per device, with that device current: the array's device address
        std::lock_guard<std::mutex> lock(g_static_mutex);
        if (!g_static_scratch_dev[dev]) {
            void* ptr = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
            g_static_scratch_dev[dev] = static_cast<uint8_t*>(ptr);
        }
        base = g_static_scratch_dev[dev];
    }
    // the bound scratch layout, moved onto the static array (the error word leads the layout and
    // the RoPE table ends it)
    Params p = c->base;
    uint8_t* bound = reinterpret_cast<uint8_t*>(p.err);
    const size_t half = size_t(p.d / 2);
    const size_t need = size_t(reinterpret_cast<const uint8_t*>(p.rope) - bound) + size_t(p.max_seq) * half * 8;
    if (need > kStaticScratchBytes)
        return fail(MK_ERR_CAPACITY, "step needs %zu bytes of scratch, the static array holds %zu", need,
                    kStaticScratchBytes);
    for (int b = 0; b < c->cfg.batch; ++b) {
        if (tokens[b] < 0 || tokens[b] >= c->cfg.vocab) return fail(MK_ERR_ARG, "token %d out of range", tokens[b]);
        if (pos[b] < 0 || pos[b] >= c->cfg.max_seq)
            return fail(MK_ERR_ARG, "pos %d outside the KV capacity [0, %d)", pos[b], c->cfg.max_seq);
        if (pos[b] >= c->geo.kv_limit[b])
            return fail(MK_ERR_ARG, "sequence %d: pos %d outside the schedule's window [0, %d)", b, pos[b],
                        c->geo.kv_limit[b]);
        p.tok[b] = tokens[b];
        p.pos[b] = pos[b];
    }
    auto move = [&](auto* ptr) {
        using T = std::remove_pointer_t<decltype(ptr)>;
        return reinterpret_cast<T*>(base + (reinterpret_cast<const uint8_t*>(ptr) - bound));
    };
    p.err = move(p.err);
    p.tokens_out = move(p.tokens_out);
    p.x_attn = move(p.x_attn);
    p.x_out = move(p.x_out);
    p.qkv = move(p.qkv);
    p.part = move(p.part);
    p.o = move(p.o);
    p.h = move(p.h);
    p.dpart = move(p.dpart);
    p.lm_part = move(p.lm_part);
    p.rope = move(const_cast<float2*>(p.rope));
    // the array keeps the previous call's contents: reset what must start fresh (error word and
    // output tokens; the activation words -- another context may have left its own tags there --;
    // the LM-head partials' epochs) and rebuild the RoPE table for this model
    cudaError_t e;
    if ((e = cudaMemsetAsync(p.err, 0, 256, c->stream)) != cudaSuccess || (e = clear_scratch(p, c->stream)) != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync(static scratch)");
    if ((e = launch_rope_table(const_cast<float2*>(p.rope), c->cfg.max_seq, c->cfg.head_dim, c->cfg.rope_theta,
                               c->stream)) != cudaSuccess)
        return cuda_fail(e, "rope table kernel");
    p.logits = logits;
    p.next_dev = nullptr;
    p.tok_dev = nullptr;
    const mk_status st = launch_params(c, p);
    if (st != MK_OK) return st;
    // the bound scratch's activation tags fell behind the epoch: its next step clears them first
    c->bound_stale = true;
    const mk_status rs = read_status(c, nullptr);
    if (rs != MK_OK) return rs;
    for (int b = 0; b < c->cfg.batch; ++b) next_tokens[b] = c->h_result[16 + b];
    return MK_OK;
}
