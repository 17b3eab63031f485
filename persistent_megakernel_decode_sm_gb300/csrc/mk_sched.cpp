// Host scheduler: operator -> tiles -> dependency DAG (counters) -> waves -> memory/compute pool
// placement on S queues -> [S, Q, 32] int32 encoding.
//
// Follows the "Inference MegaKernel" page, section "Hand-written whole-model MegaKernel"
// (principle, scheduling and data flow): every operator of a fixed Llama configuration is cut
// into tiles, the tile dependency DAG is built, waves and a memory/compute pool are assigned,
// and each SM's plan is tensorised into an instruction queue held in HBM for the life of the
// kernel (the page's object table gives the queue only as an int32 tensor of shape [S, Q, 32]).
// The page fixes none of the concrete rules; this file states them:
//  * tiles per layer: QKV row tiles (<= head_dim rows: a tile touches one or two KV groups and
//    completes each), attention chunks (sequence, group, chunk of attn_chunk positions; only the
//    chunks inside the sequence's kv_limit window; at batch > 1 then one combine tile per
//    (sequence, group)), O row tiles, gate/up row-pair tiles, down row tiles; then
//    LM-head row tiles and one argmax per sequence;
//  * DAG: a consumer waits on one counter per producer set -- QKV(l) on down(l-1), attention
//    chunks of group g on the QKV tiles of group g, O on the combined attention of every group,
//    up/gate on O, down on up/gate, LM head on the last layer's down, argmax on the LM head.
//    At batch > 1 a down projection with rows longer than kMmvRange has a tile per (staging
//    range, row block); the tile of the last range (enumerated after every other range's tiles)
//    reads their tagged partial sums as they land, adds them in range order, writes the rows and
//    alone carries the completion.
//    At batch 1 the combine of a group's chunk partials is done by the chunk tile that holds the
//    step's position (known only at run time), which alone carries the completion O waits on; it
//    reads the other chunks' tagged partials as they land (a wait inside the wave, on tiles of
//    lower id, which every queue runs first).  At batch > 1 a COMB tile per (sequence, group),
//    enumerated after every chunk tile of the layer, does it and carries the completion, and the
//    chunk tiles complete nothing -- a chunk tile then never holds its SM for a combine while
//    chunks of later rounds queue behind it;
//  * waves = longest-path level (5 per layer, then LM head, then argmax); the waits of a tile
//    point only at lower waves (forward-progress contract);
//  * pools: memory = tiles that stream weights or KV, compute = argmax and combine; within a
//    wave memory tiles are placed first;
//  * rows per tile: about one tile per operator per SM (streamed through the page ring page by
//    page: at batch 1 whole rows per page, at batch > 1 a 16-row block over page_bytes / 32
//    positions per page, at most 64 rows per tile for rows longer than kMmvRange), or about
//    tile_bytes;
//  * placement: within a wave, tiles in (cost desc, id asc) order -- or a seeded splitmix64
//    Fisher-Yates order when shuffle_seed != 0 -- each to the queue with the smallest
//    accumulated cost (ties to the lowest SM) among the queues holding at most k / S of the
//    wave's tiles of that pool for the k-th tile (rounds of S tiles, one per SM), the
//    accumulated cost carried across waves;
//    cost = streamed bytes + a fixed per-tile overhead.  Each queue then runs its tiles of a wave
//    in id order (so a wait inside a wave is always on tiles that every queue runs earlier).
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <queue>
#include <string>
#include <utility>
#include <vector>

#include "mk_internal.h"

namespace mk {

static thread_local std::string g_last_error;

mk_status fail(mk_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

namespace {

struct Tile {
    int32_t op, layer, b, a0, a1, a2, wave;
    int32_t nwait, npub;
    int32_t wait[kMaxWait][2];
    int32_t pub[kMaxPub][2];
    int64_t stream_bytes;
    int32_t id;
    bool cond;   // ATTN: completions only from the tile that combines its group
    bool memory() const { return op != OP_ARGMAX && op != OP_COMB; }
    int64_t cost() const { return stream_bytes + kTileOverhead; }
};

int32_t cdiv(int64_t a, int64_t b) { return int32_t((a + b - 1) / b); }

int32_t fit(int32_t limit, int64_t tile_bytes, int64_t row_bytes) {
    int64_t r = tile_bytes / row_bytes;
    if (r > limit) r = limit;
    if (r < 1) r = 1;
    return int32_t(r);
}

struct SplitMix64 {
    uint64_t s;
    uint64_t next() {
        s += 0x9E3779B97F4A7C15ull;
        uint64_t z = s;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        return z ^ (z >> 31);
    }
};

mk_status check_cfg(const mk_model_cfg& c) {
    if (c.n_layers < 1 || c.hidden < 8 || c.n_q_heads < 1 || c.n_kv_heads < 1 || c.head_dim < 16 ||
        c.ffn < 8 || c.vocab < 1 || c.batch < 1 || c.max_seq < 1)
        return fail(MK_ERR_ARG, "model config: every size must be positive");
    if (c.batch > kMaxBatch) return fail(MK_ERR_ARG, "batch %d > %d", c.batch, kMaxBatch);
    if (c.n_q_heads % c.n_kv_heads) return fail(MK_ERR_ARG, "n_q_heads %% n_kv_heads != 0");
    if (c.n_q_heads / c.n_kv_heads > kMaxHpg)
        return fail(MK_ERR_ARG, "more than %d query heads per KV head", kMaxHpg);
    // (the attention reduces a K row over head_dim / 8 lanes with butterfly shuffles: a power of two)
    if ((c.head_dim != 32 && c.head_dim != 64 && c.head_dim != 128) || c.head_dim > kMaxHeadDim)
        return fail(MK_ERR_ARG, "head_dim must be 32, 64 or 128");
    const int64_t qd = int64_t(c.n_q_heads) * c.head_dim;
    if (c.hidden % 8 || c.ffn % 8 || qd % 8 || c.hidden > kMaxK || c.ffn > kMaxK || qd > kMaxK)
        return fail(MK_ERR_ARG, "hidden, ffn and n_q_heads*head_dim must be multiples of 8 and <= %d",
                    kMaxK);
    if (!(c.rms_eps >= 0.0) || !(c.rope_theta > 0.0)) return fail(MK_ERR_ARG, "bad rms_eps / rope_theta");
    if (int64_t(c.vocab) * c.hidden > (int64_t(1) << 40)) return fail(MK_ERR_CAPACITY, "vocab too large");
    return MK_OK;
}

}  // namespace
}  // namespace mk

using namespace mk;

extern "C" mk_status mk_build_schedule(const mk_model_cfg* cfgp, int32_t S, const mk_sched_opts* opts,
                                       mk_schedule** out) {
    if (!cfgp || !out) return fail(MK_ERR_ARG, "null argument");
    *out = nullptr;
    const mk_model_cfg c = *cfgp;
    mk_status st = check_cfg(c);
    if (st != MK_OK) return st;
    if (S < 1 || S > 4096) return fail(MK_ERR_ARG, "sm_count %d out of [1, 4096]", S);
    mk_sched_opts o{};
    if (opts) o = *opts;
    Geometry g{};
    // default page: 32768 at batch 1; at batch > 1 one 16-row block over kMmvRange positions
    g.page_bytes = o.page_bytes ? o.page_bytes : (c.batch > 1 ? 32 * kMmvRange : 32768);
    g.tile_bytes = o.tile_bytes;   // 0: matvec tiles sized per SM (see the rows per tile below)
    // attention chunk: 128 positions, doubled (up to 512) while the chunks of all sequences and KV
    // heads would outnumber the 152 SMs of a GB300 (long contexts, batches): fewer, larger split-K
    // tiles.  A property of the model configuration alone, like every tile shape: the results do
    // not depend on the SM count the schedule is built for.
    g.attn_chunk = o.attn_chunk;
    if (g.attn_chunk == 0) {
        g.attn_chunk = 128;
        while (g.attn_chunk < 512 &&
               int64_t(c.batch) * c.n_kv_heads * cdiv(c.max_seq, g.attn_chunk) > kAttnChunkTiles)
            g.attn_chunk *= 2;
    }
    g.shuffle_seed = o.shuffle_seed;
    for (int b = 0; b < kMaxBatch; ++b) {
        if (o.kv_limit[b] < 0 || o.kv_limit[b] > c.max_seq) return fail(MK_ERR_ARG, "kv_limit[%d] out of [0, max_seq]", b);
        g.kv_limit[b] = o.kv_limit[b] ? o.kv_limit[b] : c.max_seq;
    }
    if (g.page_bytes < 1024 || g.page_bytes % 128 || g.page_bytes > (1 << 20))
        return fail(MK_ERR_ARG, "page_bytes must be a multiple of 128 in [1024, 1 MiB]");
    if (g.tile_bytes != 0 && g.tile_bytes < 16) return fail(MK_ERR_ARG, "tile_bytes too small");
    if (g.attn_chunk < 1 || g.attn_chunk > 1024) return fail(MK_ERR_ARG, "attn_chunk out of [1, 1024]");

    const int32_t L = c.n_layers, H = c.hidden, F = c.ffn, V = c.vocab, B = c.batch;
    const int32_t nq = c.n_q_heads, nkv = c.n_kv_heads, d = c.head_dim, hpg = nq / nkv;
    const int32_t qd = nq * d, kvd = nkv * d, nqkv = qd + 2 * kvd;

    // rows per tile.  tile_bytes 0: about one tile per operator per SM -- a tile streams through
    // the page ring page by page, so it need not fit the ring, and the per-tile costs (dispatch,
    // input vector, first touch of its pages, completion) are paid once per operator and SM.  At
    // batch 1 the rows are rounded up to whole consumer groups (two pages of whole rows; gate/up:
    // a gate page and its up page), at most 16 rows (8 pairs), so no tile ends in a partly filled
    // group (measured: 1B step 722 -> 709 us); at batch > 1 only the QKV rows are rounded up, to
    // a 16-row MMA block (measured: the others' rounding cost 10 us at batch 8).  QKV tiles keep
    // <= head_dim rows (a tile then touches at most two KV groups).  At batch > 1 the MLP down
    // projection, when its rows are longer than kMmvRange, is cut into one tile per (staging
    // range, row block): each tile polls its inputs once instead of once per range (measured:
    // every poll of a 64 KB input range is a loaded-memory round trip of about 4 us), the tile of
    // the last range adds the partial sums of the others; any other operator with such rows keeps
    // the sums of all its rows over the ranges, so its tiles take at most 64 rows.  An explicit
    // tile_bytes: tiles of about tile_bytes.
    if (g.tile_bytes == 0) {
        auto grp = [&](int64_t K, bool pair) -> int32_t {   // rows (pairs) a tile is rounded up to
            if (B > 1) return 1;
            const int64_t rpp = std::max<int64_t>(1, g.page_bytes / (2 * K));
            return int32_t(pair ? std::min<int64_t>(rpp, 8) : std::min<int64_t>(2 * rpp, 16));
        };
        auto up_to = [](int32_t r, int32_t m) { return (r + m - 1) / m * m; };
        g.r_qkv = std::min(d, up_to(cdiv(nqkv, S), B > 1 ? 16 : grp(H, false)));
        g.r_o = up_to(cdiv(H, S), grp(qd, false));
        if (B > 1 && qd > kMmvRange) g.r_o = std::min(64, g.r_o);   // (sums over ranges: <= 4 row blocks)
        g.r_up = up_to(cdiv(F, S), grp(H, true));
        // (batch > 1, rows longer than kMmvRange: one tile per staging range of a row block, so
        // about one tile per SM takes H * ranges / S rows, in whole 16-row blocks, at most 64)
        const int32_t nrg_dn = mmv_down_ranges(B, F);
        g.r_dn = nrg_dn > 1 ? std::min(64, up_to(cdiv(H * nrg_dn, S), 16)) : up_to(cdiv(H, S), grp(F, false));
        g.r_lm = up_to(cdiv(V, S), grp(H, false));
    } else {
        const int64_t tb = g.tile_bytes ? g.tile_bytes : 131072;
        g.r_qkv = fit(8, tb, 2ll * H);
        while (d % g.r_qkv) --g.r_qkv;
        g.r_o = fit(8, tb, 2ll * qd);
        g.r_up = fit(16, tb, 4ll * H);
        g.r_dn = fit(8, tb, 2ll * F);
        g.r_lm = fit(32, tb, 2ll * H);
    }
    if (o.rows_qkv) g.r_qkv = o.rows_qkv;
    if (o.rows_o) g.r_o = o.rows_o;
    if (o.pairs_up) g.r_up = o.pairs_up;
    if (o.rows_down) g.r_dn = o.rows_down;
    if (o.rows_lm) g.r_lm = o.rows_lm;
    if (g.r_qkv < 1 || g.r_qkv > d) return fail(MK_ERR_ARG, "rows_qkv must be in [1, head_dim]");
    if (B > 1 && ((qd > kMmvRange && g.r_o > 64) || (F > kMmvRange && g.r_dn > 64)))
        return fail(MK_ERR_ARG, "at batch > 1 a tile of rows longer than %d takes at most 64 rows", kMmvRange);
    if (g.r_o < 1 || g.r_up < 1 || g.r_lm < 1 || g.r_dn < 1) return fail(MK_ERR_ARG, "rows per tile must be >= 1");
    if (B == 1 && g.page_bytes < 2 * std::max(H, std::max(qd, F)))   // batch 1: whole rows per page
        return fail(MK_ERR_ARG, "page_bytes %d holds no matvec row (%d bytes)", g.page_bytes, 2 * std::max(H, std::max(qd, F)));
    if (B > 1 && (g.page_bytes > 32 * kMmvRange || kMmvRange % (g.page_bytes / 32)))   // a 16-row block over
        return fail(MK_ERR_ARG, "at batch > 1 page_bytes / 32 must divide %d", kMmvRange);   // a part of a range
    g.n_qkv = cdiv(nqkv, g.r_qkv);
    g.n_o = cdiv(H, g.r_o);
    g.n_up = cdiv(F, g.r_up);
    g.n_dn = cdiv(H, g.r_dn);
    g.n_lm = cdiv(V, g.r_lm);
    g.n_chunk = cdiv(c.max_seq, g.attn_chunk);
    CounterMap cm(c);
    g.n_counters = cm.count();

    // ---- tiles in enumeration order (ids) ------------------------------------------------
    std::vector<Tile> tiles;
    tiles.reserve(size_t(L) * (g.n_qkv + B * nkv * (g.n_chunk + 1) + g.n_o + g.n_up + g.n_dn * mmv_down_ranges(B, F)) +
                  g.n_lm + B);
    auto add = [&](int32_t op, int32_t layer, int32_t b, int32_t a0, int32_t a1, int32_t a2, int32_t wave,
                   std::initializer_list<std::pair<int32_t, int32_t>> waits,
                   std::pair<int32_t, int32_t> pub, int64_t bytes) {
        Tile t{};
        t.op = op; t.layer = layer; t.b = b; t.a0 = a0; t.a1 = a1; t.a2 = a2; t.wave = wave;
        for (auto& w : waits) { t.wait[t.nwait][0] = w.first; t.wait[t.nwait][1] = w.second; ++t.nwait; }
        t.pub[0][0] = pub.first; t.pub[0][1] = pub.second; t.npub = 1;
        t.stream_bytes = bytes;
        t.cond = false;
        t.id = int32_t(tiles.size());
        tiles.push_back(t);
    };
    auto group_of_row = [&](int32_t r) {
        if (r < qd) return (r / d) / hpg;
        if (r < qd + kvd) return (r - qd) / d;
        return (r - qd - kvd) / d;
    };
    // QKV tiles of <= head_dim rows touch one or two KV groups (ranges are >= head_dim rows):
    // a tile completes every group it touches; attention of a group waits for all of them
    std::vector<int32_t> qkv_tiles_of_group(nkv, 0);
    for (int32_t t = 0; t < g.n_qkv; ++t) {
        const int32_t r0 = t * g.r_qkv, n = std::min(g.r_qkv, nqkv - r0);
        const int32_t g0 = group_of_row(r0), g1 = group_of_row(r0 + n - 1);
        ++qkv_tiles_of_group[g0];
        if (g1 != g0) ++qkv_tiles_of_group[g1];
    }
    for (int32_t l = 0; l < L; ++l) {
        for (int32_t t = 0; t < g.n_qkv; ++t) {
            int32_t r0 = t * g.r_qkv, n = std::min(g.r_qkv, nqkv - r0);
            const int32_t g0 = group_of_row(r0), g1 = group_of_row(r0 + n - 1);
            if (l == 0)
                add(OP_QKV, l, 0, r0, n, 0, 5 * l, {}, {cm.qkv(l, g0), 1}, int64_t(n) * H * 2);
            else
                add(OP_QKV, l, 0, r0, n, 0, 5 * l, {{cm.down(l - 1), g.n_dn}}, {cm.qkv(l, g0), 1},
                    int64_t(n) * H * 2);
            if (g1 != g0) {
                Tile& tq = tiles.back();
                tq.pub[1][0] = cm.qkv(l, g1);
                tq.pub[1][1] = 1;
                tq.npub = 2;
            }
        }
        for (int32_t b = 0; b < B; ++b)
            for (int32_t gr = 0; gr < nkv; ++gr)
                for (int32_t ch = 0; ch < g.n_chunk && int64_t(ch) * g.attn_chunk < g.kv_limit[b]; ++ch) {
                    // (its stream: the chunk's K and V rows inside the window -- the last chunk of a
                    // window is partly filled, so it costs less and is placed last in its wave)
                    const int64_t rows = std::min<int64_t>(g.attn_chunk, int64_t(g.kv_limit[b]) - int64_t(ch) * g.attn_chunk);
                    add(OP_ATTN, l, b, gr, ch, g.attn_chunk, 5 * l + 1, {{cm.qkv(l, gr), qkv_tiles_of_group[gr]}},
                        {cm.comb(l), 1}, int64_t(2) * rows * d * 2);
                    if (B == 1) tiles.back().cond = true;   // the chunk holding pos combines and completes
                    else tiles.back().npub = 0;               // combined by the group's COMB tile
                }
        if (B > 1)   // one combine tile per (sequence, KV group), after every chunk tile of the layer
            for (int32_t b = 0; b < B; ++b)
                for (int32_t gr = 0; gr < nkv; ++gr)
                    add(OP_COMB, l, b, gr, 0, g.attn_chunk, 5 * l + 1, {}, {cm.comb(l), 1}, 0);
        for (int32_t t = 0; t < g.n_o; ++t) {
            int32_t r0 = t * g.r_o, n = std::min(g.r_o, H - r0);
            add(OP_OPROJ, l, 0, r0, n, 0, 5 * l + 2, {{cm.comb(l), B * nkv}}, {cm.o(l), 1}, int64_t(n) * qd * 2);
        }
        for (int32_t t = 0; t < g.n_up; ++t) {
            int32_t r0 = t * g.r_up, n = std::min(g.r_up, F - r0);
            add(OP_UPGATE, l, 0, r0, n, 0, 5 * l + 3, {{cm.o(l), g.n_o}}, {cm.up(l), 1}, int64_t(2) * n * H * 2);
        }
        // at batch > 1 with rows longer than kMmvRange: a tile per (staging range a2, row block),
        // the ranges in order; the tile of the last range (highest ids) adds the others' partial
        // sums and alone completes the rows
        const int32_t nrg_dn = mmv_down_ranges(B, F);
        for (int32_t r = 0; r < nrg_dn; ++r)
            for (int32_t t = 0; t < g.n_dn; ++t) {
                int32_t r0 = t * g.r_dn, n = std::min(g.r_dn, H - r0);
                const int64_t kr = nrg_dn > 1 ? std::min<int64_t>(kMmvRange, F - int64_t(r) * kMmvRange) : F;
                add(OP_DOWN, l, 0, r0, n, r, 5 * l + 4, {{cm.up(l), g.n_up}}, {cm.down(l), 1}, int64_t(n) * kr * 2);
                if (r + 1 < nrg_dn) tiles.back().npub = 0;
            }
    }
    for (int32_t t = 0; t < g.n_lm; ++t) {
        int32_t r0 = t * g.r_lm, n = std::min(g.r_lm, V - r0);
        add(OP_LMHEAD, L, 0, r0, n, t, 5 * L, {{cm.down(L - 1), g.n_dn}}, {cm.lm(), 1}, int64_t(n) * H * 2);
    }
    for (int32_t b = 0; b < B; ++b)
        add(OP_ARGMAX, L, b, 0, g.n_lm, 0, 5 * L + 1, {{cm.lm(), g.n_lm}}, {cm.fin(), 1}, 0);

    // ---- placement ------------------------------------------------------------------------
    // each tile, in order, to the SM with the smallest accumulated cost (ties: lowest SM) among
    // those holding at most k / S of the wave's tiles of this pool for the k-th tile: rounds of S
    // tiles, one per SM, so tiles of neighbouring ids run at about the same time (an attention
    // group's combining tile then waits on chunks of its own round or an earlier one)
    std::vector<int64_t> acc(S, 0);
    std::vector<int32_t> in_wave(S, 0);
    std::vector<std::vector<int32_t>> per_sm(S);
    SplitMix64 rng{g.shuffle_seed};
    size_t i = 0;
    while (i < tiles.size()) {
        size_t j = i;
        while (j < tiles.size() && tiles[j].wave == tiles[i].wave) ++j;  // tiles of one wave are contiguous
        std::vector<int32_t> mem, cmp;
        for (size_t k = i; k < j; ++k) (tiles[k].memory() ? mem : cmp).push_back(tiles[k].id);
        auto order = [&](std::vector<int32_t>& v) {
            if (g.shuffle_seed == 0) {
                std::stable_sort(v.begin(), v.end(), [&](int32_t a, int32_t b) {
                    if (tiles[a].cost() != tiles[b].cost()) return tiles[a].cost() > tiles[b].cost();
                    return a < b;
                });
            } else {
                for (size_t k = v.size(); k-- > 1;) {
                    size_t r = size_t(rng.next() % uint64_t(k + 1));
                    std::swap(v[k], v[r]);
                }
            }
        };
        order(mem);
        order(cmp);
        std::vector<size_t> start(S);
        for (int32_t s = 0; s < S; ++s) start[s] = per_sm[s].size();
        for (auto* v : {&mem, &cmp}) {
            std::fill(in_wave.begin(), in_wave.end(), 0);
            for (size_t k = 0; k < v->size(); ++k) {
                const int32_t id = (*v)[k];
                const int32_t cap = int32_t(k / size_t(S)) + 1;   // round k / S: one tile per SM
                int32_t best = -1;
                for (int32_t s = 0; s < S; ++s)
                    if (in_wave[s] < cap && (best < 0 || acc[s] < acc[best])) best = s;
                per_sm[best].push_back(id);
                acc[best] += tiles[id].cost();
                ++in_wave[best];
            }
        }
        for (int32_t s = 0; s < S; ++s) std::sort(per_sm[s].begin() + ptrdiff_t(start[s]), per_sm[s].end());
        i = j;
    }

    // ---- encoding -------------------------------------------------------------------------
    auto* sch = new mk_schedule();
    sch->cfg = c;
    sch->geo = g;
    sch->S = S;
    size_t qmax = 0;
    for (auto& v : per_sm) qmax = std::max(qmax, v.size());
    sch->Q = int32_t(qmax + 1);
    sch->queues.assign(size_t(S) * sch->Q * kWords, 0);
    sch->totals.assign(g.n_counters, 0u);
    sch->max_pages = 0;
    for (int32_t s = 0; s < S; ++s)
        for (size_t k = 0; k < per_sm[s].size(); ++k) {
            const Tile& t = tiles[per_sm[s][k]];
            int32_t* w = &sch->queues[(size_t(s) * sch->Q + k) * kWords];
            w[W_OP] = t.op; w[W_LAYER] = t.layer; w[W_B] = t.b;
            w[W_A0] = t.a0; w[W_A1] = t.a1; w[W_A2] = t.a2;
            w[W_NWAIT] = t.nwait;
            for (int q = 0; q < t.nwait; ++q) { w[W_WAIT + 2 * q] = t.wait[q][0]; w[W_WAIT + 2 * q + 1] = t.wait[q][1]; }
            w[W_NPUB] = t.npub;
            for (int q = 0; q < t.npub; ++q) { w[W_PUB + 2 * q] = t.pub[q][0]; w[W_PUB + 2 * q + 1] = t.pub[q][1]; }
            // matvec tiles stream whole rows per page (gate/up: gate and up row groups in alternate
            // pages); an attention tile streams its K rows, then its V rows
            int64_t pages = (t.stream_bytes + g.page_bytes - 1) / g.page_bytes;
            if (t.op == OP_QKV || t.op == OP_OPROJ || t.op == OP_UPGATE || t.op == OP_DOWN || t.op == OP_LMHEAD) {
                const int64_t K = t.op == OP_OPROJ ? qd : (t.op == OP_DOWN ? F : H);
                if (B > 1) {   // 16-row blocks (gate/up: 8 pairs) over page_bytes / 32 positions
                    const int64_t kp = g.page_bytes / 32, rb = t.op == OP_UPGATE ? 8 : 16;
                    const int64_t Kt = (t.op == OP_DOWN && mmv_down_ranges(B, F) > 1)
                                           ? std::min<int64_t>(kMmvRange, K - int64_t(t.a2) * kMmvRange) : K;
                    pages = ((t.a1 + rb - 1) / rb) * ((Kt + kp - 1) / kp);
                } else {
                    const int64_t rpp = g.page_bytes / (2 * K);
                    pages = ((t.a1 + rpp - 1) / rpp) * (t.op == OP_UPGATE ? 2 : 1);
                }
            }
            if (pages > (1 << 20)) { delete sch; return fail(MK_ERR_CAPACITY, "tile too large"); }
            w[W_NPAGES] = int32_t(pages);
            w[W_TILE] = t.id;
            w[W_WAVE] = t.wave;
            if (t.cond) w[W_COND] = 1;
            sch->max_pages = std::max(sch->max_pages, int32_t(pages));
        }
    for (const Tile& t : tiles) {
        if (t.cond && t.a1 != 0) continue;   // one completion per group (from its combining tile)
        for (int q = 0; q < t.npub; ++q) sch->totals[t.pub[q][0]] += uint32_t(t.pub[q][1]);
    }

    // ---- structural validation (waits point at lower waves; queues in wave order) ------------
    std::vector<int32_t> prod_wave(g.n_counters, -1);
    for (const Tile& t : tiles)
        for (int q = 0; q < t.npub; ++q) prod_wave[t.pub[q][0]] = t.wave;
    for (const Tile& t : tiles)
        for (int q = 0; q < t.nwait; ++q) {
            int32_t cid = t.wait[q][0];
            if (prod_wave[cid] < 0 || prod_wave[cid] >= t.wave || uint32_t(t.wait[q][1]) != sch->totals[cid]) {
                delete sch;
                return fail(MK_ERR_CAPACITY, "internal: tile %d waits on a counter outside lower waves", t.id);
            }
        }
    *out = sch;
    return MK_OK;
}

extern "C" mk_status mk_schedule_queues(const mk_schedule* s, const int32_t** q, int32_t* S, int32_t* Q) {
    if (!s || !q || !S || !Q) return fail(MK_ERR_ARG, "null argument");
    *q = s->queues.data();
    *S = s->S;
    *Q = s->Q;
    return MK_OK;
}

extern "C" mk_status mk_schedule_attn_chunk(const mk_schedule* s, int32_t* out) {
    if (!s || !out) return fail(MK_ERR_ARG, "null argument");
    *out = s->geo.attn_chunk;
    return MK_OK;
}

extern "C" mk_status mk_schedule_counters(const mk_schedule* s, const uint32_t** t, int32_t* n) {
    if (!s || !t || !n) return fail(MK_ERR_ARG, "null argument");
    *t = s->totals.data();
    *n = int32_t(s->totals.size());
    return MK_OK;
}

extern "C" mk_status mk_schedule_patch(mk_schedule* s, int32_t sm, int32_t slot, int32_t word, int32_t value) {
    if (!s) return fail(MK_ERR_ARG, "null schedule");
    if (sm < 0 || sm >= s->S || slot < 0 || slot >= s->Q || word < 0 || word >= kWords)
        return fail(MK_ERR_ARG, "patch index out of range");
    s->queues[(size_t(sm) * s->Q + slot) * kWords + word] = value;
    return MK_OK;
}

extern "C" size_t mk_scratch_bytes(const mk_schedule* s) {
    if (!s) return 0;
    return scratch_layout(s->cfg, s->geo, s->S).total;
}

extern "C" void mk_schedule_free(mk_schedule* s) { delete s; }

extern "C" const char* mk_last_error(void) { return mk::g_last_error.c_str(); }
