/*
 * ORACLE -- test infrastructure only.  Nothing in the library's product path includes,
 * links or calls this code; only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no header, helper or constant with the CUDA path.
 *
 * A plain, slow, obviously correct CPU decode step of a Llama-style decoder, written from
 * the "Inference MegaKernel" page (section "Hand-written whole-model MegaKernel": the
 * opcode list RMS_NORM, QKV_MATVEC, ATTENTION, MLP_UP_GATE, MLP_DOWN, LM_HEAD, and the
 * statement that the megakernel keeps every operator's logical semantics and changes only
 * the physical execution boundary).  The page never writes the per-operator mathematics
 * out, so every operator below is the textbook definition of the Llama decoder layer the
 * page names (Llama-3.2-1B, batch 1):
 *
 *   x  = E[token]
 *   per layer:  xn = rmsnorm(x, g_attn);  q,k,v = Wq xn, Wk xn, Wv xn;  rope(q), rope(k) at pos;
 *               k,v -> bf16 cache[pos];   o_h = softmax(q_h K^T / sqrt(d)) V  over 0..pos (GQA);
 *               x += Wo o;  xn = rmsnorm(x, g_mlp);  x += Wd (silu(Wg xn) * (Wu xn))
 *   logits = W_lm rmsnorm(x, g_final);  next = argmax (lowest index on ties)
 *
 * Readings where the page is silent (each listed in the design notes): no O-projection is
 * named, so one is added with the residual; RoPE pairs (i, i + d/2) ("rotate half") with
 * theta_i = theta^(-2i/d) and no frequency scaling; the current token's k and v are rounded
 * to bf16 and read back from the cache like every other position; eps inside the sqrt.
 *
 * This file is included twice by oracle.c: once with REAL = float (the fp32 oracle, sums in
 * sequential order) and once with REAL = double (the fp64 oracle, used to bound the fp32
 * oracle's own rounding error).  Weights and caches are bf16 bit patterns (uint16_t) widened
 * exactly to REAL.  Angles for RoPE are computed in double in both builds.
 */

/* the including file defines REAL and PFX(name) */

/* bf16 bits -> REAL, exact (bf16 is the top half of an IEEE binary32). */
static REAL PFX(widen)(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (REAL)f;
}

/* REAL -> bf16 bits, round to nearest, ties to even, from the binary32 value.  (The fp64 build
 * first rounds to binary32; the double rounding this allows is irrelevant at its use.) */
uint16_t PFX(bf16_round)(REAL v) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* RMSNorm: r = sqrt(mean(x^2) + eps); out_j = (x_j / r) * g_j. */
void PFX(rmsnorm)(const REAL* x, const uint16_t* g, int n, double eps, REAL* out) {
    REAL ss = 0;
    for (int j = 0; j < n; ++j) ss += x[j] * x[j];
    REAL r = (REAL)sqrt((double)(ss / (REAL)n + (REAL)eps));
    for (int j = 0; j < n; ++j) out[j] = (x[j] / r) * PFX(widen)(g[j]);
}

/* y_i = sum_j W[i, j] x_j, W row-major bf16 [rows, cols]; each row summed in order j = 0.. */
void PFX(matvec)(const uint16_t* W, int rows, int cols, const REAL* x, REAL* y) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < rows; ++i) {
        const uint16_t* w = W + (size_t)i * cols;
        REAL acc = 0;
        for (int j = 0; j < cols; ++j) acc += PFX(widen)(w[j]) * x[j];
        y[i] = acc;
    }
}

/* RoPE on n_heads consecutive head vectors of length d, rotate-half pairing (i, i + d/2):
 *   x'_i = x_i cos(a) - x_{i+d/2} sin(a),  x'_{i+d/2} = x_i sin(a) + x_{i+d/2} cos(a),
 *   a = pos * theta^(-2i/d), computed in double and then rounded to REAL. */
void PFX(rope)(REAL* v, int n_heads, int d, int pos, double theta) {
    int half = d / 2;
    for (int i = 0; i < half; ++i) {
        double inv = pow(theta, -2.0 * (double)i / (double)d);
        double a = (double)pos * inv;
        REAL c = (REAL)cos(a), s = (REAL)sin(a);
        for (int h = 0; h < n_heads; ++h) {
            REAL* x = v + (size_t)h * d;
            REAL x0 = x[i], x1 = x[i + half];
            x[i] = x0 * c - x1 * s;
            x[i + half] = x0 * s + x1 * c;
        }
    }
}

/* Decode attention for one sequence and one layer.
 * q: [nq, d] (already rotated).  kc, vc: bf16 [nkv, max_seq, d] for this (sequence, layer).
 * Query head h reads KV head h / (nq / nkv).  Positions 0..pos inclusive.
 *   s_t = (q_h . k_t) / sqrt(d);  m = max_t s_t;  w_t = exp(s_t - m);  l = sum_t w_t;
 *   o_h = sum_t (w_t / l) v_t.
 * probs (optional, [nq, pos + 1]) receives w_t / l. */
void PFX(attention)(const REAL* q, const uint16_t* kc, const uint16_t* vc, int nq, int nkv,
                    int d, int max_seq, int pos, REAL* out, REAL* probs) {
    int group = nq / nkv;
    int T = pos + 1;
#pragma omp parallel for schedule(static)
    for (int h = 0; h < nq; ++h) {
        int g = h / group;
        const uint16_t* K = kc + (size_t)g * max_seq * d;
        const uint16_t* V = vc + (size_t)g * max_seq * d;
        const REAL* qh = q + (size_t)h * d;
        REAL* s = (REAL*)malloc(sizeof(REAL) * (size_t)T);
        REAL scale = (REAL)(1.0 / sqrt((double)d));
        REAL m = -INFINITY;
        for (int t = 0; t < T; ++t) {
            REAL acc = 0;
            for (int j = 0; j < d; ++j) acc += qh[j] * PFX(widen)(K[(size_t)t * d + j]);
            s[t] = acc * scale;
            if (s[t] > m) m = s[t];
        }
        REAL l = 0;
        for (int t = 0; t < T; ++t) {
            s[t] = (REAL)exp((double)(s[t] - m));
            l += s[t];
        }
        REAL* o = out + (size_t)h * d;
        for (int j = 0; j < d; ++j) o[j] = 0;
        for (int t = 0; t < T; ++t) {
            REAL p = s[t] / l;
            if (probs) probs[(size_t)h * T + t] = p;
            for (int j = 0; j < d; ++j) o[j] += p * PFX(widen)(V[(size_t)t * d + j]);
        }
        free(s);
    }
}

REAL PFX(silu)(REAL z) { return z / ((REAL)1 + (REAL)exp(-(double)z)); }

/* h_i = silu(a_i) * u_i */
void PFX(swiglu)(const REAL* a, const REAL* u, int n, REAL* out) {
    for (int i = 0; i < n; ++i) out[i] = PFX(silu)(a[i]) * u[i];
}

/* index of the largest value; ties go to the lowest index */
int PFX(argmax)(const REAL* v, int n) {
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

/* One decode step for every sequence b of the batch: token tokens[b] at position pos[b].
 * Writes K/V of position pos[b] into the caches (bf16 [B, L, nkv, max_seq, d]), the logits
 * [B, vocab] and the greedy next token of each sequence.  Returns 0, or -1 on a bad argument. */
int PFX(decode_step)(const or_cfg* c, const or_weights* w, uint16_t* kcache, uint16_t* vcache,
                     const int* tokens, const int* pos, REAL* logits, int* next_tokens) {
    int L = c->n_layers, H = c->hidden, nq = c->n_q_heads, nkv = c->n_kv_heads, d = c->head_dim;
    int F = c->ffn, Vv = c->vocab, S = c->max_seq;
    int qd = nq * d, kvd = nkv * d;
    if (nq % nkv || d % 2) return -1;
    REAL* x = (REAL*)malloc(sizeof(REAL) * H);
    REAL* xn = (REAL*)malloc(sizeof(REAL) * H);
    REAL* qkv = (REAL*)malloc(sizeof(REAL) * (qd + 2 * kvd));
    REAL* att = (REAL*)malloc(sizeof(REAL) * qd);
    REAL* tmp = (REAL*)malloc(sizeof(REAL) * (H > 2 * F ? H : 2 * F));
    REAL* hmid = (REAL*)malloc(sizeof(REAL) * F);
    int rc = 0;
    for (int b = 0; b < c->batch; ++b) {
        int tok = tokens[b], p = pos[b];
        if (tok < 0 || tok >= Vv || p < 0 || p >= S) { rc = -1; break; }
        for (int j = 0; j < H; ++j) x[j] = PFX(widen)(w->embed[(size_t)tok * H + j]);
        for (int l = 0; l < L; ++l) {
            size_t cache_off = (((size_t)b * L + l) * nkv) * (size_t)S * d;
            uint16_t* kc = kcache + cache_off;
            uint16_t* vc = vcache + cache_off;
            /* attention block */
            PFX(rmsnorm)(x, w->attn_norm[l], H, c->rms_eps, xn);
            PFX(matvec)(w->wqkv[l], qd + 2 * kvd, H, xn, qkv);
            REAL* q = qkv;
            REAL* k = qkv + qd;
            REAL* v = qkv + qd + kvd;
            PFX(rope)(q, nq, d, p, c->rope_theta);
            PFX(rope)(k, nkv, d, p, c->rope_theta);
            for (int g = 0; g < nkv; ++g)
                for (int j = 0; j < d; ++j) {
                    kc[((size_t)g * S + p) * d + j] = PFX(bf16_round)(k[g * d + j]);
                    vc[((size_t)g * S + p) * d + j] = PFX(bf16_round)(v[g * d + j]);
                }
            PFX(attention)(q, kc, vc, nq, nkv, d, S, p, att, NULL);
            PFX(matvec)(w->wo[l], H, qd, att, tmp);
            for (int j = 0; j < H; ++j) x[j] += tmp[j];
            /* MLP block */
            PFX(rmsnorm)(x, w->mlp_norm[l], H, c->rms_eps, xn);
            PFX(matvec)(w->wgate_up[l], 2 * F, H, xn, tmp); /* gate rows, then up rows */
            PFX(swiglu)(tmp, tmp + F, F, hmid);
            PFX(matvec)(w->wdown[l], H, F, hmid, tmp);
            for (int j = 0; j < H; ++j) x[j] += tmp[j];
        }
        PFX(rmsnorm)(x, w->final_norm, H, c->rms_eps, xn);
        REAL* lg = logits + (size_t)b * Vv;
        PFX(matvec)(w->lm_head, Vv, H, xn, lg);
        next_tokens[b] = PFX(argmax)(lg, Vv);
    }
    free(x); free(xn); free(qkv); free(att); free(tmp); free(hmid);
    return rc;
}
