/*
 * ORACLE -- test infrastructure only (see oracle_impl.h).  Builds the fp32 oracle (or_f32_*)
 * and the fp64 oracle (or_f64_*) from one definition, plus a thread-count switch.
 * Compile: gcc -O2 -fopenmp -shared -fPIC oracle.c -o liboracle.so -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab, batch, max_seq;
    double rms_eps, rope_theta;
} or_cfg;

typedef struct {
    const uint16_t* embed;
    const uint16_t* lm_head;
    const uint16_t* final_norm;
    const uint16_t* const* attn_norm;
    const uint16_t* const* wqkv;
    const uint16_t* const* wo;
    const uint16_t* const* mlp_norm;
    const uint16_t* const* wgate_up;
    const uint16_t* const* wdown;
} or_weights;

#define REAL float
#define PFX(name) or_f32_##name
#include "oracle_impl.h"
#undef REAL
#undef PFX

#define REAL double
#define PFX(name) or_f64_##name
#include "oracle_impl.h"
#undef REAL
#undef PFX

/* Number of host threads the oracle's loops over output rows and heads use (each row's sum
 * keeps its sequential order, so results do not depend on it).  Returns the count in force. */
int or_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
