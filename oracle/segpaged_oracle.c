/*
 * Plain CPU oracle for head-aware (SegPaged) attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or table with the CUDA path.
 *
 * What it computes is the plain definition the RedKnot SegPagedAttention
 * runtime article states its fused kernel must equal (section 4,
 * "mask-free fused kernel": same result as dense attention under an explicit
 * head-wise mask): for every query head h of KV head h / (Hq / Hkv) (GQA
 * grouping, KV-cache tutorial section 5.3, written 0-indexed) and every query
 * at absolute position i,
 *
 *     O_i = sum_{j in V(i)} softmax_j(q_i . k_j / sqrt(d)) v_j
 *
 * where V(i) is the head's visibility set, materialised from its class
 * (runtime article section 2, "four head-class policies"):
 *     GLOBAL          V(i) = {0, ..., i}                        (full history)
 *     LOCAL(s, W)     V(i) = [0, min(s, i+1)) u [max(0, i-W+1), i]
 *                     (sink tokens plus the W most recent, query included)
 *     RETRIEVAL(I)    V(i) = I n [0, i]                 (selected tokens only)
 * The scale 1/sqrt(d) is the tutorial's FlashAttention section 10.2 default.
 * An empty V(i) gives O_i = 0 and LSE = -inf.
 *
 * Arithmetic: two passes over V(i) -- the maximum score, then the sum of
 * exp(score - max) and the weighted sum of v -- and one division at the end;
 * no blocking and no online rescaling.  The file is compiled twice, with
 * real_t = float (the plain fp32 oracle) and real_t = double (used to check
 * the fp32 one), selected by ORACLE_DOUBLE.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ORACLE_MUTATION (0 = none) plants one deliberate mistake; only the
 * mutation test builds such a variant, to show that the pins catch it. */
#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

#ifdef ORACLE_DOUBLE
typedef double real_t;
#define R_EXP exp
#define R_LOG log
#define R_SQRT sqrt
#define ORACLE_FN(name) name##_f64
#else
typedef float real_t;
#define R_EXP expf
#define R_LOG logf
#define R_SQRT sqrtf
#define ORACLE_FN(name) name##_f32
#endif

enum { OR_GLOBAL = 0, OR_LOCAL = 1, OR_RETRIEVAL = 2 };

#ifndef ORACLE_COMMON_DEFINED
#define ORACLE_COMMON_DEFINED
/*
 * V(i) for one head, written into out[] in ascending order; returns |V(i)|,
 * or -1 for an unknown class.  out[] must hold i+1 entries.
 */
static int64_t visible_set(int kind, int64_t sink, int64_t window,
                           const int32_t* idx, int64_t n_idx, int64_t i,
                           int64_t* out)
{
    int64_t n = 0;
    if (i < 0) return 0;
    if (kind == OR_GLOBAL) {
        for (int64_t j = 0; j <= i; ++j) out[n++] = j;
    } else if (kind == OR_LOCAL) {
        /* sink part: [0, min(s, i+1)) */
#if ORACLE_MUTATION == 6
        int64_t sink_end = sink + 1 < i + 1 ? sink + 1 : i + 1;   /* planted: sink one too long */
#else
        int64_t sink_end = sink < i + 1 ? sink : i + 1;
#endif
        for (int64_t j = 0; j < sink_end; ++j) out[n++] = j;
        /* window part: [max(0, i-W+1), i], minus what the sink already holds */
#if ORACLE_MUTATION == 1
        int64_t w0 = i - window;                       /* planted: window one too wide */
#else
        int64_t w0 = i - window + 1;
#endif
        if (w0 < 0) w0 = 0;
        if (w0 < sink_end) w0 = sink_end;
        for (int64_t j = w0; j <= i; ++j) out[n++] = j;
    } else if (kind == OR_RETRIEVAL) {
        for (int64_t k = 0; k < n_idx; ++k)
#if ORACLE_MUTATION == 2
            if (idx[k] < i) out[n++] = idx[k];         /* planted: query itself dropped */
#else
            if (idx[k] <= i) out[n++] = idx[k];
#endif
    } else {
        return -1;
    }
    return n;
}
#endif

/*
 * Attention for n_rows queries of one sequence.
 *   row_pos [n_rows]            absolute position i of each query
 *   kind/sink/window [Hkv]      head class of each KV head
 *   idx_off [Hkv+1], idx[]      RETRIEVAL lists (CSR by KV head), ascending
 *   Q [n_rows][Hq][d]           queries
 *   K, V [n_keys][Hkv][d]       keys/values at positions 0 .. n_keys-1
 *   O [n_rows][Hq][d], LSE [n_rows][Hq] (natural log; may be NULL)
 * Returns 0, or -1 if a visible position is >= n_keys or a class is unknown.
 */
int ORACLE_FN(oracle_attend)(int64_t n_rows, const int64_t* row_pos,
                             int hq, int hkv, int d,
                             const int32_t* kind, const int32_t* sink,
                             const int32_t* window, const int64_t* idx_off,
                             const int32_t* idx,
                             const real_t* Q, int64_t n_keys,
                             const real_t* K, const real_t* V,
                             real_t* O, real_t* LSE, int n_threads)
{
    const int group = hq / hkv;
#if ORACLE_MUTATION == 3
    const real_t scale = (real_t)1;                    /* planted: scale dropped */
#else
    const real_t scale = (real_t)1 / R_SQRT((real_t)d);
#endif
    int failed = 0;
    int64_t max_pos = 0;
    for (int64_t r = 0; r < n_rows; ++r)
        if (row_pos[r] > max_pos) max_pos = row_pos[r];
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel reduction(| : failed)
    {
        int64_t* vis = (int64_t*)malloc(sizeof(int64_t) * (size_t)(max_pos + 1));
        real_t* score = (real_t*)malloc(sizeof(real_t) * (size_t)(max_pos + 1));
        real_t* acc = (real_t*)malloc(sizeof(real_t) * (size_t)d);
#pragma omp for collapse(2) schedule(dynamic, 4)
        for (int64_t r = 0; r < n_rows; ++r) {
            for (int h = 0; h < hq; ++h) {
#if ORACLE_MUTATION == 4
                const int g = h % hkv;                 /* planted: interleaved grouping */
#else
                const int g = h / group;              /* KV head of query head h */
#endif
                const int64_t i = row_pos[r];
                const int64_t nv = visible_set(kind[g], sink[g], window[g],
                                               idx + idx_off[g],
                                               idx_off[g + 1] - idx_off[g], i, vis);
                const real_t* q = Q + ((size_t)r * hq + h) * d;
                real_t* o = O + ((size_t)r * hq + h) * d;
                if (nv < 0) { failed = 1; continue; }
                if (nv > 0 && vis[nv - 1] >= n_keys) { failed = 1; continue; }
                if (nv == 0) {
                    for (int c = 0; c < d; ++c) o[c] = 0;
                    if (LSE) LSE[(size_t)r * hq + h] = -INFINITY;
                    continue;
                }
                /* pass 1: scores and their maximum */
                real_t m = -INFINITY;
                for (int64_t t = 0; t < nv; ++t) {
                    const real_t* k = K + ((size_t)vis[t] * hkv + g) * d;
                    real_t s = 0;
#if ORACLE_MUTATION == 7
                    for (int c = 0; c < d; ++c) s += q[c] * k[(c + 1) % d];  /* planted: index shift */
#else
                    for (int c = 0; c < d; ++c) s += q[c] * k[c];
#endif
                    s *= scale;
                    score[t] = s;
                    if (s > m) m = s;
                }
                /* pass 2: normaliser and unnormalised weighted sum of values */
                real_t denom = 0;
                for (int c = 0; c < d; ++c) acc[c] = 0;
                for (int64_t t = 0; t < nv; ++t) {
                    const real_t p = R_EXP(score[t] - m);
                    const real_t* v = V + ((size_t)vis[t] * hkv + g) * d;
#if ORACLE_MUTATION == 8
                    if (t > 0) denom += p;                     /* planted: first term dropped */
#else
                    denom += p;
#endif
                    for (int c = 0; c < d; ++c) acc[c] += p * v[c];
                }
                for (int c = 0; c < d; ++c) o[c] = acc[c] / denom;
#if ORACLE_MUTATION == 5
                if (LSE) LSE[(size_t)r * hq + h] = m + R_LOG(denom) / (real_t)0.6931471805599453; /* planted: log2 */
#else
                if (LSE) LSE[(size_t)r * hq + h] = m + R_LOG(denom);
#endif
            }
        }
        free(vis);
        free(score);
        free(acc);
    }
    return failed ? -1 : 0;
}

/* |V(i)| and V(i) itself for one head, exported for the tests. */
int64_t ORACLE_FN(oracle_visible)(int kind, int64_t sink, int64_t window,
                                  const int32_t* idx, int64_t n_idx, int64_t i,
                                  int64_t* out)
{
    return visible_set(kind, sink, window, idx, n_idx, i, out);
}
