/*
 * gqa_oracle.c -- slow, plain fp64 CPU oracle for grouped-query attention
 * forward (causal prefill and single-token decode).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package smoke check and the bench's
 * CPU-baseline arm use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes (chowfi/kernels README, "Result" section and the settings
 * line under its table; "What helped most", item 3 for the causal mask):
 * the attention step of a Llama-3-8B-size model, forward only, with 32 query
 * heads sharing 8 KV heads and head size 128, in bf16.  Written out, for
 * every query head h with KV head g = floor(h / (Hq / Hkv)):
 *
 *     s_j    = (sum_d q[i,h,d] * k[j,g,d]) / sqrt(D)       for j in J(i)
 *     m      = max_j s_j
 *     w_j    = exp(s_j - m)
 *     out[i,h,:] = (sum_j w_j * v[j,g,:]) / (sum_j w_j)
 *
 * with J(i) = {0..i} for causal prefill (query i sees itself and the past),
 * J(i) = {0..S-1} for non-causal prefill, and J = {0..L-1} for decode (one
 * new query against a KV cache of length L, every cached position visible).
 *
 * Everything is fp64, from the exact values of the bf16 inputs; the result
 * is left unrounded.  The head counts and head size are parameters so the
 * tests can compare grouped heads with plain multi-head attention.
 *
 * Layout: q [n_q][hq][d], k and v [n_kv][hkv][d], out [n_q][hq][d], all
 * row-major (batch 1, sequence-major "BSHD").  Inputs are raw bf16 bit
 * patterns (uint16).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE-754 binary32: widen by a 16-bit shift. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One (query row, query head) of softmax attention over keys 0..n_keys-1
 * of KV head g.  w is caller scratch of n_keys doubles; on return it holds
 * the normalised softmax weights.  Returns the log-sum-exp of the scaled
 * scores (natural log). */
static double attend_one(const uint16_t *qrow, const uint16_t *k,
                         const uint16_t *v, int hkv, int d, int g,
                         long n_keys, double *w, double *out)
{
    const double scale = 1.0 / sqrt((double)d);
    double m = -INFINITY;
    for (long j = 0; j < n_keys; ++j) {
        const uint16_t *krow = k + ((size_t)j * hkv + g) * d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c)
            dot += bf16_bits_to_double(qrow[c]) * bf16_bits_to_double(krow[c]);
        w[j] = dot * scale;
        if (w[j] > m)
            m = w[j];
    }
    double l = 0.0;
    for (long j = 0; j < n_keys; ++j) {
        w[j] = exp(w[j] - m);
        l += w[j];
    }
    for (int c = 0; c < d; ++c)
        out[c] = 0.0;
    for (long j = 0; j < n_keys; ++j) {
        const uint16_t *vrow = v + ((size_t)j * hkv + g) * d;
        w[j] /= l;
        for (int c = 0; c < d; ++c)
            out[c] += w[j] * bf16_bits_to_double(vrow[c]);
    }
    return m + log(l);
}

static int check_geometry(int hq, int hkv, int d)
{
    if (hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv != 0)
        return 1;
    return 0;
}

static void set_threads(int n_threads)
{
#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
}

/*
 * Attention for the listed query rows of a prefill of length S.
 * rows[r] in [0, S); out is [n_rows][hq][d]; lse (may be NULL) [n_rows][hq].
 * Returns 0, or 1 on bad arguments, 2 on allocation failure.
 */
int gqa_oracle_prefill_rows(const uint16_t *q, const uint16_t *k,
                            const uint16_t *v, long S, int hq, int hkv, int d,
                            int causal, const int64_t *rows, long n_rows,
                            double *out, double *lse, int n_threads)
{
    if (check_geometry(hq, hkv, d) || S <= 0 || n_rows < 0)
        return 1;
    for (long r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= S)
            return 1;
    const int group = hq / hkv;
    int failed = 0;
    set_threads(n_threads);
#pragma omp parallel
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)S);
        if (!w) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long t = 0; t < n_rows * hq; ++t) {
            if (!w)
                continue;
            const long r = t / hq;
            const int h = (int)(t % hq);
            const long i = rows[r];
            const long n_keys = causal ? i + 1 : S;
            double x = attend_one(q + ((size_t)i * hq + h) * d, k, v, hkv, d,
                                  h / group, n_keys, w,
                                  out + ((size_t)r * hq + h) * d);
            if (lse)
                lse[(size_t)r * hq + h] = x;
        }
        free(w);
    }
    return failed ? 2 : 0;
}

/* Full prefill: every query row 0..S-1.  out [S][hq][d], lse [S][hq]. */
int gqa_oracle_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       long S, int hq, int hkv, int d, int causal, double *out,
                       double *lse, int n_threads)
{
    if (S <= 0)
        return 1;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)S);
    if (!rows)
        return 2;
    for (long i = 0; i < S; ++i)
        rows[i] = i;
    int rc = gqa_oracle_prefill_rows(q, k, v, S, hq, hkv, d, causal, rows, S,
                                     out, lse, n_threads);
    free(rows);
    return rc;
}

/*
 * Decode: one query q [hq][d] against a KV cache kc, vc [L][hkv][d]; every
 * cached position is visible.  out [hq][d], lse (may be NULL) [hq].
 */
int gqa_oracle_decode(const uint16_t *q, const uint16_t *kc,
                      const uint16_t *vc, long L, int hq, int hkv, int d,
                      double *out, double *lse, int n_threads)
{
    if (check_geometry(hq, hkv, d) || L <= 0)
        return 1;
    const int group = hq / hkv;
    int failed = 0;
    set_threads(n_threads);
#pragma omp parallel
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)L);
        if (!w) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(static, 1)
        for (int h = 0; h < hq; ++h) {
            if (!w)
                continue;
            double x = attend_one(q + (size_t)h * d, kc, vc, hkv, d, h / group,
                                  L, w, out + (size_t)h * d);
            if (lse)
                lse[h] = x;
        }
        free(w);
    }
    return failed ? 2 : 0;
}

/*
 * The normalised softmax weights of one (query row i, query head h) of a
 * prefill: w [n_keys] with n_keys = i + 1 (causal) or S.  Exposed so the
 * tests can check that every row of weights is a probability vector.
 */
int gqa_oracle_weights(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       long S, int hq, int hkv, int d, int causal, long i,
                       int h, double *w, double *out_row)
{
    if (check_geometry(hq, hkv, d) || S <= 0 || i < 0 || i >= S || h < 0 ||
        h >= hq)
        return 1;
    const long n_keys = causal ? i + 1 : S;
    attend_one(q + ((size_t)i * hq + h) * d, k, v, hkv, d, h / (hq / hkv),
               n_keys, w, out_row);
    return 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int gqa_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
