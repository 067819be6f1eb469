/*
 * bitdelta_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what the BitDelta hot path computes.
 * It exists so that tests, the package's smoke check and the benchmark's CPU
 * baseline have something independent to compare the CUDA library against.
 * Nothing on the product path may call it; it shares no code, header, table
 * or helper with the CUDA library.
 *
 * Source of every formula: the web page "BitDelta: serving 14 Zen models from
 * one GPU cluster" (Hanzo blog, 2026-02-28), in its sections
 *   "The mathematical foundation"   -- the delta, the 1-bit approximation and
 *                                      the per-matrix scale alpha = mean|delta|,
 *   "Serving architecture"          -- the reconstruction
 *                                      W_eff = W_base + alpha * sign(delta) and
 *                                      the conceptual fused_bitdelta_linear
 *                                      listing (reconstruct, then linear),
 *   "Infrastructure details"        -- storage: sign bits packed 8 per byte
 *                                      (a 4096 x 4096 weight packs to
 *                                      4096 x 512 bytes), alpha kept as f32.
 *
 * Readings where the page is silent:
 *   - sign(0) is +1, stored as bit 1; -0 also gives bit 1.
 *   - bit order: row-major [N, K/32] little-endian u32 words, bit j of word w
 *     in row n <-> column 32*w + j (LSB first).  Byte-for-byte this is the
 *     page's int8 [N, K/8] layout with bit i of byte b <-> column 8*b + i.
 *   - K must be a multiple of 32.
 *   - alpha is one scalar per matrix (the formula); it is stored as the f32
 *     nearest to the fp64 mean.  The per-output-row variant (the storage
 *     paragraph) is bdo_compress_rows.
 *   - the linear uses the STORED f32 alpha (the value a server would hold).
 *   - variant id -1 means "the base model": y = x * W_base^T.
 *
 * Parity status of each function is stated next to it (all are pinned by
 * tests/test_oracle_pins.py; see that file for what pins what).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#include <pthread.h>

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Compression: delta, alpha = mean|delta|, sign bits.                      */
/* "The mathematical foundation": delta = W_ft - W_base;                    */
/* alpha = (1/n) * ||delta||_1 with n the number of entries of the matrix;  */
/* the sign keeps one bit per entry.                                        */
/* Pinned: brute-force packer, hand alpha, closed form, Laplace, zero delta. */
/* ------------------------------------------------------------------------ */

static double load_elem(const void *m, int is_bf16, int64_t e)
{
    return is_bf16 ? bf16_to_double(((const uint16_t *)m)[e])
                   : (double)((const float *)m)[e];
}

/* One pass over the flattened matrix, in index order. */
static int compress_generic(const void *w_ft, const void *w_base, int is_bf16,
                            int64_t N, int64_t K,
                            double *alpha64, float *alpha32, uint32_t *bits)
{
    if (N <= 0 || K <= 0 || K % 32 != 0) return -1;
    int64_t n_elems = N * K;
    memset(bits, 0, (size_t)(n_elems / 32) * sizeof(uint32_t));
    double abs_sum = 0.0;
    for (int64_t e = 0; e < n_elems; ++e) {
        /* delta = W_ft - W_base: exact in fp64 for bf16 inputs and for f32
         * inputs of similar magnitude; never zero unless the inputs are equal */
        double delta = load_elem(w_ft, is_bf16, e) - load_elem(w_base, is_bf16, e);
        abs_sum += fabs(delta);
        if (delta >= 0.0)                      /* sign(0) := +1 -> bit 1 */
            bits[e / 32] |= (uint32_t)1u << (e % 32);
    }
    *alpha64 = abs_sum / (double)n_elems;      /* alpha = (1/n) ||delta||_1 */
    *alpha32 = (float)*alpha64;                /* stored as the nearest f32 */
    return 0;
}

int bdo_compress_f32(const float *w_ft, const float *w_base, int64_t N, int64_t K,
                     double *alpha64, float *alpha32, uint32_t *bits)
{
    return compress_generic(w_ft, w_base, 0, N, K, alpha64, alpha32, bits);
}

int bdo_compress_bf16(const uint16_t *w_ft, const uint16_t *w_base, int64_t N, int64_t K,
                      double *alpha64, float *alpha32, uint32_t *bits)
{
    return compress_generic(w_ft, w_base, 1, N, K, alpha64, alpha32, bits);
}

/* Per-output-row scale, the "Infrastructure details" storage reading:
 * alpha[n] = mean over k of |W_ft[n,k] - W_base[n,k]|; bits as above.
 * Pinned: rows-vs-scalar consistency (N = 1), hand values, Laplace. */
int bdo_compress_rows(const void *w_ft, const void *w_base, int is_bf16,
                      int64_t N, int64_t K, double *alpha64, float *alpha32,
                      uint32_t *bits)
{
    if (N <= 0 || K <= 0 || K % 32 != 0) return -1;
    memset(bits, 0, (size_t)(N * K / 32) * sizeof(uint32_t));
    for (int64_t n = 0; n < N; ++n) {
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            int64_t e = n * K + k;
            double delta = load_elem(w_ft, is_bf16, e) - load_elem(w_base, is_bf16, e);
            s += fabs(delta);
            if (delta >= 0.0)
                bits[e / 32] |= (uint32_t)1u << (e % 32);
        }
        alpha64[n] = s / (double)K;
        alpha32[n] = (float)alpha64[n];
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Materialised reconstruction.                                             */
/* "Serving architecture": the conceptual listing rebuilds                  */
/* W_eff = W_base + alpha * sign(delta) in the base dtype (bf16 here).      */
/* w_eff[n,k] = nearest bf16 (ties to even) of W_base[n,k] + a * s[n,k],    */
/* a = alpha[0] or alpha[n]; the sum is exact in fp64 whenever the two      */
/* terms' exponents differ by less than 29 (always for these workloads).    */
/* Values stay in the normal binary32 range.                                */
/* Pinned: exact closed form, hand-computed ties, exact rational rounding.  */
/* ------------------------------------------------------------------------ */

static uint16_t nearest_bf16(double d)
{
    if (d == 0.0) return signbit(d) ? (uint16_t)0x8000u : (uint16_t)0u;
    int e;
    double m = frexp(fabs(d), &e);              /* |d| = m 2^e, m in [0.5, 1) */
    double q = nearbyint(m * 256.0);            /* 8 significant bits, ties to even */
    float f = (float)ldexp(q, e - 8);           /* exact: at most 9 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t h = (uint16_t)(u >> 16);
    return d < 0.0 ? (uint16_t)(h | 0x8000u) : h;
}

int bdo_reconstruct(const uint16_t *w_base, const float *alpha, int per_row,
                    const uint32_t *bits, int64_t N, int64_t K, uint16_t *w_eff)
{
    if (N <= 0 || K <= 0 || K % 32 != 0) return -1;
    for (int64_t n = 0; n < N; ++n) {
        double a = (double)alpha[per_row ? n : 0];
        for (int64_t k = 0; k < K; ++k) {
            int bit = (int)((bits[(n * K + k) / 32] >> ((n * K + k) % 32)) & 1u);
            double s = (double)(2 * bit - 1);
            w_eff[n * K + k] = nearest_bf16(bf16_to_double(w_base[n * K + k]) + a * s);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Multi-variant linear.                                                    */
/* "Serving architecture": reconstruct W_eff = W_base + alpha_v * sign(d_v), */
/* then y = x * W_eff^T (the conceptual fused_bitdelta_linear listing).     */
/* Each token t uses the variant its request names (variant_ids[t]);        */
/* id -1 is the base model.                                                 */
/* Pinned: zero delta vs numpy matmul, all-ones bits closed form, one-hot x, */
/* closed-form exact reconstruction, linearity identity, torch fp64         */
/* restatement of the listing.                                              */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *x;            /* bf16 [M, K] */
    const int32_t *vid;           /* [M] */
    int64_t M, N, K;
    const uint16_t *w_base;       /* bf16 [N, K] */
    const float *alphas;          /* [V] (per matrix) or [V*N] (per row) */
    int per_row_alpha;
    const uint32_t *const *bits;  /* V pointers, each [N, K/32] */
    int32_t V;
    const int64_t *rows;          /* output rows to compute */
    int64_t nrows;
    double *y;                    /* [M, nrows] */
    int64_t r_begin, r_end;
} linear_job;

static int sign_bit(const uint32_t *bits, int64_t K, int64_t n, int64_t k)
{
    uint32_t word = bits[n * (K / 32) + k / 32];
    return (int)((word >> (k % 32)) & 1u);
}

static void *linear_worker(void *arg)
{
    linear_job *j = (linear_job *)arg;
    int64_t K = j->K;
    double *w_eff = (double *)malloc((size_t)K * sizeof(double));
    double *xrow = (double *)malloc((size_t)K * sizeof(double));
    for (int64_t ri = j->r_begin; ri < j->r_end; ++ri) {
        int64_t n = j->rows[ri];
        for (int64_t t = 0; t < j->M; ++t) {
            int32_t v = j->vid[t];
            /* step 3 of the serving pipeline: the effective weight row */
            for (int64_t k = 0; k < K; ++k) {
                double wb = bf16_to_double(j->w_base[n * K + k]);
                if (v < 0) {
                    w_eff[k] = wb;
                } else {
                    double a = j->per_row_alpha ? (double)j->alphas[(int64_t)v * j->N + n]
                                                : (double)j->alphas[v];
                    double s = sign_bit(j->bits[v], K, n, k) ? 1.0 : -1.0;
                    w_eff[k] = wb + a * s;
                }
            }
            for (int64_t k = 0; k < K; ++k)
                xrow[k] = bf16_to_double(j->x[t * K + k]);
            /* step 4: the forward pass with the reconstructed weight */
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += xrow[k] * w_eff[k];
            j->y[t * j->nrows + ri] = acc;
        }
    }
    free(w_eff);
    free(xrow);
    return NULL;
}

/* y[t, i] = sum_k x[t,k] * W_eff_{v(t)}[rows[i], k], in fp64.
 * Returns -1 on a bad shape and -3 when a variant id lies outside [-1, V). */
int bdo_linear(const uint16_t *x, const int32_t *variant_ids,
               int64_t M, int64_t N, int64_t K,
               const uint16_t *w_base, const float *alphas, int per_row_alpha,
               const uint32_t *const *bits, int32_t V,
               const int64_t *rows, int64_t nrows, double *y, int nthreads)
{
    if (M < 0 || N <= 0 || K <= 0 || K % 32 != 0 || nrows < 0) return -1;
    for (int64_t t = 0; t < M; ++t)
        if (variant_ids[t] < -1 || variant_ids[t] >= V) return -3;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= N) return -1;
    if (M == 0 || nrows == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nrows) nthreads = (int)nrows;
    pthread_t *th = (pthread_t *)malloc((size_t)nthreads * sizeof(pthread_t));
    linear_job *jobs = (linear_job *)malloc((size_t)nthreads * sizeof(linear_job));
    for (int i = 0; i < nthreads; ++i) {
        linear_job j = {x, variant_ids, M, N, K, w_base, alphas, per_row_alpha,
                        bits, V, rows, nrows, y,
                        nrows * i / nthreads, nrows * (i + 1) / nthreads};
        jobs[i] = j;
        pthread_create(&th[i], NULL, linear_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    free(jobs);
    return 0;
}
