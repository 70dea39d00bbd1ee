/*
 * Grouped differential attention: float64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes (plain definition, no blocking, no online softmax):
 *
 *   For batch b, signal head h (noise head g = h / r, r = h_s / h_n) and
 *   query row i, over the visible keys J(i):
 *     s1_j = q1[b,i,h] . k1[b,j,h] / sqrt(d)
 *     s2_j = q2[b,i,g] . k2[b,j,g] / sqrt(d)
 *     a1   = softmax(s1),  a2 = softmax(s2)          (max-shifted, float64)
 *     o    = sum_j (a1_j - lambda_h * a2_j) * v[b,j,h]      (length dv)
 *     y    = (1 - lambda_init) * o / sqrt(mean(o^2) + eps)   (if norm)
 *
 * Sources:
 *   - "Differential Attention in Large Language Models: How Denoising
 *     Subtraction Eliminates Attention Noise and Outlier Activations",
 *     section "Differential Attention Architecture" (the DiffAttn equation:
 *     two softmax maps, the second weighted by lambda, subtracted and applied
 *     to a shared V whose head width is 2d) and section "Headwise
 *     Normalization" (head_bar = (1 - lambda_init) * RMSNorm(head)).
 *   - "Grouped Differential Attention" (arXiv 2510.06949), abstract: fewer
 *     noise-control heads than signal heads, each noise head reused by a
 *     group of signal heads in the manner of grouped-query attention.  The
 *     group of signal head h is g = floor(h / r) (contiguous groups).
 *   - J(i) = {0..i} when causal, {0..L-1} otherwise; for decode J = {0..len-1}.
 *   - RMSNorm has no learnable gain here (gain = 1).
 *
 * Inputs are float32 arrays holding exactly the values the GPU sees (bf16
 * values widen to float32 without rounding); all arithmetic is float64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* One query row of one signal head.  k1/k2/v point at key row 0 of the head;
 * *_stride is the element distance between consecutive key rows.  s1 and s2
 * are caller scratch of length >= nkeys.  o receives dv doubles. */
static void oracle_row(const float *q1, const float *q2,
                       const float *k1, int64_t k1_stride,
                       const float *k2, int64_t k2_stride,
                       const float *v, int64_t v_stride,
                       int64_t nkeys, int d, int dv,
                       double lam, double lambda_init, double eps, int norm,
                       double *s1, double *s2, double *o)
{
    const double scale = 1.0 / sqrt((double)d);

    /* logits of both maps */
    for (int64_t j = 0; j < nkeys; ++j) {
        const float *k1j = k1 + j * k1_stride;
        const float *k2j = k2 + j * k2_stride;
        double acc1 = 0.0, acc2 = 0.0;
        for (int e = 0; e < d; ++e) {
            acc1 += (double)q1[e] * (double)k1j[e];
            acc2 += (double)q2[e] * (double)k2j[e];
        }
        s1[j] = acc1 * scale;
        s2[j] = acc2 * scale;
    }

    /* softmax of each map, shifted by its own maximum */
    double m1 = -INFINITY, m2 = -INFINITY;
    for (int64_t j = 0; j < nkeys; ++j) {
        if (s1[j] > m1) m1 = s1[j];
        if (s2[j] > m2) m2 = s2[j];
    }
    double z1 = 0.0, z2 = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        s1[j] = exp(s1[j] - m1);
        s2[j] = exp(s2[j] - m2);
        z1 += s1[j];
        z2 += s2[j];
    }
    for (int64_t j = 0; j < nkeys; ++j) {
        s1[j] /= z1;
        s2[j] /= z2;
    }

    /* difference map applied to V */
    for (int c = 0; c < dv; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        const double w = s1[j] - lam * s2[j];
        const float *vj = v + j * v_stride;
        for (int c = 0; c < dv; ++c) o[c] += w * (double)vj[c];
    }

    /* headwise RMSNorm scaled by (1 - lambda_init) */
    if (norm) {
        double ss = 0.0;
        for (int c = 0; c < dv; ++c) ss += o[c] * o[c];
        const double inv = 1.0 / sqrt(ss / (double)dv + eps);
        for (int c = 0; c < dv; ++c) o[c] = (1.0 - lambda_init) * o[c] * inv;
    }
}

static int shapes_ok(int B, int L, int hs, int hn, int d, int dv)
{
    return B >= 0 && L >= 0 && hs > 0 && hn > 0 && hs % hn == 0 && d > 0 && dv > 0;
}

/*
 * Prefill.  q1,k1: [B,L,hs,d]; q2,k2: [B,L,hn,d]; v: [B,L,hs,dv]; lam: [hs].
 * rows == NULL: every query row, out is [B,L,hs,dv].
 * rows != NULL: only the nrows listed query positions, out is [B,nrows,hs,dv].
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int gda_oracle_prefill(const float *q1, const float *k1, const float *q2, const float *k2,
                       const float *v, const double *lam, double lambda_init,
                       int B, int L, int hs, int hn, int d, int dv, int causal,
                       double eps, int norm, const int64_t *rows, int64_t nrows,
                       double *out)
{
    if (!shapes_ok(B, L, hs, hn, d, dv)) return -1;
    const int r = hs / hn;
    const int64_t nq = rows ? nrows : (int64_t)L;
    for (int64_t t = 0; rows && t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= L) return -1;
    const int64_t total = (int64_t)B * nq * hs;
    int failed = 0;

#pragma omp parallel reduction(| : failed)
    {
        double *s1 = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double *s2 = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        if (!s1 || !s2) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t w = 0; w < total; ++w) {
                const int h = (int)(w % hs);
                const int64_t t = (w / hs) % nq;
                const int b = (int)(w / ((int64_t)hs * nq));
                const int64_t i = rows ? rows[t] : t;
                const int g = h / r;
                const int64_t nkeys = causal ? i + 1 : (int64_t)L;
                const float *q1r = q1 + (((int64_t)b * L + i) * hs + h) * d;
                const float *q2r = q2 + (((int64_t)b * L + i) * hn + g) * d;
                const float *k1b = k1 + ((int64_t)b * L * hs + h) * d;
                const float *k2b = k2 + ((int64_t)b * L * hn + g) * d;
                const float *vb = v + ((int64_t)b * L * hs + h) * dv;
                double *o = out + (((int64_t)b * nq + t) * hs + h) * dv;
                oracle_row(q1r, q2r, k1b, (int64_t)hs * d, k2b, (int64_t)hn * d,
                           vb, (int64_t)hs * dv, nkeys, d, dv, lam[h], lambda_init,
                           eps, norm, s1, s2, o);
            }
        }
        free(s1);
        free(s2);
    }
    return failed ? -1 : 0;
}

/*
 * Decode: one new query token per sequence against its key/value cache.
 * q1: [B,hs,d]; q2: [B,hn,d]; k1c: [B,Lcap,hs,d]; k2c: [B,Lcap,hn,d];
 * vc: [B,Lcap,hs,dv]; lens: [B] with 1 <= lens[b] <= Lcap (the new token is
 * already in the cache at position lens[b]-1); out: [B,hs,dv].
 */
int gda_oracle_decode(const float *q1, const float *q2, const float *k1c, const float *k2c,
                      const float *vc, const int32_t *lens, const double *lam,
                      double lambda_init, int B, int Lcap, int hs, int hn, int d, int dv,
                      double eps, int norm, double *out)
{
    if (!shapes_ok(B, Lcap, hs, hn, d, dv)) return -1;
    for (int b = 0; b < B; ++b)
        if (lens[b] < 1 || lens[b] > Lcap) return -1;
    const int r = hs / hn;
    const int64_t total = (int64_t)B * hs;
    int failed = 0;

#pragma omp parallel reduction(| : failed)
    {
        double *s1 = (double *)malloc(sizeof(double) * (size_t)(Lcap > 0 ? Lcap : 1));
        double *s2 = (double *)malloc(sizeof(double) * (size_t)(Lcap > 0 ? Lcap : 1));
        if (!s1 || !s2) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t w = 0; w < total; ++w) {
                const int h = (int)(w % hs);
                const int b = (int)(w / hs);
                const int g = h / r;
                const float *q1r = q1 + ((int64_t)b * hs + h) * d;
                const float *q2r = q2 + ((int64_t)b * hn + g) * d;
                const float *k1b = k1c + ((int64_t)b * Lcap * hs + h) * d;
                const float *k2b = k2c + ((int64_t)b * Lcap * hn + g) * d;
                const float *vb = vc + ((int64_t)b * Lcap * hs + h) * dv;
                double *o = out + ((int64_t)b * hs + h) * dv;
                oracle_row(q1r, q2r, k1b, (int64_t)hs * d, k2b, (int64_t)hn * d,
                           vb, (int64_t)hs * dv, lens[b], d, dv, lam[h], lambda_init,
                           eps, norm, s1, s2, o);
            }
        }
        free(s1);
        free(s2);
    }
    return failed ? -1 : 0;
}

/* Threads the OpenMP runtime will use for the calls above. */
int gda_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Restrict the oracle to n threads (n >= 1). */
void gda_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
