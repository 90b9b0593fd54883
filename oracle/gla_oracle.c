/*
 * fp64 CPU oracle for gated linear attention (GLA) — TEST INFRASTRUCTURE.
 *
 * This file is the definition of what the CUDA path computes, written out as
 * a plain token-by-token loop.  It is used only by the tests, by the package
 * entry's smoke check and by the benchmark's CPU-baseline leg.  It shares no
 * code, header, table or helper with the CUDA library, and the product path
 * never calls it.
 *
 * Source: "Gated Linear Attention (GLA): Mathematical Foundations, Data-
 * Dependent Gating, Chunkwise Parallel Forms, and Sub-Quadratic Sequence
 * Modeling" (llms.blog), section "The Gated Recurrent Update":
 *
 *     S_t = diag(alpha_t) S_{t-1} + k_t^T v_t,     S in R^{dk x dv}
 *     o_t = q_t S_t
 *
 * with S_0 = 0 (section "Linearized Attention as Associative Memory") unless
 * an initial state h0 is given.  Readings taken where the page is silent:
 *   - the gate is supplied in log space, A_t = log(alpha_t) ("Sequence
 *     Partitioning and State Factorization" defines A the same way), so
 *     alpha_t = exp(A_t);
 *   - the output carries a caller-chosen factor `scale`: o_t = scale * q_t S_t;
 *     the state does not carry it;
 *   - o_t reads the state AFTER the token-t update (the page's equation order).
 *
 * Inputs are the exact values the GPU sees (bf16 and fp32 both convert to
 * float exactly); every operation below is carried out in double.
 *
 * Layout (row-major, contiguous): q, k, log_alpha [BH][T][dk]; v [BH][T][dv];
 * h0, hT [BH][dk][dv] (row = key channel); o [BH][T][dv].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* One recurrence step on one head: S <- diag(exp(a)) S + k^T v, then
 * o = scale * q S.  S is dk x dv doubles, updated in place. */
static void gla_oracle_token(double *S, const float *q, const float *k, const float *v,
                             const float *a, double scale, double *o, int dk, int dv) {
    for (int d = 0; d < dk; ++d) {
        const double alpha = exp((double)a[d]);
        const double kd = (double)k[d];
        double *row = S + (int64_t)d * dv;
        for (int c = 0; c < dv; ++c) row[c] = alpha * row[c] + kd * (double)v[c];
    }
    for (int c = 0; c < dv; ++c) {
        double acc = 0.0;
        for (int d = 0; d < dk; ++d) acc += (double)q[d] * S[(int64_t)d * dv + c];
        o[c] = scale * acc;
    }
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Number of threads OpenMP will use for the next parallel region. */
int gla_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Full-sequence forward: for every (batch, head) pair independently, run the
 * recurrence over T tokens from h0 (or zero when h0 == NULL).  Writes o for
 * every token and, when hT != NULL, the state after the last token.
 * Returns 0, or -1 when a work buffer cannot be allocated.
 */
int gla_oracle_forward(const float *q, const float *k, const float *v, const float *log_alpha,
                       double scale, const double *h0, double *o, double *hT, int64_t BH,
                       int64_t T, int dk, int dv, int nthreads) {
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *S = (double *)malloc(sizeof(double) * (size_t)dk * (size_t)dv);
        if (!S) { failed |= 1; continue; }
        if (h0) memcpy(S, h0 + bh * dk * dv, sizeof(double) * (size_t)dk * (size_t)dv);
        else memset(S, 0, sizeof(double) * (size_t)dk * (size_t)dv);
        for (int64_t t = 0; t < T; ++t) {
            const int64_t rk = (bh * T + t) * dk, rv = (bh * T + t) * dv;
            gla_oracle_token(S, q + rk, k + rk, v + rv, log_alpha + rk, scale, o + rv, dk, dv);
        }
        if (hT) memcpy(hT + bh * dk * dv, S, sizeof(double) * (size_t)dk * (size_t)dv);
        free(S);
    }
    return failed ? -1 : 0;
}

/*
 * One decode step for BH independent heads: the same update as one token of
 * the forward, applied to a state h [BH][dk][dv] carried in double and
 * updated in place; q, k, log_alpha are [BH][dk], v and o are [BH][dv].
 */
void gla_oracle_step(const float *q, const float *k, const float *v, const float *log_alpha,
                     double scale, double *h, double *o, int64_t BH, int dk, int dv,
                     int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t bh = 0; bh < BH; ++bh) {
        gla_oracle_token(h + bh * dk * dv, q + bh * dk, k + bh * dk, v + bh * dv,
                         log_alpha + bh * dk, scale, o + bh * dv, dk, dv);
    }
}
