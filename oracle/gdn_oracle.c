/*
 * fp64 CPU oracle for the gated delta rule (Gated DeltaNet) — TEST
 * INFRASTRUCTURE.  Used only by the tests; it shares no code with any CUDA
 * path.
 *
 * Source: "Qwen Team Releases FlashQLA for High-Performance Linear Attention"
 * (todayforai.com), sections "Core Technical Principles" and the discussion of
 * the sliding-window property: per token and head, a scalar forget gate
 * alpha_t in (0, 1) and a scalar write strength beta_t in (0, 1) act on the
 * state through alpha_t (I - beta_t k_t^T k_t) with L2-normalised keys.  In
 * the standard gated-delta-rule reading, with S in R^{dk x dv} and row
 * vectors q_t, k_t (dk) and v_t (dv):
 *
 *     S_t = alpha_t (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t
 *     o_t = scale * q_t S_t
 *
 * from S_0 = h0 (zero when absent).  The gate arrives in log space,
 * g_t = log alpha_t.  The keys are used as given (the caller normalises
 * them).  Every operation is carried out in double on the exact input values.
 *
 * Layout (row-major, contiguous): q, k [BH][T][dk]; v, o [BH][T][dv];
 * g, beta [BH][T]; h0, hT [BH][dk][dv].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* One token: S <- alpha (S - beta k^T (k S)) + beta k^T v, then o = scale q S. */
static void gdn_token(double *S, const float *q, const float *k, const float *v, double g,
                      double beta, double scale, double *o, double *kS, int dk, int dv) {
    const double alpha = exp(g);
    for (int c = 0; c < dv; ++c) {            /* kS = k S (1 x dv) */
        double acc = 0.0;
        for (int d = 0; d < dk; ++d) acc += (double)k[d] * S[(int64_t)d * dv + c];
        kS[c] = acc;
    }
    for (int d = 0; d < dk; ++d) {
        const double kd = (double)k[d];
        double *row = S + (int64_t)d * dv;
        for (int c = 0; c < dv; ++c)
            row[c] = alpha * (row[c] - beta * kd * kS[c]) + beta * kd * (double)v[c];
    }
    for (int c = 0; c < dv; ++c) {
        double acc = 0.0;
        for (int d = 0; d < dk; ++d) acc += (double)q[d] * S[(int64_t)d * dv + c];
        o[c] = scale * acc;
    }
}

/*
 * Full-sequence forward for BH independent (batch, head) rows.  Writes o for
 * every token and, when hT != NULL, the state after the last token.
 * Returns 0, or -1 when a work buffer cannot be allocated.
 */
int gdn_oracle_forward(const float *q, const float *k, const float *v, const float *g,
                       const float *beta, double scale, const double *h0, double *o, double *hT,
                       int64_t BH, int64_t T, int dk, int dv, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *S = (double *)malloc(sizeof(double) * (size_t)dk * (size_t)dv);
        double *kS = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!S || !kS) {
            free(S); free(kS);
            failed |= 1;
            continue;
        }
        if (h0) memcpy(S, h0 + bh * dk * dv, sizeof(double) * (size_t)dk * (size_t)dv);
        else memset(S, 0, sizeof(double) * (size_t)dk * (size_t)dv);
        for (int64_t t = 0; t < T; ++t) {
            const int64_t rk = (bh * T + t) * dk, rv = (bh * T + t) * dv, rs = bh * T + t;
            gdn_token(S, q + rk, k + rk, v + rv, (double)g[rs], (double)beta[rs], scale, o + rv,
                      kS, dk, dv);
        }
        if (hT) memcpy(hT + bh * dk * dv, S, sizeof(double) * (size_t)dk * (size_t)dv);
        free(S);
        free(kS);
    }
    return failed ? -1 : 0;
}
