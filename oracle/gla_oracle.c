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

/* ------------------------------------------------------------------------ */
/*
 * Backward pass — gradients of a scalar loss through the same recurrence.
 *
 * Source: the recurrence of "The Gated Recurrent Update" above; the same
 * page's section "I/O-Aware Kernel Design in FlashLinearAttention" names a
 * backward pass that recomputes the chunk states instead of caching them.
 * The pages print no backward equations, so this is reverse-mode
 * differentiation of the token loop, written out.  With the loss
 *
 *     L = sum_t <do_t, o_t> + <dhT, hT>,
 *
 * the adjoint G_t = dL/dS_t obeys G_T = dhT + scale q_T^T do_T and
 * G_{t-1} = diag(alpha_t) G_t + scale q_{t-1}^T do_{t-1}; per token t:
 *
 *     dq_t = scale * S_t do_t                   (S_t after token t)
 *     dk_t = G_t v_t^T,  dv_t = k_t G_t
 *     dlog_alpha_t = alpha_t (.) rowsum(G_t (.) S_{t-1})
 *     dh0 = diag(alpha_1) G_1
 *
 * (the last because S_{t-1} -> S_t multiplies row d by alpha_t[d], and
 * d alpha / d log alpha = alpha).
 *
 * Memory schedule: the loop needs S_{t-1} and S_t going backward in t.  States
 * are kept at checkpoints every `ck` tokens and each block of tokens is
 * replayed from its checkpoint with the same update as the forward pass, so
 * every state is bit-identical to the one the forward loop computes.  `ck` is
 * a memory setting only (0 = about sqrt(T)); results do not depend on it.
 */

/* S <- diag(exp(a)) S + k^T v, the state half of gla_oracle_token. */
static void gla_oracle_update(double *S, const float *k, const float *v, const float *a, int dk,
                              int dv) {
    for (int d = 0; d < dk; ++d) {
        const double alpha = exp((double)a[d]);
        const double kd = (double)k[d];
        double *row = S + (int64_t)d * dv;
        for (int c = 0; c < dv; ++c) row[c] = alpha * row[c] + kd * (double)v[c];
    }
}

/*
 * q, k, log_alpha [BH][T][dk]; v, d_o [BH][T][dv]; h0, dhT [BH][dk][dv]
 * (either may be NULL = zero).  Writes grad_q, grad_k, grad_log_alpha
 * [BH][T][dk], grad_v [BH][T][dv] and, when grad_h0 != NULL, [BH][dk][dv].
 * Returns 0, or -1 when a work buffer cannot be allocated.
 */
int gla_oracle_backward(const float *q, const float *k, const float *v, const float *log_alpha,
                        double scale, const double *h0, const float *d_o, const double *dhT,
                        double *grad_q, double *grad_k, double *grad_v, double *grad_log_alpha,
                        double *grad_h0, int64_t BH, int64_t T, int dk, int dv, int64_t ck,
                        int nthreads) {
    set_threads(nthreads);
    if (ck <= 0) {
        ck = 1;
        while (ck * ck < T) ++ck;
    }
    const int64_t nck = T > 0 ? (T + ck - 1) / ck : 0;  /* checkpoints at t = 0, ck, 2ck, ... */
    const size_t ssz = (size_t)dk * (size_t)dv;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *cp = (double *)malloc(sizeof(double) * ssz * (size_t)(nck > 0 ? nck : 1));
        double *blk = (double *)malloc(sizeof(double) * ssz * (size_t)(ck + 1));
        double *G = (double *)malloc(sizeof(double) * ssz);
        if (!cp || !blk || !G) {
            free(cp); free(blk); free(G);
            failed |= 1;
            continue;
        }
        const float *qh = q + bh * T * dk, *kh = k + bh * T * dk, *ah = log_alpha + bh * T * dk;
        const float *vh = v + bh * T * dv, *doh = d_o + bh * T * dv;
        /* forward sweep: keep S_t at t = 0, ck, 2ck, ... (S_0 = h0) */
        double *S = blk;
        if (h0) memcpy(S, h0 + bh * (int64_t)ssz, sizeof(double) * ssz);
        else memset(S, 0, sizeof(double) * ssz);
        for (int64_t t = 0; t < T; ++t) {
            if (t % ck == 0) memcpy(cp + (t / ck) * (int64_t)ssz, S, sizeof(double) * ssz);
            gla_oracle_update(S, kh + t * dk, vh + t * dv, ah + t * dk, dk, dv);
        }
        /* adjoint of the final state */
        if (dhT) memcpy(G, dhT + bh * (int64_t)ssz, sizeof(double) * ssz);
        else memset(G, 0, sizeof(double) * ssz);
        for (int64_t b = nck - 1; b >= 0; --b) {
            const int64_t t0 = b * ck, t1 = (t0 + ck < T) ? t0 + ck : T;
            /* replay: blk[j] = S_{t0 + j} for j = 0 .. t1 - t0 */
            memcpy(blk, cp + b * (int64_t)ssz, sizeof(double) * ssz);
            for (int64_t t = t0; t < t1; ++t) {
                double *nxt = blk + (t - t0 + 1) * (int64_t)ssz;
                memcpy(nxt, blk + (t - t0) * (int64_t)ssz, sizeof(double) * ssz);
                gla_oracle_update(nxt, kh + t * dk, vh + t * dv, ah + t * dk, dk, dv);
            }
            /* token t (0-based) maps S_t -> S_{t+1}; o_t reads S_{t+1} */
            for (int64_t t = t1 - 1; t >= t0; --t) {
                const double *Sprev = blk + (t - t0) * (int64_t)ssz;
                const double *Scur = blk + (t - t0 + 1) * (int64_t)ssz;
                const float *qt = qh + t * dk, *kt = kh + t * dk, *at = ah + t * dk;
                const float *vt = vh + t * dv, *dot = doh + t * dv;
                double *gq = grad_q + (bh * T + t) * dk, *gk = grad_k + (bh * T + t) * dk;
                double *ga = grad_log_alpha + (bh * T + t) * dk, *gv = grad_v + (bh * T + t) * dv;
                /* o_t = scale q_t S_{t+1}: add its share to the adjoint of S_{t+1} */
                for (int d = 0; d < dk; ++d) {
                    const double sq = scale * (double)qt[d];
                    double *row = G + (int64_t)d * dv;
                    for (int c = 0; c < dv; ++c) row[c] += sq * (double)dot[c];
                }
                for (int d = 0; d < dk; ++d) {
                    const double *srow = Scur + (int64_t)d * dv, *grow = G + (int64_t)d * dv;
                    const double *prow = Sprev + (int64_t)d * dv;
                    double aq = 0.0, ak = 0.0, aa = 0.0;
                    for (int c = 0; c < dv; ++c) {
                        aq += srow[c] * (double)dot[c];
                        ak += grow[c] * (double)vt[c];
                        aa += grow[c] * prow[c];
                    }
                    gq[d] = scale * aq;
                    gk[d] = ak;
                    ga[d] = exp((double)at[d]) * aa;
                }
                for (int c = 0; c < dv; ++c) {
                    double acc = 0.0;
                    for (int d = 0; d < dk; ++d) acc += (double)kt[d] * G[(int64_t)d * dv + c];
                    gv[c] = acc;
                }
                /* S_{t+1} = diag(alpha_t) S_t + ...: pass the adjoint back to S_t */
                for (int d = 0; d < dk; ++d) {
                    const double alpha = exp((double)at[d]);
                    double *row = G + (int64_t)d * dv;
                    for (int c = 0; c < dv; ++c) row[c] *= alpha;
                }
            }
        }
        if (grad_h0) memcpy(grad_h0 + bh * (int64_t)ssz, G, sizeof(double) * ssz);
        free(cp); free(blk); free(G);
    }
    return failed ? -1 : 0;
}
