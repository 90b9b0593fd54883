// gla_backward.cu — gradients of the gated recurrence (chunkwise backward).
//
// Forward, per (batch, head) ("Gated Linear Attention (GLA): Mathematical
// Foundations, ..." (llms.blog), section "The Gated Recurrent Update"):
//     S_t = diag(alpha_t) S_{t-1} + k_t^T v_t,   o_t = scale q_t S_t.
// For the loss L = sum_t <do_t, o_t> + <dhT, hT>, the gradients in chunk form
// (chunk of BC tokens, in-chunk inclusive prefix sums Gamma of log alpha as in
// section "Cumulative Decay Representation", S_u = the state entering chunk
// u, R_u = dL/d(state leaving chunk u)):
//
//     A      = tril(dO V^T)                                       (C x C)
//     M      = tril((Q e^Gamma)(K e^-Gamma)^T)                    (decay inside
//              the key-channel sum, as in "Intra-Chunk Matrix Multiplications")
//     dQ     = scale [ e^Gamma (dO S_u^T) + e^Gamma (A (K e^-Gamma)) ]
//     dK     = scale e^-Gamma (A^T (Q e^Gamma)) + e^(Gamma_C - Gamma) (V R_u^T)
//     dV     = scale M^T dO + (K e^(Gamma_C - Gamma)) R_u
//     dlog_alpha_t = rowsum(R_u * S_(u+1)) + sum_{tau >= t in chunk}
//                    (q_tau dq_tau - k_tau dk_tau)
//     R_(u-1) = diag(e^Gamma_C) R_u + scale (Q e^Gamma)^T dO,   R_last = dhT,
//     dh0     = R_(-1),
//
// where the states are recomputed ("Inter-Chunk Recurrence and Output
// Projection": S_(u+1) = diag(e^Gamma_C) S_u + (K e^(Gamma_C - Gamma))^T V).
// The log-gate carry is the gradient of the first token of the next chunk:
// shifting log alpha there scales the state leaving chunk u row by row.
//
// Three kernels, all on CUDA cores in fp32:
//   1. bwd_states:  one CTA per (32-column tile, head) walks the chunks
//      forward and writes S_u for u = 0 .. NC (S_0 = h0) to scratch;
//   2. bwd_adjoint: the same tiling walks the chunks backward, writes R_u,
//      the per-tile row sums of R_u * S_(u+1) (the log-gate carry), and dh0;
//   3. bwd_grads:   one CTA per (chunk, head), independent of every other
//      chunk, computes dq, dk, dv and dlog_alpha.
// Inside a chunk the decay factor e^(Gamma_t - Gamma_j) (t >= j) is split
// around a per-channel reference r = (Gamma_0 + Gamma_(C-1)) / 2, so both
// halves stay within 2^+-60 when the chunk's decay spans at most 2^120; a
// chunk that decays further takes each factor as one exponential ("exact"
// path).  All exponentials are base 2 on log2-scaled prefix sums.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr int BC = 64;          // tokens per backward chunk
constexpr int TW = 32;          // value columns per state tile (bwd_states / bwd_adjoint)
constexpr int NT = 256;         // threads per CTA
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaxSpan = 120.f;  // log2 units: larger in-chunk decay spans take the exact path

__device__ __forceinline__ float bf(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}

// Load one chunk of log-gates (log2 units, rows past the sequence end zero,
// so the prefix sum stays flat there) and take the inclusive prefix sum per
// channel.  sG is [BC][LD].
template <int DK, int LD>
__device__ __forceinline__ void load_prefix(float *sG, const float *__restrict__ la, int n) {
    for (int e = threadIdx.x; e < BC * DK; e += NT) {
        const int t = e / DK, i = e % DK;
        sG[t * LD + i] = t < n ? la[static_cast<size_t>(t) * DK + i] * kLog2e : 0.f;
    }
    __syncthreads();
    if (threadIdx.x < DK) {
        float acc = 0.f;
        for (int t = 0; t < BC; ++t) {
            acc += sG[t * LD + threadIdx.x];
            sG[t * LD + threadIdx.x] = acc;
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// 1. chunk-start states.  Thread (warp w, lane c) owns column c of the tile and
//    rows w, w + 8, w + 16, ...
template <int DK, int DV>
__global__ void __launch_bounds__(NT) bwd_states_kernel(BwdLaunch p) {
    constexpr int RPT = DK / 8;
    extern __shared__ float smem[];
    float *sG = smem;                  // [BC][DK]
    float *sK = sG + BC * DK;          // [BC][DK]: k e^(Gamma_C - Gamma)
    float *sV = sK + BC * DK;          // [BC][TW]
    const int tile = blockIdx.x, bh = blockIdx.y;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int c0 = tile * TW;
    const size_t base_k = static_cast<size_t>(bh) * p.T * DK;
    const size_t base_v = static_cast<size_t>(bh) * p.T * DV;
    float *Sout = p.states + static_cast<size_t>(bh) * (p.NC + 1) * DK * DV;

    float S[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m)
        S[m] = p.h0 ? p.h0[(static_cast<size_t>(bh) * DK + w + 8 * m) * DV + c0 + lane] : 0.f;

    for (int u = 0; u < p.NC; ++u) {
        const int t0 = u * BC, n = min(BC, p.T - t0);
        load_prefix<DK, DK>(sG, p.log_alpha + base_k + static_cast<size_t>(t0) * DK, n);
        for (int e = threadIdx.x; e < BC * DK; e += NT) {
            const int t = e / DK, i = e % DK;
            const float kk = t < n ? bf(p.k, base_k + static_cast<size_t>(t0 + t) * DK + i) : 0.f;
            sK[e] = kk * exp2f(sG[(BC - 1) * DK + i] - sG[e]);
        }
        for (int e = threadIdx.x; e < BC * TW; e += NT) {
            const int t = e / TW, c = e % TW;
            sV[e] = t < n ? bf(p.v, base_v + static_cast<size_t>(t0 + t) * DV + c0 + c) : 0.f;
        }
        __syncthreads();
        float *dst = Sout + static_cast<size_t>(u) * DK * DV;
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int i = w + 8 * m;
            dst[static_cast<size_t>(i) * DV + c0 + lane] = S[m];
            float acc = exp2f(sG[(BC - 1) * DK + i]) * S[m];
            for (int j = 0; j < BC; ++j) acc = fmaf(sK[j * DK + i], sV[j * TW + lane], acc);
            S[m] = acc;
        }
        __syncthreads();
    }
    float *dst = Sout + static_cast<size_t>(p.NC) * DK * DV;
#pragma unroll
    for (int m = 0; m < RPT; ++m) dst[static_cast<size_t>(w + 8 * m) * DV + c0 + lane] = S[m];
}

// ---------------------------------------------------------------------------
// 2. adjoint states, walking the chunks backward.  Same thread layout.
template <int DK, int DV>
__global__ void __launch_bounds__(NT) bwd_adjoint_kernel(BwdLaunch p) {
    constexpr int RPT = DK / 8;
    constexpr int NTILE = DV / TW;
    extern __shared__ float smem[];
    float *sG = smem;                  // [BC][DK]
    float *sQ = sG + BC * DK;          // [BC][DK]: q e^Gamma
    float *sD = sQ + BC * DK;          // [BC][TW]: do
    const int tile = blockIdx.x, bh = blockIdx.y;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int c0 = tile * TW;
    const size_t base_k = static_cast<size_t>(bh) * p.T * DK;
    const size_t base_v = static_cast<size_t>(bh) * p.T * DV;
    const float *Sin = p.states + static_cast<size_t>(bh) * (p.NC + 1) * DK * DV;
    float *Rout = p.adjoints + static_cast<size_t>(bh) * p.NC * DK * DV;
    float *carry = p.carry + static_cast<size_t>(bh) * p.NC * NTILE * DK;

    float R[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m)
        R[m] = p.dhT ? p.dhT[(static_cast<size_t>(bh) * DK + w + 8 * m) * DV + c0 + lane] : 0.f;

    for (int u = p.NC - 1; u >= 0; --u) {
        const int t0 = u * BC, n = min(BC, p.T - t0);
        load_prefix<DK, DK>(sG, p.log_alpha + base_k + static_cast<size_t>(t0) * DK, n);
        for (int e = threadIdx.x; e < BC * DK; e += NT) {
            const int t = e / DK, i = e % DK;
            const float qq = t < n ? bf(p.q, base_k + static_cast<size_t>(t0 + t) * DK + i) : 0.f;
            sQ[e] = qq * exp2f(sG[e]);
        }
        for (int e = threadIdx.x; e < BC * TW; e += NT) {
            const int t = e / TW, c = e % TW;
            sD[e] = t < n ? bf(p.d_o, base_v + static_cast<size_t>(t0 + t) * DV + c0 + c) : 0.f;
        }
        __syncthreads();
        float *dst = Rout + static_cast<size_t>(u) * DK * DV;
        const float *snext = Sin + static_cast<size_t>(u + 1) * DK * DV;
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int i = w + 8 * m;
            const size_t off = static_cast<size_t>(i) * DV + c0 + lane;
            dst[off] = R[m];
            float part = R[m] * snext[off];
#pragma unroll
            for (int s = 16; s > 0; s >>= 1) part += __shfl_xor_sync(0xffffffffu, part, s);
            if (lane == 0) carry[(static_cast<size_t>(u) * NTILE + tile) * DK + i] = part;
            float acc = 0.f;
            for (int t = 0; t < BC; ++t) acc = fmaf(sQ[t * DK + i], sD[t * TW + lane], acc);
            R[m] = fmaf(exp2f(sG[(BC - 1) * DK + i]), R[m], p.scale * acc);
        }
        __syncthreads();
    }
    if (p.gh0) {
#pragma unroll
        for (int m = 0; m < RPT; ++m)
            p.gh0[(static_cast<size_t>(bh) * DK + w + 8 * m) * DV + c0 + lane] = R[m];
    }
}

// ---------------------------------------------------------------------------
// 3. per-chunk gradients.  Thread (ty, tx) = (tid / 16, tid % 16) owns rows
//    4 ty .. 4 ty + 3 and columns tx, tx + 16, ... of every C x C, C x dk and
//    C x 32 block it computes.
template <int DK>
struct GradSmem {
    static constexpr int LD = DK + 1;      // odd strides: conflict-free column walks
    static constexpr int LA = BC + 1;
    static constexpr int LS = TW + 1;
    static constexpr int kG = 0, kQ = kG + BC * LD, kK = kQ + BC * LD, kP = kK + BC * LD;
    static constexpr int kAM = kP + BC * LD;
    static constexpr int kDo = kAM + BC * LA, kV = kDo + BC * LS;
    static constexpr int kS = kV + BC * LS, kR = kS + DK * LS;
    static constexpr int kRef = kR + DK * LS, kGC = kRef + DK, kCarry = kGC + DK;
    static constexpr int kFloats = kCarry + DK;
    static constexpr size_t kBytes = sizeof(float) * kFloats;
};

template <int DK, int DV>
__global__ void __launch_bounds__(NT, 1) bwd_grads_kernel(BwdLaunch p) {
    using L = GradSmem<DK>;
    constexpr int LD = L::LD, LA = L::LA, LS = L::LS;
    constexpr int NB = DK / 16;            // key-channel columns per thread
    constexpr int NTILE = DV / TW;
    extern __shared__ float smem[];
    float *sG = smem + L::kG, *sQ = smem + L::kQ, *sK = smem + L::kK, *sP = smem + L::kP;
    float *sAM = smem + L::kAM, *sDo = smem + L::kDo, *sV = smem + L::kV;
    float *sS = smem + L::kS, *sR = smem + L::kR;
    float *sRef = smem + L::kRef, *sGC = smem + L::kGC, *sCarry = smem + L::kCarry;

    const int u = blockIdx.x, bh = blockIdx.y;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int t0 = u * BC, n = min(BC, p.T - t0);
    const size_t rk = (static_cast<size_t>(bh) * p.T + t0) * DK;   // first row, key tensors
    const size_t rv = (static_cast<size_t>(bh) * p.T + t0) * DV;   // first row, value tensors
    const float *Su = p.states + (static_cast<size_t>(bh) * (p.NC + 1) + u) * DK * DV;
    const float *Ru = p.adjoints + (static_cast<size_t>(bh) * p.NC + u) * DK * DV;
    const float s = p.scale;

    // prefix sums, the reference and the path choice
    load_prefix<DK, LD>(sG, p.log_alpha + rk, n);
    int wide = 0;
    if (tid < DK) {
        const float g0 = sG[tid], gl = sG[(BC - 1) * LD + tid];
        sRef[tid] = 0.5f * (g0 + gl);
        sGC[tid] = gl;
        wide = (g0 - gl) > kMaxSpan;
        float c = 0.f;
        for (int x = 0; x < NTILE; ++x)
            c += p.carry[((static_cast<size_t>(bh) * p.NC + u) * NTILE + x) * DK + tid];
        sCarry[tid] = c;
    }
    const bool exact = __syncthreads_or(wide) || p.force_exact;

    // q and k: rescaled around the reference (fast path) or raw (exact path)
    for (int e = tid; e < BC * DK; e += NT) {
        const int t = e / DK, i = e % DK;
        const float qq = t < n ? bf(p.q, rk + static_cast<size_t>(t) * DK + i) : 0.f;
        const float kk = t < n ? bf(p.k, rk + static_cast<size_t>(t) * DK + i) : 0.f;
        const float d = exact ? 0.f : sG[t * LD + i] - sRef[i];
        sQ[t * LD + i] = qq * exp2f(d);
        sK[t * LD + i] = kk * exp2f(-d);
    }

    // phase 1: stream the value columns: A = dO V^T, dO S_u^T, V R_u^T
    float accA[4][4] = {}, accQ[4][NB] = {}, accK[4][NB] = {};
    for (int c0 = 0; c0 < DV; c0 += TW) {
        __syncthreads();
        for (int e = tid; e < BC * TW; e += NT) {
            const int t = e / TW, c = e % TW;
            const bool in = t < n;
            sDo[t * LS + c] = in ? bf(p.d_o, rv + static_cast<size_t>(t) * DV + c0 + c) : 0.f;
            sV[t * LS + c] = in ? bf(p.v, rv + static_cast<size_t>(t) * DV + c0 + c) : 0.f;
        }
        for (int e = tid; e < DK * TW; e += NT) {
            const int i = e / TW, c = e % TW;
            sS[i * LS + c] = Su[static_cast<size_t>(i) * DV + c0 + c];
            sR[i * LS + c] = Ru[static_cast<size_t>(i) * DV + c0 + c];
        }
        __syncthreads();
#pragma unroll 4
        for (int c = 0; c < TW; ++c) {
            float dr[4], vr[4], vj[4], sc[NB], rc[NB];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                dr[a] = sDo[(4 * ty + a) * LS + c];
                vr[a] = sV[(4 * ty + a) * LS + c];
                vj[a] = sV[(tx + 16 * a) * LS + c];
            }
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                sc[b] = sS[(tx + 16 * b) * LS + c];
                rc[b] = sR[(tx + 16 * b) * LS + c];
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
#pragma unroll
                for (int b = 0; b < 4; ++b) accA[a][b] = fmaf(dr[a], vj[b], accA[a][b]);
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    accQ[a][b] = fmaf(dr[a], sc[b], accQ[a][b]);
                    accK[a][b] = fmaf(vr[a], rc[b], accK[a][b]);
                }
            }
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int t = 4 * ty + a, j = tx + 16 * b;
            sAM[t * LA + j] = j <= t ? accA[a][b] : 0.f;
        }
    __syncthreads();

    // phase 2: dQ and dK (both owned as rows 4ty+a, channels tx+16b)
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int t = 4 * ty + a;
        float iq[NB] = {}, ik[NB] = {};
        if (!exact) {
            for (int j = 0; j <= t; ++j) {
                const float aij = sAM[t * LA + j];
#pragma unroll
                for (int b = 0; b < NB; ++b) iq[b] = fmaf(aij, sK[j * LD + tx + 16 * b], iq[b]);
            }
            for (int x = t; x < BC; ++x) {
                const float axt = sAM[x * LA + t];
#pragma unroll
                for (int b = 0; b < NB; ++b) ik[b] = fmaf(axt, sQ[x * LD + tx + 16 * b], ik[b]);
            }
        } else {
            for (int j = 0; j <= t; ++j) {
                const float aij = sAM[t * LA + j];
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const int i = tx + 16 * b;
                    iq[b] = fmaf(aij * sK[j * LD + i], exp2f(sG[t * LD + i] - sG[j * LD + i]), iq[b]);
                }
            }
            for (int x = t; x < BC; ++x) {
                const float axt = sAM[x * LA + t];
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const int i = tx + 16 * b;
                    ik[b] = fmaf(axt * sQ[x * LD + i], exp2f(sG[x * LD + i] - sG[t * LD + i]), ik[b]);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int i = tx + 16 * b;
            const float g = sG[t * LD + i];
            const float d = exact ? 0.f : g - sRef[i];
            const float dq = s * (exp2f(d) * iq[b] + exp2f(g) * accQ[a][b]);
            const float dk = s * exp2f(-d) * ik[b] + exp2f(sGC[i] - g) * accK[a][b];
            float pr = 0.f;
            if (t < n) {
                const size_t off = rk + static_cast<size_t>(t) * DK + i;
                p.gq[off] = __float2bfloat16_rn(dq);
                p.gk[off] = __float2bfloat16_rn(dk);
                pr = bf(p.q, off) * dq - bf(p.k, off) * dk;
            }
            sP[t * LD + i] = pr;
        }
    }
    __syncthreads();

    // phase 3: M = scale tril(Q K^T with the decay), over the A buffer
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int t = 4 * ty + a;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int j = tx + 16 * b;
            float m = 0.f;
            if (j <= t) {
                if (!exact) {
                    for (int i = 0; i < DK; ++i) m = fmaf(sQ[t * LD + i], sK[j * LD + i], m);
                } else {
                    for (int i = 0; i < DK; ++i)
                        m = fmaf(sQ[t * LD + i] * sK[j * LD + i],
                                 exp2f(sG[t * LD + i] - sG[j * LD + i]), m);
                }
            }
            accA[a][b] = s * m;
        }
    }
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) sAM[(4 * ty + a) * LA + tx + 16 * b] = accA[a][b];
    // keys for the state term of dV: k e^(Gamma_C - Gamma)
    for (int e = tid; e < BC * DK; e += NT) {
        const int t = e / DK, i = e % DK;
        const float f = exact ? exp2f(sGC[i] - sG[t * LD + i]) : exp2f(sGC[i] - sRef[i]);
        sK[t * LD + i] *= f;
    }

    // phase 4: dV = M^T dO + K' R_u, one slice of value columns at a time
    for (int c0 = 0; c0 < DV; c0 += TW) {
        __syncthreads();
        for (int e = tid; e < BC * TW; e += NT) {
            const int t = e / TW, c = e % TW;
            sDo[t * LS + c] = t < n ? bf(p.d_o, rv + static_cast<size_t>(t) * DV + c0 + c) : 0.f;
        }
        for (int e = tid; e < DK * TW; e += NT) {
            const int i = e / TW, c = e % TW;
            sR[i * LS + c] = Ru[static_cast<size_t>(i) * DV + c0 + c];
        }
        __syncthreads();
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int j = 4 * ty + a;
            float acc0 = 0.f, acc1 = 0.f;
            for (int x = j; x < BC; ++x) {
                const float mxj = sAM[x * LA + j];
                acc0 = fmaf(mxj, sDo[x * LS + tx], acc0);
                acc1 = fmaf(mxj, sDo[x * LS + tx + 16], acc1);
            }
            for (int i = 0; i < DK; ++i) {
                const float kji = sK[j * LD + i];
                acc0 = fmaf(kji, sR[i * LS + tx], acc0);
                acc1 = fmaf(kji, sR[i * LS + tx + 16], acc1);
            }
            if (j < n) {
                const size_t off = rv + static_cast<size_t>(j) * DV + c0;
                p.gv[off + tx] = __float2bfloat16_rn(acc0);
                p.gv[off + tx + 16] = __float2bfloat16_rn(acc1);
            }
        }
    }

    // phase 5: dlog_alpha = carry + reverse in-chunk sum of q dq - k dk
    if (tid < DK) {
        float acc = sCarry[tid];
        for (int t = n - 1; t >= 0; --t) {
            acc += sP[t * LD + tid];
            p.ga[rk + static_cast<size_t>(t) * DK + tid] = acc;
        }
    }
}

template <int DK, int DV>
int launch_bwd_dims(const BwdLaunch &p, cudaStream_t stream) {
    const size_t seq_bytes = sizeof(float) * (2 * BC * DK + BC * TW);
    const size_t grad_bytes = GradSmem<DK>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(bwd_states_kernel<DK, DV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(seq_bytes));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_adjoint_kernel<DK, DV>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(seq_bytes));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_grads_kernel<DK, DV>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(grad_bytes));
    if (e != cudaSuccess) return static_cast<int>(e);
    const dim3 tiles(DV / TW, p.BH), chunks(p.NC, p.BH);
    bwd_states_kernel<DK, DV><<<tiles, NT, seq_bytes, stream>>>(p);
    bwd_adjoint_kernel<DK, DV><<<tiles, NT, seq_bytes, stream>>>(p);
    bwd_grads_kernel<DK, DV><<<chunks, NT, grad_bytes, stream>>>(p);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace

int bwd_chunk_tokens() { return BC; }
int bwd_value_tiles(int dv) { return dv / TW; }

int launch_chunk_bwd(const BwdLaunch &p, cudaStream_t stream) {
    switch (p.dk * 1000 + p.dv) {
        case 64064: return launch_bwd_dims<64, 64>(p, stream);
        case 64128: return launch_bwd_dims<64, 128>(p, stream);
        case 64256: return launch_bwd_dims<64, 256>(p, stream);
        case 128064: return launch_bwd_dims<128, 64>(p, stream);
        case 128128: return launch_bwd_dims<128, 128>(p, stream);
        case 128256: return launch_bwd_dims<128, 256>(p, stream);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

}  // namespace gla
