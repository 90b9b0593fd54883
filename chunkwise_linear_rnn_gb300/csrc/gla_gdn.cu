// gla_gdn.cu — the gated delta rule (Gated DeltaNet) forward, token-recurrent.
//
// Per (batch, head) ("Qwen Team Releases FlashQLA for High-Performance Linear
// Attention" (todayforai.com), "Core Technical Principles", in the standard
// gated-delta-rule reading), with S in R^{dk x dv} and row vectors q, k, v:
//     S_t = alpha_t (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t
//     o_t = scale q_t S_t
// The transition mixes the rows of S and never its columns, so every value
// column evolves on its own.  A column's dk rows are split over dk/32 adjacent
// lanes, 32 rows each in registers (fp32); per token the lanes of a column form
// their part of k S[:, c], sum the parts with xor-shuffles, rewrite their rows
// and do the same for q S[:, c].  The CTA's four warps cover adjacent columns
// of one head and share its per-token q, k, v tile and gates, staged in shared
// memory 32 tokens at a time; each 32-row part of a staged q or k row is padded
// by four words so that the lanes of one column read different banks.  The
// next round's tokens are loaded into registers (16-byte loads) while the
// current round computes, so the staging barrier never waits on HBM.
//
// This is the first CUDA path of the workload: exact recurrence, no chunking,
// so it is bound by the per-token chain, not by HBM; the chunked form (the
// page's four steps on the tensor cores) is the next one.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gla.h"

namespace {

constexpr int kTok = 32;   // tokens staged per round
constexpr int kRows = 32;  // state rows one lane holds
constexpr int kPad = 4;    // words between the 32-row parts of a staged row
constexpr int kWarps = 4;

template <int DK>
struct GdnTile {
    static constexpr int kParts = DK / kRows;                 // lanes per column
    static constexpr int kCols = kWarps * 32 / kParts;        // columns per CTA
    static constexpr int kRow = kParts * (kRows + kPad);      // padded words per staged row
};

// One round of staged tokens in flight, held in registers: this thread's
// 16-byte pieces of the q, k and v tiles and (threads < kTok) one token's gates.
template <int DK>
struct GdnRound {
    static constexpr int kQ = kTok * DK / 8 / (kWarps * 32);                // q or k pieces
    static constexpr int kV = kTok * GdnTile<DK>::kCols / 8 / (kWarps * 32);  // v pieces
    uint4 q[kQ], k[kQ], v[kV];
    float g, b;
};

__device__ __forceinline__ void bf16x8_to_f32(uint4 u, float *f) {
    const unsigned w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // little-endian: the lower half holds the even element
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Loads tokens [t0, t0 + kTok) of one head (zeros past T).
template <int DK>
__device__ __forceinline__ void gdn_load_round(GdnRound<DK> &r, const __nv_bfloat16 *q,
                                               const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                                               const float *g, const float *beta, size_t rk,
                                               size_t rv, size_t rg, int c0, int t0, int T,
                                               int dv) {
    constexpr int NC = GdnTile<DK>::kCols;
    const int n = min(kTok, T - t0);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int j = 0; j < GdnRound<DK>::kQ; ++j) {
        const int i = threadIdx.x + j * kWarps * 32, t = i / (DK / 8), d0 = (i % (DK / 8)) * 8;
        const size_t off = rk + static_cast<size_t>(t0 + t) * DK + d0;
        r.q[j] = t < n ? *reinterpret_cast<const uint4 *>(q + off) : zero;
        r.k[j] = t < n ? *reinterpret_cast<const uint4 *>(k + off) : zero;
    }
#pragma unroll
    for (int j = 0; j < GdnRound<DK>::kV; ++j) {
        const int i = threadIdx.x + j * kWarps * 32, t = i / (NC / 8), j0 = (i % (NC / 8)) * 8;
        r.v[j] = t < n ? *reinterpret_cast<const uint4 *>(v + rv + static_cast<size_t>(t0 + t) * dv + c0 + j0)
                       : zero;
    }
    const bool gate = threadIdx.x < n;
    r.g = gate ? g[rg + t0 + threadIdx.x] : 0.f;
    r.b = gate ? beta[rg + t0 + threadIdx.x] : 0.f;
}

template <int DK>
__global__ void __launch_bounds__(kWarps * 32) gdn_recurrent_kernel(
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
    const __nv_bfloat16 *__restrict__ v, const float *__restrict__ g,
    const float *__restrict__ beta, float scale, const float *__restrict__ h0,
    __nv_bfloat16 *__restrict__ o, float *__restrict__ hT, int T, int dv) {
    using Tile = GdnTile<DK>;
    constexpr int P = Tile::kParts, NC = Tile::kCols, ROW = Tile::kRow;
    __shared__ __align__(16) float sq[kTok][ROW];
    __shared__ __align__(16) float sk[kTok][ROW];
    __shared__ __align__(16) float sv[kTok][NC];
    __shared__ float sa[kTok], sb[kTok];
    const int bh = blockIdx.y;
    const int cl = threadIdx.x / P, part = threadIdx.x % P;   // local column, row part
    const int c0 = blockIdx.x * NC, c = c0 + cl;              // c < dv: dv is a multiple of NC
    const int r0 = part * kRows, w0 = part * (kRows + kPad);  // first row, its staged word
    const size_t rk = static_cast<size_t>(bh) * T * DK, rv = static_cast<size_t>(bh) * T * dv;
    const unsigned full = 0xffffffffu;
    float S[kRows];
#pragma unroll
    for (int d = 0; d < kRows; ++d)
        S[d] = h0 ? h0[(static_cast<size_t>(bh) * DK + r0 + d) * dv + c] : 0.f;

    const size_t rg = static_cast<size_t>(bh) * T;
    GdnRound<DK> next;
    gdn_load_round<DK>(next, q, k, v, g, beta, rk, rv, rg, c0, 0, T, dv);
    for (int t0 = 0; t0 < T; t0 += kTok) {
        const int n = min(kTok, T - t0);
        __syncthreads();   // the previous round is done with the staged tokens
#pragma unroll
        for (int j = 0; j < GdnRound<DK>::kQ; ++j) {
            const int i = threadIdx.x + j * kWarps * 32, t = i / (DK / 8), d0 = (i % (DK / 8)) * 8;
            const int w = (d0 / kRows) * (kRows + kPad) + d0 % kRows;   // 8 words in one part
            float f[8];
            bf16x8_to_f32(next.q[j], f);
            *reinterpret_cast<float4 *>(&sq[t][w]) = make_float4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<float4 *>(&sq[t][w + 4]) = make_float4(f[4], f[5], f[6], f[7]);
            bf16x8_to_f32(next.k[j], f);
            *reinterpret_cast<float4 *>(&sk[t][w]) = make_float4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<float4 *>(&sk[t][w + 4]) = make_float4(f[4], f[5], f[6], f[7]);
        }
#pragma unroll
        for (int j = 0; j < GdnRound<DK>::kV; ++j) {
            const int i = threadIdx.x + j * kWarps * 32, t = i / (NC / 8), j0 = (i % (NC / 8)) * 8;
            float f[8];
            bf16x8_to_f32(next.v[j], f);
            *reinterpret_cast<float4 *>(&sv[t][j0]) = make_float4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<float4 *>(&sv[t][j0 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
        }
        if (threadIdx.x < kTok) {
            sa[threadIdx.x] = expf(next.g);   // e^0 = 1 past T
            sb[threadIdx.x] = next.b;
        }
        __syncthreads();
        if (t0 + kTok < T)   // the next round's loads stay in flight while this one computes
            gdn_load_round<DK>(next, q, k, v, g, beta, rk, rv, rg, c0, t0 + kTok, T, dv);
        for (int t = 0; t < n; ++t) {
            const float *kt = &sk[t][w0], *qt = &sq[t][w0];
            float ks0 = 0.f, ks1 = 0.f, ks2 = 0.f, ks3 = 0.f;   // this part of k S[:, c]
#pragma unroll
            for (int d = 0; d < kRows; d += 4) {
                ks0 = fmaf(kt[d], S[d], ks0);
                ks1 = fmaf(kt[d + 1], S[d + 1], ks1);
                ks2 = fmaf(kt[d + 2], S[d + 2], ks2);
                ks3 = fmaf(kt[d + 3], S[d + 3], ks3);
            }
            float ks = (ks0 + ks1) + (ks2 + ks3);
#pragma unroll
            for (int m = 1; m < P; m <<= 1) ks += __shfl_xor_sync(full, ks, m);
            const float alpha = sa[t];
            const float e = sb[t] * (sv[t][cl] - alpha * ks);   // the write error, scaled by beta
            float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
            for (int d = 0; d < kRows; d += 4) {
                // S = alpha S + k^T (beta (v - alpha k S)): the rule, rearranged
                S[d] = fmaf(alpha, S[d], kt[d] * e);
                S[d + 1] = fmaf(alpha, S[d + 1], kt[d + 1] * e);
                S[d + 2] = fmaf(alpha, S[d + 2], kt[d + 2] * e);
                S[d + 3] = fmaf(alpha, S[d + 3], kt[d + 3] * e);
                o0 = fmaf(qt[d], S[d], o0);
                o1 = fmaf(qt[d + 1], S[d + 1], o1);
                o2 = fmaf(qt[d + 2], S[d + 2], o2);
                o3 = fmaf(qt[d + 3], S[d + 3], o3);
            }
            float ot = (o0 + o1) + (o2 + o3);
#pragma unroll
            for (int m = 1; m < P; m <<= 1) ot += __shfl_xor_sync(full, ot, m);
            if (part == 0) o[rv + static_cast<size_t>(t0 + t) * dv + c] = __float2bfloat16_rn(scale * ot);
        }
    }
    if (hT) {
#pragma unroll
        for (int d = 0; d < kRows; ++d) hT[(static_cast<size_t>(bh) * DK + r0 + d) * dv + c] = S[d];
    }
}

bool misaligned(const void *p, uintptr_t b) { return (reinterpret_cast<uintptr_t>(p) & (b - 1)) != 0; }

}  // namespace

extern "C" int gla_gdn_fwd(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float scale, const float *h0, void *o, float *hT,
                           int B, int H, int T, int dk, int dv, cudaStream_t stream) {
    if (!q || !k || !v || !g || !beta || !o) return GLA_ERR_ARG;
    if (B <= 0 || H <= 0 || T <= 0 || H > 65535 || static_cast<long long>(B) * H > 65535)
        return GLA_ERR_ARG;
    if (!(dk == 64 || dk == 128) || !(dv == 64 || dv == 128 || dv == 256)) return GLA_ERR_SHAPE;
    if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 2) ||
        misaligned(g, 4) || misaligned(beta, 4) || (h0 && misaligned(h0, 4)) ||
        (hT && misaligned(hT, 4)))
        return GLA_ERR_ARG;
    int dev = -1, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_DEVICE;
    }
    if (major != 10 || minor != 3) return GLA_ERR_DEVICE;
    const int cols = dk == 64 ? GdnTile<64>::kCols : GdnTile<128>::kCols;
    if (dv % cols) return GLA_ERR_SHAPE;
    const dim3 grid(dv / cols, B * H), block(kWarps * 32);
    const auto *qb = static_cast<const __nv_bfloat16 *>(q);
    const auto *kb = static_cast<const __nv_bfloat16 *>(k);
    const auto *vb = static_cast<const __nv_bfloat16 *>(v);
    auto *ob = static_cast<__nv_bfloat16 *>(o);
    if (dk == 64)
        gdn_recurrent_kernel<64><<<grid, block, 0, stream>>>(qb, kb, vb, g, beta, scale, h0, ob, hT, T, dv);
    else
        gdn_recurrent_kernel<128><<<grid, block, 0, stream>>>(qb, kb, vb, g, beta, scale, h0, ob, hT, T, dv);
    return cudaGetLastError() == cudaSuccess ? GLA_OK : GLA_ERR_LAUNCH;
}
