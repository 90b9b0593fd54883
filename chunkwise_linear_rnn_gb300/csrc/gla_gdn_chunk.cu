// gla_gdn_chunk.cu — the gated delta rule (Gated DeltaNet) forward by chunks on
// the tensor cores: the four-step chunk algorithm of "Qwen Team Releases
// FlashQLA for High-Performance Linear Attention" (todayforai.com), "Core
// Technical Principles", in the standard gated-delta-rule reading
//     S_t = alpha_t (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t,
//     o_t = scale q_t S_t,
// with chunks of C = 64 tokens, gamma_t the in-chunk product of the gates
// (G = log2 gamma, prefix sums in log2 units) and the chunk's write errors D:
//   1. T = (I + L)^-1, L strictly lower, L_ti = beta_t (gamma_t / gamma_i) k_t.k_i;
//   2. W = T diag(beta gamma) K,  U = T diag(beta) V;
//   3. S_C = gamma_C S_0 + (diag(gamma_C / gamma) K)^T D,  D = U - W S_0;
//   4. O = scale (diag(gamma) Q S_0 + tril(Q K^T gamma_t / gamma_i) D).
//
// Two kernels, split as the page splits its operators (an inversion operator,
// then one fused operator for the rest):
//   gdn_wy_kernel   one CTA per (chunk, head), three CTAs per SM: step 1 and W.
//                   K K^T on the tensor cores; the unit lower triangular
//                   inverse by 16 x 16 blocks (each diagonal block by
//                   substitution in the warp that formed its rows of L, then
//                   two merge levels of small products); to scratch, bf16,
//                   2 dk + 128 bytes per token: W = (T diag(beta gamma)) K and
//                   (T - I) diag(beta), the off-diagonal part of U's factor.
//   gdn_seq_kernel  one CTA per (head, 64-column value tile), chunks in order,
//                   the state's 128 key rows in the registers of warps 0-3
//                   (one row per thread); each chunk's operands loaded by TMA
//                   one chunk ahead into the other of two stages; steps 3-4 as
//                   tensor-core products W S, (T - I) diag(beta) V, Q K^T, Q S,
//                   K^T D' and P D, with D' = diag(gamma_C / gamma) D.
//
// Precision: bf16 operands with fp32 accumulation.  The operands whose
// rounding would enter every later state (T diag(beta gamma) in W, S, D, D',
// P) are bf16 hi/lo pairs (16 significant bits); the stored W and
// (T - I) diag(beta) are single bf16, and U's diagonal term beta_t v_t is
// added exactly in fp32.  K and V enter as the exact bf16 inputs.  o is
// rounded once to bf16; the state and hT are fp32.
//
// Every mbarrier wait is bounded (the library's limit); an expired wait sets
// the status word and the CTA stops at the next chunk boundary.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gla.h"
#include "gla_internal.h"
#include "gla_ptx.cuh"

namespace gla {
namespace {

constexpr int C = 64;             // tokens per chunk
constexpr int NT = 256;           // threads per CTA (both kernels)
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void split_pair(float x, float y, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ uint32_t pack_bf16(float x, float y) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Inclusive prefix sum of one chunk's log-gates in log2 units (rows past n
// are zero, so the sum stays flat there) and the chunk's beta; warp 0.
__device__ __forceinline__ void chunk_gates(float *sG, float *sB, const float *g, const float *beta,
                                            size_t r0, int n) {
    if (threadIdx.x < 32) {
        const int l = threadIdx.x;
        float a = l < n ? g[r0 + l] * kLog2e : 0.f, b = l + 32 < n ? g[r0 + l + 32] * kLog2e : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o);
            if (l >= o) { a += ya; b += yb; }
        }
        b += __shfl_sync(0xffffffffu, a, 31);
        sG[l] = a;
        sG[l + 32] = b;
        sB[l] = l < n ? beta[r0 + l] : 0.f;
        sB[l + 32] = l + 32 < n ? beta[r0 + l + 32] : 0.f;
    }
}

// ------------------------------------------------------------------ WY pre-pass
struct WySmem {
    static constexpr int DK = 128;
    static constexpr int LS = 68;                                // fp32 row stride (16-byte rows)
    static constexpr uint32_t kBlk = C * 128;                    // 64 rows x 64 bf16
    static constexpr uint32_t kK = 0;                            // K [t][c] (2 channel blocks)
    static constexpr uint32_t kTh = kK + 2 * kBlk;               // T diag(beta gamma) [t][i] K-major, hi
    static constexpr uint32_t kTl = kTh + kBlk;                  // and lo
    static constexpr uint32_t kL = kTl + kBlk;                   // fp32 [64][LS]: L
    static constexpr uint32_t kTf = kL + C * LS * 4;             // fp32 [64][LS]: T
    static constexpr uint32_t kX = kTf + C * LS * 4;             // merge products, up to [32][32]
    static constexpr uint32_t kG = kX + 32 * 32 * 4;
    static constexpr uint32_t kBeta = kG + C * 4;
    static constexpr uint32_t kE = kBeta + C * 4;                // 2^-G per token
    static constexpr uint32_t kBar = kE + C * 4;
    static constexpr uint32_t kSlot = kBar + 16;
    static constexpr uint32_t kBytes = kSlot + 16 + 1024;
    static_assert(kBytes <= 75 * 1024, "three CTAs per SM");
};

// The diagonal 16 x 16 block o..o+15 of T = (I + L)^-1 by substitution:
// column j per thread (lanes 0-15 of the warp whose TMEM quarter holds those
// rows of L), in registers; x_i = -sum_{m<i} L_im x_m below the unit diagonal.
__device__ __forceinline__ void invert_diagonal_block(const float *sL, float *sTf, int o, int j) {
    constexpr int LS = WySmem::LS;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = i == j ? 1.f : 0.f;
#pragma unroll
    for (int i = 1; i < 16; ++i) {
        const float *row = sL + (o + i) * LS + o;
        float acc = 0.f;
#pragma unroll
        for (int m4 = 0; m4 < i; m4 += 4) {
            const float4 l4 = *reinterpret_cast<const float4 *>(row + m4);
            acc = fmaf(l4.x, x[m4], acc);
            if (m4 + 1 < i) acc = fmaf(l4.y, x[m4 + 1], acc);
            if (m4 + 2 < i) acc = fmaf(l4.z, x[m4 + 2], acc);
            if (m4 + 3 < i) acc = fmaf(l4.w, x[m4 + 3], acc);
        }
        if (i > j) x[i] = -acc;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) sTf[(o + i) * LS + o + j] = x[i];
}

// The rest of T = (I + L)^-1 (64 x 64 fp32, row stride LS) once its four
// diagonal 16 x 16 blocks are in sTf: merge pairs of blocks, then the halves,
// each as T_ba = -T_bb (L_ba T_aa) with T_aa, T_bb lower triangular (inverse
// of a block lower-triangular matrix).  Four output columns per thread,
// 16-byte shared-memory loads.  Only the blocks on and below the diagonal of
// sTf are written.  Needs NT == 256.
__device__ __forceinline__ void merge_inverse_blocks(const float *sL, float *sTf, float *sX) {
    static_assert(NT == 256, "four-column strips of a 32 x 32 block per thread");
    constexpr int LS = WySmem::LS;
    const int tid = threadIdx.x;
    // 16 x 16 merges: (rows 16-31, cols 0-15) and (rows 48-63, cols 32-47);
    // threads 0-127: block p = tid / 64, row r, columns c4..c4+3
    {
        const int pb = tid >> 6, r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
        const int a = 32 * pb, bb = a + 16;   // T_aa at (a, a), T_bb at (bb, bb)
        if (tid < 128) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            const float *lrow = sL + (bb + r) * LS + a;
#pragma unroll
            for (int m = 0; m < 16; m += 4) {
                const float4 l4 = *reinterpret_cast<const float4 *>(lrow + m);
                const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(sTf + (a + m + e) * LS + a + c4);
                    acc.x = fmaf(lv[e], t4.x, acc.x);
                    acc.y = fmaf(lv[e], t4.y, acc.y);
                    acc.z = fmaf(lv[e], t4.z, acc.z);
                    acc.w = fmaf(lv[e], t4.w, acc.w);
                }
            }
            *reinterpret_cast<float4 *>(sX + pb * 256 + r * 16 + c4) = acc;
        }
        __syncthreads();
        if (tid < 128) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            const float *trow = sTf + (bb + r) * LS + bb;
#pragma unroll
            for (int m = 0; m < 16; m += 4) {
                const float4 t4 = *reinterpret_cast<const float4 *>(trow + m);
                const float tv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 x4 = *reinterpret_cast<const float4 *>(sX + pb * 256 + (m + e) * 16 + c4);
                    acc.x = fmaf(tv[e], x4.x, acc.x);
                    acc.y = fmaf(tv[e], x4.y, acc.y);
                    acc.z = fmaf(tv[e], x4.z, acc.z);
                    acc.w = fmaf(tv[e], x4.w, acc.w);
                }
            }
            *reinterpret_cast<float4 *>(sTf + (bb + r) * LS + a + c4) =
                make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        __syncthreads();
    }
    // 32 x 32 merge: rows 32-63, cols 0-31; thread = row r, columns c4..c4+3.
    // T_A (rows, cols 0-31) and T_B (rows, cols 32-63) are lower triangular,
    // so X = L_BA T_A sums m >= c and T_B X sums m <= r; the loops still run
    // over all 32 (the zero entries above the diagonal blocks were never
    // written, so they are skipped by block: m-blocks of 16 below c's block
    // and above r's block contribute nothing).
    {
        const int r = tid >> 3, c4 = (tid & 7) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float *lrow = sL + (32 + r) * LS;
        for (int m = (c4 >> 4) * 16; m < 32; m += 4) {
            const float4 l4 = *reinterpret_cast<const float4 *>(lrow + m);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 t4 = *reinterpret_cast<const float4 *>(sTf + (m + e) * LS + c4);
                acc.x = fmaf(lv[e], t4.x, acc.x);
                acc.y = fmaf(lv[e], t4.y, acc.y);
                acc.z = fmaf(lv[e], t4.z, acc.z);
                acc.w = fmaf(lv[e], t4.w, acc.w);
            }
        }
        *reinterpret_cast<float4 *>(sX + r * 32 + c4) = acc;
        __syncthreads();
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float *trow = sTf + (32 + r) * LS + 32;
        const int mend = (r >> 4) * 16 + 16;
        for (int m = 0; m < mend; m += 4) {
            const float4 t4 = *reinterpret_cast<const float4 *>(trow + m);
            const float tv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 x4 = *reinterpret_cast<const float4 *>(sX + (m + e) * 32 + c4);
                acc.x = fmaf(tv[e], x4.x, acc.x);
                acc.y = fmaf(tv[e], x4.y, acc.y);
                acc.z = fmaf(tv[e], x4.z, acc.z);
                acc.w = fmaf(tv[e], x4.w, acc.w);
            }
        }
        *reinterpret_cast<float4 *>(sTf + (32 + r) * LS + c4) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        __syncthreads();
    }
}

// Grid (chunks per head, B*H), three CTAs per SM.  Per chunk: L from K K^T
// (tensor cores), T = (I + L)^-1, then
//   Tout = (T - I) diag(beta) (bf16, [BH][nch*C][64]): the off-diagonal part
//          of T diag(beta), for U = beta v + (T - I) diag(beta) V;
//   Wout = T diag(beta gamma) K (bf16, [BH][nch*C][DK]), from T diag(beta
//          gamma) as a hi/lo pair times the raw K tile (tensor cores).
template <int DK>
__global__ void __launch_bounds__(NT, 3) gdn_wy_kernel(
    const __nv_bfloat16 *__restrict__ k, const float *__restrict__ g,
    const float *__restrict__ beta, __nv_bfloat16 *__restrict__ Wout,
    __nv_bfloat16 *__restrict__ Tout, int T, unsigned int *status) {
    static_assert(DK == WySmem::DK, "dk = 128");
    using L = WySmem;
    constexpr int LS = L::LS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *sL = reinterpret_cast<float *>(sm + L::kL), *sTf = reinterpret_cast<float *>(sm + L::kTf);
    float *sG = reinterpret_cast<float *>(sm + L::kG), *sB = reinterpret_cast<float *>(sm + L::kBeta);
    float *sE = reinterpret_cast<float *>(sm + L::kE);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::kBar);
    uint32_t *slot = reinterpret_cast<uint32_t *>(sm + L::kSlot);
    const int u = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = (T + C - 1) / C, t0 = u * C, n = min(C, T - t0);
    const size_t rg = static_cast<size_t>(bh) * T + t0;
    const size_t rk = rg * DK;
    const size_t orow = (static_cast<size_t>(bh) * nch + u) * C;   // first scratch row

    if (warp == 0) tmem_alloc(slot, 128);   // K K^T, then W over it: four CTAs' worth per SM
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    chunk_gates(sG, sB, g, beta, rg, n);
    // K as bf16 [t][c] K-major (exact input; rows past n zero)
    constexpr int KPER = C * DK / 8 / NT;
#pragma unroll
    for (int m = 0; m < KPER; ++m) {
        const int e = tid + m * NT, t = e / (DK / 8), c = (e % (DK / 8)) * 8;
        const uint4 kr = t < n ? *reinterpret_cast<const uint4 *>(k + rk + static_cast<size_t>(t) * DK + c)
                               : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(sm + L::kK + sw128_offset(t, c, L::kBlk)) = kr;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot, a0 = smem_u32(sm);

    // K K^T: M = 64 (t), N = 64 (i), K = DK; both operands K-major
    if (tid == 0) {
        constexpr uint32_t id = idesc_bf16(64, C, false, false);
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
            const uint32_t o = (kk >> 2) * L::kBlk + (kk & 3) * 32;
            const uint64_t d = sw128_desc(a0 + L::kK + o, 16, 1024);
            mma_bf16_ss(tmem, d, d, id, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar[0]);
    }
    // 2^(G_t - G_i) = 2^G_t 2^-G_i while the chunk's total decay keeps 2^-G_i
    // within 2^60 (G falls over the chunk); else one exponential per element
    const bool split_exp = sG[C - 1] >= -60.f;
    if (split_exp && tid < C) sE[tid] = exp2f(-sG[tid]);
    bool ok = mbar_wait_bounded(&bar[0], 0, status);
    tc_fence_after();
    __syncthreads();   // sE
    // L_ti = beta_t 2^(G_t - G_i) (k_t . k_i) for i < t: warps 0-3, row
    // t = 16 q + (lane & 15), 16 columns per half-split load; then each of
    // these warps inverts the diagonal block of its own 16 rows
    if (warp < 4) {
        const int t = 16 * warp + (lane & 15), hc = (lane >> 4) * 16;
        const float Gt = sG[t], bt = sB[t], rt = bt * exp2f(Gt);
#pragma unroll 1
        for (int ib = 0; ib < C; ib += 32) {
            uint32_t r[16];
            tmem_ld16x2<16>(tmem + (static_cast<uint32_t>(32 * warp) << 16) + ib, r);
            tmem_wait_ld();
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int i = ib + hc + j;
                const float f = split_exp ? rt * sE[i] : bt * exp2f(Gt - sG[i]);
                v[j] = (ok && i < t) ? f * __uint_as_float(r[j]) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4 *>(sL + t * LS + ib + hc + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
        __syncwarp();
        if (lane < 16) invert_diagonal_block(sL, sTf, 16 * warp, lane);
    }
    tc_fence_before();   // K K^T is read: W may take its columns
    __syncthreads();
    merge_inverse_blocks(sL, sTf, reinterpret_cast<float *>(sm + L::kX));
    // T diag(beta gamma) as a hi/lo pair, K-major [t][i] (A of W), and
    // (T - I) diag(beta) row-major to the scratch
    __nv_bfloat16 *tdst = Tout + orow * C;
#pragma unroll
    for (int m = 0; m < C * C / 8 / NT; ++m) {
        const int e = tid + m * NT, t = e / (C / 8), i0 = (e % (C / 8)) * 8;
        uint32_t hi[4], lo[4], tb[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int i = i0 + 2 * x;
            // blocks above the diagonal were never written: zero there
            const bool low0 = (i >> 4) <= (t >> 4), low1 = ((i + 1) >> 4) <= (t >> 4);
            const float x0 = low0 ? sTf[t * LS + i] : 0.f, x1 = low1 ? sTf[t * LS + i + 1] : 0.f;
            split_pair(x0 * sB[i] * exp2f(sG[i]), x1 * sB[i + 1] * exp2f(sG[i + 1]), hi[x], lo[x]);
            tb[x] = pack_bf16(i == t ? 0.f : x0 * sB[i], i + 1 == t ? 0.f : x1 * sB[i + 1]);
        }
        const uint32_t off = sw128_offset(t, i0, L::kBlk);
        *reinterpret_cast<uint4 *>(sm + L::kTh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(sm + L::kTl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        if (ok) *reinterpret_cast<uint4 *>(tdst + t * C + i0) = make_uint4(tb[0], tb[1], tb[2], tb[3]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // W = (T diag(beta gamma)) K: M = 64, N = DK (two 64-channel blocks of
    // the K tile, MN-major), K = 64 tokens; hi and lo of the left factor
    if (tid == 0) {
        constexpr uint32_t idw = idesc_bf16(64, DK, false, true);
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk) {
            const uint64_t bk = sw128_desc(a0 + L::kK + kk * 2048, L::kBlk, 1024);
            mma_bf16_ss(tmem, sw128_desc(a0 + L::kTh + kk * 32, 16, 1024), bk, idw, kk > 0 ? 1u : 0u);
            mma_bf16_ss(tmem, sw128_desc(a0 + L::kTl + kk * 32, 16, 1024), bk, idw, 1u);
        }
        mma_commit(&bar[1]);
    }
    ok = mbar_wait_bounded(&bar[1], 0, status) && ok;
    tc_fence_after();
    // epilogue: warps 0-3 store W (bf16), row t, 16 columns per half-split load
    if (warp < 4) {
        const int t = 16 * warp + (lane & 15), hc = (lane >> 4) * 16;
        const uint32_t lo_ = static_cast<uint32_t>(32 * warp) << 16;
#pragma unroll 1
        for (int cb = 0; cb < DK; cb += 32) {
            uint32_t r[16];
            tmem_ld16x2<16>(tmem + lo_ + cb, r);
            tmem_wait_ld();
            if (ok) {
                __nv_bfloat16 *dst = Wout + (orow + t) * DK + cb + hc;
#pragma unroll
                for (int j = 0; j < 16; j += 8)
                    *reinterpret_cast<uint4 *>(dst + j) = make_uint4(
                        pack_bf16(__uint_as_float(r[j]), __uint_as_float(r[j + 1])),
                        pack_bf16(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3])),
                        pack_bf16(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5])),
                        pack_bf16(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7])));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ------------------------------------------------------------------ sequential chunk kernel
struct SeqSmem {
    static constexpr int DK = 128;
    static constexpr uint32_t kBlk = C * 128;       // 64 rows x 64 bf16
    static constexpr uint32_t kSBlk = DK * 128;     // 128 rows x 64 bf16
    // the loaded operands of one chunk (a stage; two stages, chunk u in u & 1)
    static constexpr uint32_t kQ = 0;               // Q [t][c] K-major (2 blocks)
    static constexpr uint32_t kK = kQ + 2 * kBlk;   // K [t][c]: B of Q K^T (K-major), A of K^T D' (MN-major)
    static constexpr uint32_t kW = kK + 2 * kBlk;   // W [t][c] K-major
    static constexpr uint32_t kT = kW + 2 * kBlk;   // (T - I) diag(beta) [t][i] K-major
    static constexpr uint32_t kV = kT + kBlk;       // V of this tile [i][c]: B of U (MN-major)
    static constexpr uint32_t kStage = kV + kBlk;
    static constexpr uint32_t kSh = 2 * kStage;     // S [i][c] MN-major (B), hi and lo
    static constexpr uint32_t kSl = kSh + kSBlk;
    static constexpr uint32_t kPh = kSl + kSBlk;    // P [t][i] K-major, hi and lo
    static constexpr uint32_t kPl = kPh + kBlk;
    static constexpr uint32_t kDh = kPl + kBlk;     // D [t][c] MN-major (B of P D), hi and lo
    static constexpr uint32_t kDl = kDh + kBlk;
    static constexpr uint32_t kEh = kDl + kBlk;     // D' = diag(2^(G_C - G)) D (B of K^T D'), hi and lo
    static constexpr uint32_t kEl = kEh + kBlk;
    static constexpr uint32_t kG = kEl + kBlk;      // G of chunk u in [u & 1]
    static constexpr uint32_t kBeta = kG + 2 * C * 4;   // beta of chunk u in [u & 1]
    static constexpr uint32_t kE = kBeta + 2 * C * 4;   // 2^-G per token (the scores' column factors)
    static constexpr uint32_t kBar = kE + C * 4;    // the kernel's mbarriers (SeqBar)
    static constexpr uint32_t kSlot = kBar + 128;
    static constexpr uint32_t kBytes = kSlot + 16 + 1024;
    static constexpr uint32_t kLoadBytes = kStage;
};
static_assert(SeqSmem::kBytes <= 227 * 1024, "shared memory of one CTA");

// The sequential kernel's operands: tensor maps of q, k, v ([BH, T, .] as
// (channel, token, head)), W ([rows, 128]) and (T - I) diag(beta) ([rows, 64]),
// 64 x 64 boxes with the 128-byte swizzle; rows past T load as zeros.
struct SeqParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_w, tm_t;
    const float *g, *beta, *h0;
    __nv_bfloat16 *o;
    float *hT;
    float scale;
    int T;
    unsigned int *status;
};

// Inclusive prefix sum (log2 units) of one chunk's log-gates into sG and its
// betas into sB (rows past n are zero, so the sum stays flat there); one warp.
__device__ __forceinline__ void gates_scan(const float *g, const float *beta, size_t r0, int n,
                                           float *sG, float *sB) {
    const int l = threadIdx.x & 31;
    sB[l] = l < n ? beta[r0 + l] : 0.f;
    sB[l + 32] = l + 32 < n ? beta[r0 + l + 32] : 0.f;
    float a = l < n ? g[r0 + l] * kLog2e : 0.f, b = l + 32 < n ? g[r0 + l + 32] * kLog2e : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o);
        if (l >= o) { a += ya; b += yb; }
    }
    b += __shfl_sync(0xffffffffu, a, 31);
    sG[l] = a;
    sG[l + 32] = b;
}

// The TMA loads of chunk u of head bh into stage u & 1: Q, K and W (two
// 64-channel blocks each), (T - I) diag(beta), and the tile's 64 columns of V; one
// thread.
__device__ __forceinline__ void chunk_loads(const SeqParams &p, uint8_t *sm, uint64_t *bar, int u,
                                            int bh, int c0, int nch) {
    using L = SeqSmem;
    uint8_t *st = sm + (u & 1) * L::kStage;
    const int t0 = u * C;
    const int orow = (bh * nch + u) * C;
    mbar_arrive_expect_tx(bar, L::kLoadBytes);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
        tma_load_3d(st + L::kQ + kb * L::kBlk, &p.tm_q, bar, kb * 64, t0, bh);
        tma_load_3d(st + L::kK + kb * L::kBlk, &p.tm_k, bar, kb * 64, t0, bh);
        tma_load_3d(st + L::kW + kb * L::kBlk, &p.tm_w, bar, kb * 64, orow, 0);
    }
    tma_load_3d(st + L::kT, &p.tm_t, bar, 0, orow, 0);
    tma_load_3d(st + L::kV, &p.tm_v, bar, c0, t0, bh);
}

// Grid (DV / 64, B*H); dk = 128.  W and (T - I) diag(beta) from gdn_wy_kernel.
// 320 threads:
//   warps 0-3 "state": thread i holds key row i of the state (this tile's 64
//     columns, fp32 registers); they form the masked scores P from Q K^T
//     while the state chain runs, then apply the state update from K^T D'
//     and write the updated state's bf16 hi/lo copy;
//   warps 4-7 "token": the write errors D = U - W S (and D' = D scaled by
//     the decay to the chunk's end), then the outputs;
//   warp 8 "issue": lane 0 issues every product;
//   warp 9 "load": lane 0 issues the next chunk's TMA loads into the other
//     stage as the chunk begins; the warp scans the next chunk's gates.
// Per chunk: (T - I) diag(beta) V and W S (commit A1), Q K^T (commit QK),
// Q S (commit A2); K^T D' once D is written (commit B1); P D once P is
// written (commit B2).  Only the state chain W S -> D -> K^T D' -> S is
// serial; the scores, P D and the outputs run beside it.  beta rides on T
// (its exact diagonal term beta_t v_t is added in fp32 where D is formed) and
// the decay to the chunk's end on D', so the raw bf16 tiles of K and V are
// the operands as loaded.  The M = 64 products (token rows in lanes 0-15 of each
// lane quarter) are read with the half-split TMEM load, so that all 32
// threads of a warp take part in their epilogues.
constexpr int NTS = 320;
enum SeqBar { kSbA1 = 0, kSbQK, kSbA2, kSbB1, kSbB2, kSbD, kSbP, kSbLd0, kSbLd1, kSbDrain, kSbDrain2, kSbCount };
static_assert(kSbCount * 8 <= 128, "mbarrier space of SeqSmem");

template <int DV>
__global__ void __launch_bounds__(NTS, 1) gdn_seq_kernel(const __grid_constant__ SeqParams p) {
    using L = SeqSmem;
    const float *__restrict__ g = p.g;
    const float *__restrict__ beta = p.beta;
    const float *__restrict__ h0 = p.h0;
    __nv_bfloat16 *__restrict__ o = p.o;
    float *__restrict__ hT = p.hT;
    const float scale = p.scale;
    const int T = p.T;
    unsigned int *status = p.status;
    constexpr int DK = L::DK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *sGb = reinterpret_cast<float *>(sm + L::kG), *sBb = reinterpret_cast<float *>(sm + L::kBeta);
    float *sE = reinterpret_cast<float *>(sm + L::kE);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::kBar);
    uint32_t *slot = reinterpret_cast<uint32_t *>(sm + L::kSlot);
    const int c0 = blockIdx.x * 64, bh = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = (T + C - 1) / C;
    const int q4 = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;

    if (warp == 0) tmem_alloc(slot, 512);
    if (tid == 0) {
        for (int i = 0; i < kSbCount; ++i) mbar_init(&bar[i], (i == kSbD || i == kSbP) ? 4u : 1u);
        fence_mbar_init();
        prefetch_tensormap(&p.tm_q);
        prefetch_tensormap(&p.tm_k);
        prefetch_tensormap(&p.tm_v);
        prefetch_tensormap(&p.tm_w);
        prefetch_tensormap(&p.tm_t);
    }
    // warps 0-3: thread = key row i, the 64 columns of this tile
    float S[64];
    const int i_row = tid;   // meaningful for tid < 128
    if (warp < 4) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
            S[c] = h0 ? h0[(static_cast<size_t>(bh) * DK + i_row) * DV + c0 + c] : 0.f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot, a0 = smem_u32(sm);
    bool ok = true;
    // the state entering a chunk as a hi/lo pair [i][c] (the B operand of W S
    // and Q S): written here for the first chunk, then by the state warps right
    // after each update, once both products of the chunk have read it
    auto state_copy = [&]() {
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) split_pair(S[c + 2 * j], S[c + 2 * j + 1], hi[j], lo[j]);
            const uint32_t so = sw128_offset(i_row, c, L::kSBlk);
            *reinterpret_cast<uint4 *>(sm + L::kSh + so) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(sm + L::kSl + so) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    };
    if (warp < 4) state_copy();
    int loads = 0;  // warp 9 lane 0: chunks whose loads are issued
    if (warp == 9) {
        gates_scan(g, beta, static_cast<size_t>(bh) * T, min(C, T), sGb, sBb);
        if (lane == 0) {
            chunk_loads(p, sm, &bar[kSbLd0], 0, bh, c0, nch);
            loads = 1;
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();   // the state copy and the first chunk's gates
    tc_fence_after();

#pragma unroll 1
    for (int u = 0; u < nch; ++u) {
        const int t0 = u * C, n = min(C, T - t0);
        const size_t rg = static_cast<size_t>(bh) * T + t0;
        const uint32_t ph = static_cast<uint32_t>(u & 1);
        const float *sG = sGb + (u & 1) * C;
        const float GC = sG[C - 1];
        const uint32_t st = a0 + (u & 1) * L::kStage;   // this chunk's stage
        // 2^(G_t - G_i) = 2^G_t 2^-G_i for the scores: one exponential per row
        // and a column table, while the chunk's total decay keeps 2^-G_i within
        // 2^60 (G falls monotonically over the chunk); else one exponential
        // per element
        const bool split_exp = GC >= -60.f;
        if (warp == 9) {
            // ======================================================= load warp
            // lane 0 issues the products of the output side, Q K^T (TMEM
            // 256-319) and Q [Sh|Sl] (TMEM 128-255), beside the issue warp's
            // state chain; then the next chunk's operands into the other
            // stage (every read of it ended with the previous chunk); the
            // warp scans the next chunk's gates
            if (lane == 0) {
                ok = mbar_wait_bounded(&bar[kSbLd0 + (u & 1)], static_cast<uint32_t>((u >> 1) & 1),
                                       status) && ok;
                tc_fence_after();
                constexpr uint32_t id_p = idesc_bf16(64, C, false, false);     // Q [t][c], K [i][c]
                constexpr uint32_t id_s2 = idesc_bf16(64, 128, false, true);   // Q [t][c], [Sh|Sl] MN-major
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t ok_ = (kk >> 2) * L::kBlk + (kk & 3) * 32;
                    mma_bf16_ss(tmem + 256, sw128_desc(st + L::kQ + ok_, 16, 1024),
                                sw128_desc(st + L::kK + ok_, 16, 1024), id_p, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bar[kSbQK]);
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t ok_ = (kk >> 2) * L::kBlk + (kk & 3) * 32;
                    mma_bf16_ss(tmem + 128, sw128_desc(st + L::kQ + ok_, 16, 1024),
                                sw128_desc(a0 + L::kSh + kk * 2048, L::kSBlk, 1024), id_s2,
                                kk > 0 ? 1u : 0u);
                }
                mma_commit(&bar[kSbA2]);
                if (u + 1 < nch) {
                    chunk_loads(p, sm, &bar[kSbLd0 + ((u + 1) & 1)], u + 1, bh, c0, nch);
                    loads = u + 2;
                }
            }
            __syncwarp();
            if (u + 1 < nch)
                gates_scan(g, beta, rg + C, min(C, T - t0 - C), sGb + ((u + 1) & 1) * C,
                           sBb + ((u + 1) & 1) * C);
        } else if (warp == 8) {
            // ======================================================= issue warp
            if (lane == 0) {
                ok = mbar_wait_bounded(&bar[kSbLd0 + (u & 1)], static_cast<uint32_t>((u >> 1) & 1),
                                       status) && ok;
                tc_fence_after();
                constexpr uint32_t id_u = idesc_bf16(64, 64, false, true);    // T [t][i], V [i][c]
                // TMEM columns: W [Sh|Sl] 0-127, Q [Sh|Sl] 128-255, Q K^T
                // 256-319, (T - I) diag(beta) V 320-383, K^T [D'h|D'l] 384-511
                // (M = 128); once D is formed, Ph [Dh|Dl] into 0-127 and Pl Dh
                // into 320-383.  A split operand's hi and lo halves sit side by
                // side as one N = 128 operand (their sum is taken where the
                // product is read): one instruction per 16-deep step for both.
                constexpr uint32_t id_s2 = idesc_bf16(64, 128, false, true);   // A [t][c] K-major, [Sh|Sl] MN-major
                // A1: W S and (T - I) diag(beta) V, the state chain's first step
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t ok_ = (kk >> 2) * L::kBlk + (kk & 3) * 32;
                    const uint32_t acc = kk > 0 ? 1u : 0u;
                    mma_bf16_ss(tmem, sw128_desc(st + L::kW + ok_, 16, 1024),
                                sw128_desc(a0 + L::kSh + kk * 2048, L::kSBlk, 1024), id_s2, acc);
                    if (kk < C / 16)
                        mma_bf16_ss(tmem + 320, sw128_desc(st + L::kT + kk * 32, 16, 1024),
                                    sw128_desc(st + L::kV + kk * 2048, L::kBlk, 1024), id_u, acc);
                }
                mma_commit(&bar[kSbA1]);
                // B1: K^T D' (M = 128 channels) once D' is written
                constexpr uint32_t id_kd = idesc_bf16(128, 128, true, true);   // K [t][c] MN-major, [D'h|D'l] MN-major
                ok = mbar_wait_bounded(&bar[kSbD], ph, status) && ok;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_bf16_ss(tmem + 384, sw128_desc(st + L::kK + kk * 2048, L::kBlk, 1024),
                                sw128_desc(a0 + L::kEh + kk * 2048, L::kBlk, 1024), id_kd,
                                kk > 0 ? 1u : 0u);
                mma_commit(&bar[kSbB1]);
                // B2: P D (K = 64 tokens) once P is written; W S and U were
                // read into D by then
                constexpr uint32_t id_pd2 = idesc_bf16(64, 128, false, true);  // P [t][i] K-major, [Dh|Dl] MN-major
                constexpr uint32_t id_pd = idesc_bf16(64, 64, false, true);
                ok = mbar_wait_bounded(&bar[kSbP], ph, status) && ok;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < C / 16; ++kk) {
                    const uint64_t dh = sw128_desc(a0 + L::kDh + kk * 2048, L::kBlk, 1024);
                    const uint32_t acc = kk > 0 ? 1u : 0u;
                    mma_bf16_ss(tmem, sw128_desc(a0 + L::kPh + kk * 32, 16, 1024), dh, id_pd2, acc);
                    mma_bf16_ss(tmem + 320, sw128_desc(a0 + L::kPl + kk * 32, 16, 1024), dh, id_pd, acc);
                }
                mma_commit(&bar[kSbB2]);
            }
            __syncwarp();
        } else if (warp >= 4) {
            // ======================================================= token warps
            // thread: row t (lanes 0-15 of the quarter) and a 16-column half
            // of each 32-column block
            const int t = 16 * q4 + (lane & 15), hc = (lane >> 4) * 16;
            const float fe = ex2f(GC - sG[t]);   // decay from token t to the chunk's end (<= 1)
            const float bt = sBb[(u & 1) * C + t];
            // D = beta_t v_t + ((T - I) diag(beta) V)_t - (W S)_t and
            // D' = 2^(G_C - G_t) D, each as a hi/lo pair [t][c]
            // (the V tile is read here too: its load is complete before A1 is)
            ok = mbar_wait_bounded(&bar[kSbLd0 + (u & 1)], static_cast<uint32_t>((u >> 1) & 1), status) && ok;
            ok = mbar_wait_bounded(&bar[kSbA1], ph, status) && ok;
            tc_fence_after();
#pragma unroll 1
            for (int cb = 0; cb < 64; cb += 32) {
                uint32_t r[16], rl[16], ru[16];
                tmem_ld16x2<16>(tmem + lane_off + cb, r);
                tmem_ld16x2<16>(tmem + lane_off + 64 + cb, rl);
                tmem_ld16x2<16>(tmem + lane_off + 320 + cb, ru);
                tmem_wait_ld();
#pragma unroll
                for (int x = 0; x < 16; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) + __uint_as_float(rl[x]));
#pragma unroll
                for (int j = 0; j < 16; j += 8) {
                    const uint32_t so = sw128_offset(t, cb + hc + j, L::kBlk);
                    const uint4 vr = *reinterpret_cast<const uint4 *>(sm + (u & 1) * L::kStage + L::kV + so);
                    const uint32_t v4[4] = {vr.x, vr.y, vr.z, vr.w};
                    float d[8];
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        d[2 * x] = fmaf(bt, __uint_as_float(v4[x] << 16),
                                        __uint_as_float(ru[j + 2 * x]) - __uint_as_float(r[j + 2 * x]));
                        d[2 * x + 1] = fmaf(bt, __uint_as_float(v4[x] & 0xffff0000u),
                                            __uint_as_float(ru[j + 2 * x + 1]) - __uint_as_float(r[j + 2 * x + 1]));
                    }
                    uint32_t hi[4], lo[4], ehi[4], elo[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        split_pair(d[2 * x], d[2 * x + 1], hi[x], lo[x]);
                        split_pair(fe * d[2 * x], fe * d[2 * x + 1], ehi[x], elo[x]);
                    }
                    *reinterpret_cast<uint4 *>(sm + L::kDh + so) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(sm + L::kDl + so) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    *reinterpret_cast<uint4 *>(sm + L::kEh + so) = make_uint4(ehi[0], ehi[1], ehi[2], ehi[3]);
                    *reinterpret_cast<uint4 *>(sm + L::kEl + so) = make_uint4(elo[0], elo[1], elo[2], elo[3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[kSbD]);
            // o_t = scale (2^G_t QS_t + PD_t) once Q S and P D are done
            ok = mbar_wait_bounded(&bar[kSbA2], ph, status) && ok;
            ok = mbar_wait_bounded(&bar[kSbB2], ph, status) && ok;
            tc_fence_after();
            const float f = scale * ex2f(sG[t]);
#pragma unroll 1
            for (int cb = 0; cb < 64; cb += 32) {
                uint32_t a[16], a2[16], b[16], b2[16], b3[16];
                tmem_ld16x2<16>(tmem + lane_off + 128 + cb, a);
                tmem_ld16x2<16>(tmem + lane_off + 192 + cb, a2);
                tmem_ld16x2<16>(tmem + lane_off + cb, b);
                tmem_ld16x2<16>(tmem + lane_off + 64 + cb, b2);
                tmem_ld16x2<16>(tmem + lane_off + 320 + cb, b3);
                tmem_wait_ld();
#pragma unroll
                for (int x = 0; x < 16; ++x) b2[x] = __float_as_uint(__uint_as_float(b2[x]) + __uint_as_float(b3[x]));
                if (t < n && ok) {
                    __nv_bfloat16 *dst = o + (rg + t) * DV + c0 + cb + hc;
#pragma unroll
                    for (int j = 0; j < 16; j += 8) {
                        float x[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            x[e] = fmaf(f, __uint_as_float(a[j + e]) + __uint_as_float(a2[j + e]),
                                        scale * (__uint_as_float(b[j + e]) + __uint_as_float(b2[j + e])));
                        *reinterpret_cast<uint4 *>(dst + j) =
                            make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]),
                                       pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
                    }
                }
            }
        } else {
            // ======================================================= state warps
            // P = tril(Q K^T 2^(G_t - G_i)) as a hi/lo pair [t][i] while the
            // state chain runs; thread: row t, a 16-column half of each block
            {
                if (split_exp && lane < 16) sE[16 * q4 + lane] = ex2f(-sG[16 * q4 + lane]);
                named_barrier(1, 128);   // the column table of the state warps
                const int t = 16 * q4 + (lane & 15), hc = (lane >> 4) * 16;
                const float Gt = sG[t];
                const float et = ex2f(Gt);
                // 16 scores of row t from column i0 on; the decay factor of
                // column i from the table or by its own exponential (eight
                // consecutive columns are one 16-byte piece of the swizzled
                // tile: one store each for hi and lo)
                auto p_block = [&](const uint32_t(&r)[16], int i0, auto factor) {
#pragma unroll
                    for (int j8 = 0; j8 < 16; j8 += 8) {
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int i = i0 + j8 + 2 * x;
                            const float x0 = i <= t ? __uint_as_float(r[j8 + 2 * x]) * factor(i) : 0.f;
                            const float x1 =
                                i + 1 <= t ? __uint_as_float(r[j8 + 2 * x + 1]) * factor(i + 1) : 0.f;
                            split_pair(x0, x1, hi[x], lo[x]);
                        }
                        const uint32_t so = sw128_offset(t, i0 + j8, L::kBlk);
                        *reinterpret_cast<uint4 *>(sm + L::kPh + so) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4 *>(sm + L::kPl + so) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                };
                ok = mbar_wait_bounded(&bar[kSbQK], ph, status) && ok;
                tc_fence_after();
#pragma unroll 1
                for (int cb = 0; cb < 64; cb += 32) {
                    uint32_t r[16];
                    tmem_ld16x2<16>(tmem + lane_off + 256 + cb, r);
                    tmem_wait_ld();
                    if (split_exp)
                        p_block(r, cb + hc, [&](int i) { return et * sE[i]; });
                    else
                        p_block(r, cb + hc, [&](int i) { return ex2f(Gt - sG[i]); });
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[kSbP]);
            }
            // S_i = 2^G_C S_i + (K^T D')_i (lane = key row, M = 128)
            ok = mbar_wait_bounded(&bar[kSbB1], ph, status) && ok;
            tc_fence_after();
            const float fc = ex2f(GC);
#pragma unroll
            for (int cb = 0; cb < 64; cb += 32) {
                uint32_t r[32], r2[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + 384 + cb, r);
                tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + 448 + cb, r2);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    S[cb + j] = fmaf(fc, S[cb + j], __uint_as_float(r[j]) + __uint_as_float(r2[j]));
            }
            // W S (before K^T D') and Q S are done reading the copy: the
            // copy for the next chunk
            ok = mbar_wait_bounded(&bar[kSbA2], ph, status) && ok;
            if (u + 1 < nch) state_copy();
            fence_proxy_async_smem();
        }
        tc_fence_before();
        ok = __syncthreads_and(ok) != 0;   // one verdict for the whole CTA; also ends the chunk
        tc_fence_after();
        if (!ok) break;
    }
    if (warp < 4 && hT && ok) {
#pragma unroll
        for (int c = 0; c < 64; c += 4)
            *reinterpret_cast<float4 *>(hT + (static_cast<size_t>(bh) * DK + i_row) * DV + c0 + c) =
                make_float4(S[c], S[c + 1], S[c + 2], S[c + 3]);
    }
    // every product issued here completes, and every chunk load lands, before
    // TMEM and shared memory are given up (a stream ended by an expired wait
    // may leave some in flight)
    if (warp == 8 && lane == 0) {
        mma_commit(&bar[kSbDrain]);
        mbar_wait_bounded(&bar[kSbDrain], 0, status);
    }
    if (warp == 9 && lane == 0) {
        mma_commit(&bar[kSbDrain2]);
        mbar_wait_bounded(&bar[kSbDrain2], 0, status);
        for (int c = max(0, loads - 2); c < loads; ++c)
            mbar_wait_bounded(&bar[kSbLd0 + (c & 1)], static_cast<uint32_t>((c >> 1) & 1), status);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ launch
template <int DV>
int launch_dv(const GdnChunkLaunch &p, cudaStream_t stream) {
    static bool attr_set = false;   // per instantiation, per process
    const int s1 = static_cast<int>(WySmem::kBytes);
    const int s2 = static_cast<int>(SeqSmem::kBytes);
    if (!attr_set) {
        if (cudaFuncSetAttribute(gdn_wy_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 s1) != cudaSuccess ||
            cudaFuncSetAttribute(gdn_seq_kernel<DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 s2) != cudaSuccess)
            return static_cast<int>(cudaGetLastError());
        attr_set = true;
    }
    const int nch = (p.T + C - 1) / C;
    const dim3 g1(static_cast<unsigned>(nch), static_cast<unsigned>(p.BH));
    const dim3 g2(DV / 64, static_cast<unsigned>(p.BH));
    const auto *kb = static_cast<const __nv_bfloat16 *>(p.k);
    gdn_wy_kernel<128><<<g1, NT, s1, stream>>>(kb, p.g, p.beta, p.W, p.Tm, p.T, p.status);
    SeqParams sp;
    sp.tm_q = p.tm_q;
    sp.tm_k = p.tm_k;
    sp.tm_v = p.tm_v;
    sp.tm_w = p.tm_w;
    sp.tm_t = p.tm_t;
    sp.g = p.g;
    sp.beta = p.beta;
    sp.h0 = p.h0;
    sp.o = static_cast<__nv_bfloat16 *>(p.o);
    sp.hT = p.hT;
    sp.scale = p.scale;
    sp.T = p.T;
    sp.status = p.status;
    gdn_seq_kernel<DV><<<g2, NTS, s2, stream>>>(sp);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace

int launch_gdn_chunk(const GdnChunkLaunch &p, cudaStream_t stream) {
    if (p.dv == 64) return launch_dv<64>(p, stream);
    if (p.dv == 128) return launch_dv<128>(p, stream);
    return launch_dv<256>(p, stream);
}

}  // namespace gla
