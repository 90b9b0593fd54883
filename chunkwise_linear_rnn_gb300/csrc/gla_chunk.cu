// gla_chunk.cu — chunkwise-parallel GLA forward on sm_103a tensor cores.
//
// Method ("Gated Linear Attention (GLA): Mathematical Foundations, ..."
// (llms.blog), sections "Sequence Partitioning and State Factorization",
// "Cumulative Decay Representation", "Intra-Chunk Matrix Multiplications",
// "Inter-Chunk Recurrence and Output Projection", "I/O-Aware Kernel Design"):
// per chunk of C tokens with A = log alpha and Gamma = in-chunk inclusive
// prefix sum of A (per key channel),
//     O     = scale * ( M V + (Q * e^Gamma) S_prev ),
//             M_ij = sum_d Q_id K_jd e^(Gamma_id - Gamma_jd)  for j <= i, else 0
//     S_new = diag(e^Gamma_C) S_prev + (K * e^(Gamma_C - Gamma))^T V,
// with the state S held on chip (TMEM, fp32) across the whole chunk loop.
//
// GB300 mapping (one CTA per (batch, head, value-column tile); C = 128 so that
// every product is a 128-row tcgen05 MMA whose TMEM row i is lane i):
//   * TMA streams the chunk's Q, K (bf16, 128-byte swizzle, directly in the
//     K-major operand layout), V (bf16, MN-major operand layout) and A (fp32).
//   * Fast path (every |Gamma| <= kExpBound in the chunk): thread d scans
//     channel d and rescales with the chunk-start reference,
//     Qh = Q e^Gamma (<= |Q|) and Kh = K e^-Gamma.  The decay then factorises:
//     the whole decayed score block is P = Qh Kh^T, and the state update is
//     S_new = diag(e^Gamma_C) (S_prev + Kh^T V): MMAs accumulating into TMEM
//     plus a per-lane scale (TMEM lane = key channel).  Every exponent is
//     bounded by kExpBound, so no factor overflows; masked entries of P are
//     selected away, never multiplied by zero.
//   * Exact path (a chunk whose decay leaves that bound, e.g. alpha -> 0): the
//     score block is built elementwise from e^(Gamma_i - Gamma_j) <= 1 and the
//     state factor from e^(Gamma_C - Gamma_j) <= 1; no exponent is positive.
//   * Precision: bf16 operands carry 8 significant bits.  The two roundings
//     that dominate the error of o and hT are removed by splitting the value
//     into a bf16 pair x = hi + lo (16 significant bits): Kh (used by the
//     score MMA and by the state MMA) and P (the A operand of P V, kept in
//     TMEM).  Q-side operands and the bf16 copy of S stay single.
//   * O = Qh S_prev + P V accumulates in TMEM; the epilogue scales, rounds to
//     bf16 and stores.  S_prev is fed to the MMA as a bf16 copy in shared
//     memory, refreshed from TMEM after each chunk.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gla_internal.h"
#include "gla_ptx.cuh"

namespace gla {
namespace {

constexpr int kChunk = 128;       // tokens per chunk = MMA M
constexpr int kThreads = 128;     // one thread per TMEM lane
constexpr float kExpBound = 30.f; // fast path needs |Gamma| <= kExpBound per chunk
constexpr uint32_t kTileRowBytes = 128;               // one swizzled row
constexpr uint32_t kBlk = kChunk * kTileRowBytes;     // 64-column block of a 128-row tile

template <int DK, int DVT>
struct Smem {
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kQBytes = kChunk * DK * 2;
    static constexpr uint32_t kK = kQ + kQBytes;          // Kh (high part)
    static constexpr uint32_t kKlo = kK + kQBytes;        // Kh low part
    static constexpr uint32_t kV = kKlo + kQBytes;
    static constexpr uint32_t kVBytes = kChunk * DVT * 2;
    static constexpr uint32_t kS = kV + kVBytes;
    static constexpr uint32_t kSBlk = DK * kTileRowBytes;  // 64-column block of the state copy
    static constexpr uint32_t kSBytes = DK * DVT * 2;
    static constexpr uint32_t kA = kS + kSBytes;
    static constexpr uint32_t kABytes = kChunk * DK * 4;
    static constexpr uint32_t kBar = kA + kABytes;
    static constexpr uint32_t kTotal = kBar + 64;
    static constexpr uint32_t kAlloc = kTotal + 1024;     // slack for 1024-byte alignment
    static_assert(kAlloc <= 232448, "shared memory budget exceeded");
};

// TMEM columns: P [0,128) (fp32 scores, then its bf16 hi/lo pair in place),
// O [128,128+DVT), S [256,256+DVT).
constexpr uint32_t kTmemP = 0, kTmemO = 128, kTmemS = 256, kTmemCols = 512;

__device__ __forceinline__ float bf16_at(const uint8_t *base, uint32_t off) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(base + off));
}
__device__ __forceinline__ void bf16_put(uint8_t *base, uint32_t off, float x) {
    *reinterpret_cast<__nv_bfloat16 *>(base + off) = __float2bfloat16_rn(x);
}
// x = hi + lo with hi = bf16(x), lo = bf16(x - hi); writes both, returns nothing.
__device__ __forceinline__ void bf16_split_put(uint8_t *hi_base, uint8_t *lo_base, uint32_t off,
                                               float x) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    *reinterpret_cast<__nv_bfloat16 *>(hi_base + off) = hi;
    *reinterpret_cast<__nv_bfloat16 *>(lo_base + off) = __float2bfloat16_rn(x - __bfloat162float(hi));
}

// Row i (= lane) of P, 32 consecutive columns starting at column 32*q, held in
// x[]: store its bf16 hi/lo pair in place as the TMEM A operand of P V —
// hi words at columns [32q, 32q+16), lo words at [32q+16, 32q+32).
__device__ __forceinline__ void store_p_split(uint32_t t_P, int q, const float (&x)[32]) {
    uint32_t hi[16], lo[16];
#pragma unroll
    for (int w = 0; w < 16; ++w) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(x[2 * w]);
        const __nv_bfloat16 h1 = __float2bfloat16_rn(x[2 * w + 1]);
        hi[w] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
                (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
        lo[w] = pack_bf16x2(x[2 * w] - __bfloat162float(h0), x[2 * w + 1] - __bfloat162float(h1));
    }
    tmem_st16(t_P + 32 * q, hi);
    tmem_st16(t_P + 32 * q + 16, lo);
}

template <int DK, int DVT>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_a,
                     const float *__restrict__ h0, float *__restrict__ hT,
                     __nv_bfloat16 *__restrict__ o, float scale, int H, int T, int dv,
                     int force_exact, unsigned int *status) {
    using L = Smem<DK, DVT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem + L::kQ;
    uint8_t *sK = smem + L::kK;
    uint8_t *sKlo = smem + L::kKlo;
    uint8_t *sV = smem + L::kV;
    uint8_t *sS = smem + L::kS;
    float *sA = reinterpret_cast<float *>(smem + L::kA);
    uint64_t *bar_tma = reinterpret_cast<uint64_t *>(smem + L::kBar);
    uint64_t *bar_mma = bar_tma + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_tma + 2);
    int *s_abort = reinterpret_cast<int *>(bar_tma + 3);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int dv_tile = blockIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    const int bh = b * H + h;
    const int dv0 = dv_tile * DVT;

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        *s_abort = 0;
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_a);
    }
    if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;  // this warp's TMEM lanes
    const uint32_t t_P = tmem + lane_base + kTmemP;
    const uint32_t t_O = tmem + lane_base + kTmemO;
    const uint32_t t_S = tmem + lane_base + kTmemS;
    const bool owns_state_row = (warp * 32) < DK;  // warp-uniform: lanes < DK are S rows
    const int d = tid;                             // key channel of this thread (if < DK)

    // ---- initial state: TMEM S (fp32) and its bf16 operand copy.
    if (owns_state_row) {
        const float *src = h0 ? h0 + (static_cast<size_t>(bh) * DK + d) * dv + dv0 : nullptr;
#pragma unroll
        for (int c0 = 0; c0 < DVT; c0 += 32) {
            uint32_t r[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                float4 x = src ? *reinterpret_cast<const float4 *>(src + c0 + j)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
                r[j] = __float_as_uint(x.x);
                r[j + 1] = __float_as_uint(x.y);
                r[j + 2] = __float_as_uint(x.z);
                r[j + 3] = __float_as_uint(x.w);
            }
            tmem_st32(t_S + c0, r);
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
                uint4 pk;
                pk.x = pack_bf16x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
                pk.y = pack_bf16x2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                pk.z = pack_bf16x2(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5]));
                pk.w = pack_bf16x2(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7]));
                *reinterpret_cast<uint4 *>(sS + sw128_offset(d, c0 + j, L::kSBlk)) = pk;
            }
        }
        tmem_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    const uint32_t load_bytes = 2u * L::kQBytes + L::kVBytes + L::kABytes;
    const uint32_t qk_bytes = 2u * L::kQBytes;
    constexpr uint32_t id_qk = idesc_bf16(128, 128, false, false);   // P = Qh Kh^T
    constexpr uint32_t id_qs = idesc_bf16(128, DVT, false, true);    // O = Qh S
    constexpr uint32_t id_pv = idesc_bf16(128, DVT, false, true);    // O += P V
    constexpr uint32_t id_kv = idesc_bf16(128, DVT, true, true);     // S += Kh^T V
    const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aKlo = smem_u32(sKlo);
    const uint32_t aV = smem_u32(sV), aS = smem_u32(sS);

    uint32_t ph_tma = 0, ph_mma = 0;
    const int n_chunks = (T + kChunk - 1) / kChunk;
    bool ok = true;

    for (int u = 0; u < n_chunks && ok; ++u) {
        const int t0 = u * kChunk;
        // ---------------- A1: TMA loads of the chunk
        if (tid == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar_tma, load_bytes);
#pragma unroll
            for (int kb = 0; kb < DK / 64; ++kb) {
                tma_load_3d(sQ + kb * kBlk, &tm_q, bar_tma, kb * 64, t0, bh);
                tma_load_3d(sK + kb * kBlk, &tm_k, bar_tma, kb * 64, t0, bh);
            }
#pragma unroll
            for (int nb = 0; nb < DVT / 64; ++nb)
                tma_load_3d(sV + nb * kBlk, &tm_v, bar_tma, dv0 + nb * 64, t0, bh);
            tma_load_3d(sA, &tm_a, bar_tma, 0, t0, bh);
        }
        if (!mbar_wait_bounded(bar_tma, ph_tma, status)) *s_abort = 1;
        ph_tma ^= 1;

        // ---------------- A2: in-chunk fp32 prefix sum of the log gates and the
        // bounded rescaling of Q and K (fast path, in place; Kh split hi + lo).
        float gC = 0.f;     // Gamma at the chunk end, channel d
        bool big = false;
        if (d < DK) {
            float g = 0.f, gmin = 0.f, gmax = 0.f;
            for (int i = 0; i < kChunk; ++i) {
                g += sA[i * DK + d];
                gmin = fminf(gmin, g);
                gmax = fmaxf(gmax, g);
                const float eq = __expf(g), ek = __expf(-g);
                const uint32_t off = sw128_offset(i, d, kBlk);
                bf16_put(sQ, off, bf16_at(sQ, off) * eq);
                bf16_split_put(sK, sKlo, off, bf16_at(sK, off) * ek);
            }
            gC = g;
            big = fmaxf(-gmin, gmax) > kExpBound;
        }
        fence_proxy_async_smem();
        const bool exact = __syncthreads_or((big || force_exact) ? 1 : 0) != 0;
        if (*s_abort) { ok = false; break; }

        if (!exact) {
            // ---------------- A3/A5: P = Qh Kh^T, O = Qh S_prev, S += Kh^T V
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks) {
                    const uint32_t koff = (ks >> 2) * kBlk + (ks & 3) * 32;
                    mma_bf16_ss(tmem + kTmemP, sw128_desc(aQ + koff, 16, 1024),
                                sw128_desc(aK + koff, 16, 1024), id_qk, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks) {
                    const uint32_t koff = (ks >> 2) * kBlk + (ks & 3) * 32;
                    mma_bf16_ss(tmem + kTmemP, sw128_desc(aQ + koff, 16, 1024),
                                sw128_desc(aKlo + koff, 16, 1024), id_qk, 1);
                }
#pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks) {
                    const uint32_t koff = (ks >> 2) * kBlk + (ks & 3) * 32;
                    mma_bf16_ss(tmem + kTmemO, sw128_desc(aQ + koff, 16, 1024),
                                sw128_desc(aS + ks * 2048, L::kSBlk, 1024), id_qs, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < kChunk / 16; ++ks) {
                    mma_bf16_ss(tmem + kTmemS, sw128_desc(aK + ks * 2048, kBlk, 1024),
                                sw128_desc(aV + ks * 2048, kBlk, 1024), id_kv, 1);
                    mma_bf16_ss(tmem + kTmemS, sw128_desc(aKlo + ks * 2048, kBlk, 1024),
                                sw128_desc(aV + ks * 2048, kBlk, 1024), id_kv, 1);
                }
                mma_commit(bar_mma);
            }
            if (!mbar_wait_bounded(bar_mma, ph_mma, status)) *s_abort = 1;
            ph_mma ^= 1;
            tc_fence_after();

            // ---------------- causal mask of P (row i = tid), split into the TMEM A operand
            {
                const int i = tid;
#pragma unroll
                for (int q = 0; q < kChunk / 32; ++q) {
                    uint32_t r[32];
                    tmem_ld32(t_P + 32 * q, r);
                    tmem_wait_ld();
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] = (32 * q + e <= i) ? __uint_as_float(r[e]) : 0.f;
                    store_p_split(t_P, q, x);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncthreads();
            if (*s_abort) { ok = false; break; }
        } else {
            // ---------------- exact path: reload raw Q, K; Gamma in place of A.
            __syncthreads();
            if (tid == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar_tma, qk_bytes);
#pragma unroll
                for (int kb = 0; kb < DK / 64; ++kb) {
                    tma_load_3d(sQ + kb * kBlk, &tm_q, bar_tma, kb * 64, t0, bh);
                    tma_load_3d(sK + kb * kBlk, &tm_k, bar_tma, kb * 64, t0, bh);
                }
            }
            if (d < DK) {
                float g = 0.f;
                for (int i = 0; i < kChunk; ++i) {
                    g += sA[i * DK + d];
                    sA[i * DK + d] = g;
                }
            }
            if (!mbar_wait_bounded(bar_tma, ph_tma, status)) *s_abort = 1;
            ph_tma ^= 1;
            __syncthreads();
            if (*s_abort) { ok = false; break; }
            // Score row i, elementwise: P_ij = sum_d Q_id K_jd e^(Gamma_id - Gamma_jd), j <= i.
            {
                const int i = tid;
#pragma unroll 1
                for (int q = 0; q < kChunk / 32; ++q) {
                    float x[32];
#pragma unroll 1
                    for (int e = 0; e < 32; ++e) {
                        const int j = 32 * q + e;
                        float acc = 0.f;
                        if (j <= i) {
                            for (int dd = 0; dd < DK; ++dd) {
                                acc += bf16_at(sQ, sw128_offset(i, dd, kBlk)) *
                                       bf16_at(sK, sw128_offset(j, dd, kBlk)) *
                                       __expf(sA[i * DK + dd] - sA[j * DK + dd]);
                            }
                        }
                        x[e] = acc;
                    }
                    store_p_split(t_P, q, x);
                }
                tmem_wait_st();
            }
            __syncthreads();
            if (d < DK) {
                for (int i = 0; i < kChunk; ++i) {
                    const float g = sA[i * DK + d];
                    const uint32_t off = sw128_offset(i, d, kBlk);
                    bf16_put(sQ, off, bf16_at(sQ, off) * __expf(g));
                    bf16_split_put(sK, sKlo, off, bf16_at(sK, off) * __expf(gC - g));
                }
            }
            // S_prev <- diag(e^Gamma_C) S_prev before the K^T V accumulation.
            if (owns_state_row) {
                const float f = __expf(gC);
#pragma unroll
                for (int c0 = 0; c0 < DVT; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(t_S + c0, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * f);
                    tmem_st32(t_S + c0, r);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks) {
                    const uint32_t koff = (ks >> 2) * kBlk + (ks & 3) * 32;
                    mma_bf16_ss(tmem + kTmemO, sw128_desc(aQ + koff, 16, 1024),
                                sw128_desc(aS + ks * 2048, L::kSBlk, 1024), id_qs, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < kChunk / 16; ++ks) {
                    mma_bf16_ss(tmem + kTmemS, sw128_desc(aK + ks * 2048, kBlk, 1024),
                                sw128_desc(aV + ks * 2048, kBlk, 1024), id_kv, 1);
                    mma_bf16_ss(tmem + kTmemS, sw128_desc(aKlo + ks * 2048, kBlk, 1024),
                                sw128_desc(aV + ks * 2048, kBlk, 1024), id_kv, 1);
                }
                // (O += P V is issued below, shared with the fast path.)
            }
        }

        // ---------------- A4: O += P V with P = hi + lo from TMEM
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < kChunk / 16; ++ks) {
                const uint32_t pcol = kTmemP + 32 * (ks >> 1) + 8 * (ks & 1);
                mma_bf16_ts(tmem + kTmemO, tmem + pcol, sw128_desc(aV + ks * 2048, kBlk, 1024),
                            id_pv, 1);
                mma_bf16_ts(tmem + kTmemO, tmem + pcol + 16, sw128_desc(aV + ks * 2048, kBlk, 1024),
                            id_pv, 1);
            }
            mma_commit(bar_mma);
        }
        if (!mbar_wait_bounded(bar_mma, ph_mma, status)) *s_abort = 1;
        ph_mma ^= 1;
        tc_fence_after();

        // ---------------- epilogue: O rows out; state scale and bf16 copy.
        {
            const int i = tid;
            const bool row_valid = (t0 + i) < T;
            __nv_bfloat16 *orow = o + (static_cast<size_t>(bh) * T + (t0 + i)) * dv + dv0;
#pragma unroll
            for (int c0 = 0; c0 < DVT; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(t_O + c0, r);
                tmem_wait_ld();
                if (row_valid) {
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        uint4 pk;
                        pk.x = pack_bf16x2(scale * __uint_as_float(r[j]), scale * __uint_as_float(r[j + 1]));
                        pk.y = pack_bf16x2(scale * __uint_as_float(r[j + 2]), scale * __uint_as_float(r[j + 3]));
                        pk.z = pack_bf16x2(scale * __uint_as_float(r[j + 4]), scale * __uint_as_float(r[j + 5]));
                        pk.w = pack_bf16x2(scale * __uint_as_float(r[j + 6]), scale * __uint_as_float(r[j + 7]));
                        *reinterpret_cast<uint4 *>(orow + c0 + j) = pk;
                    }
                }
            }
        }
        if (owns_state_row) {
            const float f = exact ? 1.f : __expf(gC);
#pragma unroll
            for (int c0 = 0; c0 < DVT; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(t_S + c0, r);
                tmem_wait_ld();
                if (!exact) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * f);
                    tmem_st32(t_S + c0, r);
                }
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    uint4 pk;
                    pk.x = pack_bf16x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
                    pk.y = pack_bf16x2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                    pk.z = pack_bf16x2(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5]));
                    pk.w = pack_bf16x2(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7]));
                    *reinterpret_cast<uint4 *>(sS + sw128_offset(d, c0 + j, L::kSBlk)) = pk;
                }
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (*s_abort) ok = false;
    }

    // ---- final state out.
    if (ok && hT && owns_state_row) {
        tc_fence_after();
        float *dst = hT + (static_cast<size_t>(bh) * DK + d) * dv + dv0;
#pragma unroll
        for (int c0 = 0; c0 < DVT; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(t_S + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4 *>(dst + c0 + j) =
                    make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int DK, int DVT>
int launch_tiles(const ChunkLaunch &p, cudaStream_t stream) {
    using L = Smem<DK, DVT>;
    auto kern = chunk_fwd_kernel<DK, DVT>;
    static bool attr_set = false;  // per instantiation, per process
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(L::kAlloc));
        if (e != cudaSuccess) return static_cast<int>(e);
        attr_set = true;
    }
    dim3 grid(p.dv / DVT, p.H, p.B);
    kern<<<grid, kThreads, L::kAlloc, stream>>>(p.tm_q, p.tm_k, p.tm_v, p.tm_a, p.h0, p.hT,
                                                static_cast<__nv_bfloat16 *>(p.o), p.scale, p.H,
                                                p.T, p.dv, p.force_exact, p.status);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace

int launch_chunk_fwd(const ChunkLaunch &p, cudaStream_t stream) {
    if (p.dk == 64) {
        if (p.dv_tile == 64) return launch_tiles<64, 64>(p, stream);
        if (p.dv_tile == 128) return launch_tiles<64, 128>(p, stream);
    } else if (p.dk == 128) {
        if (p.dv_tile == 64) return launch_tiles<128, 64>(p, stream);
        if (p.dv_tile == 128) return launch_tiles<128, 128>(p, stream);
    }
    return static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace gla
