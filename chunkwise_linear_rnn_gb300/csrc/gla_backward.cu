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
// Six launches:
//   1. bwd_sums:  every chunk independently, on the tensor cores (tcgen05,
//      TMEM accumulators): the state it adds from a zero start and the state
//      gradient its outputs add, plus its total decay;
//   2. bwd_state_scan:   S_u for u = 0 .. NC from those sums (elementwise);
//   3. bwd_adjoint_scan: R_u, the log-gate carries rowsum(R_u * S_(u+1)), dh0;
//   4. bwd_intra: every chunk's in-chunk products on the tensor cores, with
//      the state terms accumulated onto them in TMEM, written as dq, dk, dv
//      and dlog_alpha;
//   5. bwd_inter and 6. bwd_grads: the state terms (tensor cores) and the
//      in-chunk terms (CUDA cores, fp32) for the chunks that need exact decay
//      factors, flagged by bwd_intra; the other CTAs exit at once.
// Inside a chunk the decay factor e^(Gamma_t - Gamma_j) (t >= j) is split
// around a per-channel reference r = (Gamma_0 + Gamma_(C-1)) / 2, so both
// halves stay within 2^+-60 when the chunk's decay spans at most 2^120; a
// chunk that decays further takes each factor as one exponential ("exact"
// path).  All exponentials are base 2 on log2-scaled prefix sums.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gla_internal.h"
#include "gla_ptx.cuh"

namespace gla {
namespace {

constexpr int BC = 64;          // tokens per backward chunk
constexpr int TW = 32;          // value columns per log-gate carry group and per CUDA-core slice
constexpr int NT = 256;         // threads per CTA
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaxSpan = 120.f;  // log2 units: larger in-chunk decay spans take the exact path

__device__ __forceinline__ float bf(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}

// (x, y) as a bf16 pair hi plus a bf16 pair lo, x = hi + lo to 16 significant bits.
__device__ __forceinline__ void split_pair(float x, float y, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16x2(x, y);
    const float hx = __uint_as_float(hi << 16), hy = __uint_as_float(hi & 0xffff0000u);
    lo = pack_bf16x2(x - hx, y - hy);
}

// One unit (sequence n, head h; index n H + h) of the work, and where its
// pieces of scratch begin.  Chunk states and state gradients live as
// [unit][slot][dk][dv]: each chunk's dk x dv block in one piece, so that the
// chunk sums write, and the in-chunk kernel reads, whole contiguous blocks
// (the scans step one block per chunk); a unit has nch + 1 state slots and
// nch gradient slots.  Per-chunk arrays (decay, carry, flags) hold a unit's
// nch chunks from `cbase` on.
struct Unit {
    int nch;             // chunks of the sequence
    long long sbase;     // first state slot of the unit
    long long rbase;     // first gradient slot (also `cbase`)
};

__device__ __forceinline__ Unit unit_at(const BwdLaunch &p, int unit) {
    Unit w;
    if (!p.seqs) {
        w.nch = p.NC;
        w.sbase = static_cast<long long>(unit) * (p.NC + 1);
        w.rbase = static_cast<long long>(unit) * p.NC;
    } else {
        const int n = unit / p.H, h = unit % p.H;
        const int4 sq = p.seqs[n];   // {first row, length, chunks, first chunk}
        w.nch = sq.z;
        w.sbase = static_cast<long long>(sq.w + n) * p.H + static_cast<long long>(h) * (sq.z + 1);
        w.rbase = static_cast<long long>(sq.w) * p.H + static_cast<long long>(h) * sq.z;
    }
    return w;
}

// Chunk g (over all sequences) of head h.
struct Chunk {
    Unit w;
    int unit;            // n H + h
    int c;               // chunk within the sequence
    int n;               // valid rows (<= BC)
    long long row;       // its first row in the caller's tensors, in rows of dk / dv elements
};

__device__ __forceinline__ Chunk chunk_at(const BwdLaunch &p, long long g, int h) {
    Chunk k;
    if (!p.seqs) {
        const int b = static_cast<int>(g / p.NC);
        k.c = static_cast<int>(g % p.NC);
        k.unit = b * p.H + h;
        k.n = min(BC, p.T - k.c * BC);
        k.row = static_cast<long long>(k.unit) * p.T + static_cast<long long>(k.c) * BC;
    } else {
        // the last sequence whose first chunk is <= g (empty ones share a first chunk
        // with the sequence after them, which is then the one found)
        int lo = 0, hi = p.N - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.seqs[mid].w <= g) lo = mid;
            else hi = mid - 1;
        }
        const int4 sq = p.seqs[lo];
        k.c = static_cast<int>(g - sq.w);
        k.unit = lo * p.H + h;
        k.n = min(BC, sq.y - k.c * BC);
        k.row = static_cast<long long>(h) * p.T + sq.x + static_cast<long long>(k.c) * BC;
    }
    k.w = unit_at(p, k.unit);
    return k;
}

// Float offset of (row i, column c) of slot u of a unit whose slots begin at
// slot `base` of the states or gradients.
template <int DK, int DV>
__device__ __forceinline__ size_t slot_index(long long base, int i, int c, int u) {
    return ((static_cast<size_t>(base) + u) * DK + i) * DV + c;
}

// Load one chunk of log-gates (log2 units, rows past the sequence end zero,
// so the prefix sum stays flat there) and take the inclusive prefix sum per
// channel.  sG is [BC][LD].  All loads are issued before the first use.
// prefix_issue loads this thread's share into registers; prefix_finish stores
// it (log2 units) and scans.
template <int DK, int NTH>
__device__ __forceinline__ void prefix_issue(float4 (&r)[BC * DK / 4 / NTH], const float *__restrict__ la,
                                             int n) {
    constexpr int PER = BC * DK / 4 / NTH;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
        const int e = (threadIdx.x + m * NTH) * 4, t = e / DK;
        r[m] = t < n ? *reinterpret_cast<const float4 *>(la + e) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

template <int DK, int LD, int NTH>
__device__ __forceinline__ void prefix_finish(float *sG, const float4 (&r)[BC * DK / 4 / NTH]) {
    constexpr int PER = BC * DK / 4 / NTH;
#pragma unroll
    for (int m = 0; m < PER; ++m) {
        const int e = (threadIdx.x + m * NTH) * 4, t = e / DK, i = e % DK;
        float *d = sG + t * LD + i;
        d[0] = r[m].x * kLog2e;
        d[1] = r[m].y * kLog2e;
        d[2] = r[m].z * kLog2e;
        d[3] = r[m].w * kLog2e;
    }
    __syncthreads();
    if (threadIdx.x < DK) {
        // 16 rows' loads in flight at a time, then their running sums (the
        // same order of additions as one row at a time)
        float acc = 0.f;
#pragma unroll
        for (int t0 = 0; t0 < BC; t0 += 16) {
            float x[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) x[j] = sG[(t0 + j) * LD + threadIdx.x];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                acc += x[j];
                sG[(t0 + j) * LD + threadIdx.x] = acc;
            }
        }
    }
    __syncthreads();
}

template <int DK, int LD, int NTH = NT>
__device__ __forceinline__ void load_prefix(float *sG, const float *__restrict__ la, int n) {
    float4 r[BC * DK / 4 / NTH];
    prefix_issue<DK, NTH>(r, la, n);
    prefix_finish<DK, LD, NTH>(sG, r);
}

// ---------------------------------------------------------------------------
// 1. chunk sums on the tensor cores.  Work item (which, chunk, head), the
//    chunk index fastest: which = 0 gives the state a chunk adds from a zero
//    start, dS_u = (K e^(Gamma_C - Gamma))^T V; which = 1 the state gradient
//    its outputs add, dR_u = scale (Q e^Gamma)^T dO.
//    M = 128 key channels (zero rows past dk), N = dv, K = the chunk's tokens.
//    The key-side operand is split into a bf16 pair (hi + lo, 16 significant
//    bits) because these sums accumulate over the whole sequence; V and dO
//    are bf16 inputs, exact.  Operand tiles are 128-byte swizzled, 64
//    channels (or value columns) per block, read MN-major.
//    Persistent CTAs, item after item (CTA c takes items c, c + grid, ...),
//    so that loads, products and stores of neighbouring items overlap:
//      - the load warp's first thread stages an item's raw rows (log-gates,
//        key-side rows, value-side rows; only the chunk's valid rows) by bulk
//        copies into one of two staging buffers, as soon as the compute warps
//        are done with the item that used the buffer before;
//      - the 8 compute warps take the item's prefix sums in place, form the
//        operand tiles, release the staging buffer, issue the products into
//        one of two TMEM accumulators, and then store the previous item's
//        sums while these products run.
constexpr int kSumThreads = 256;                  // compute threads
constexpr int kSumLoadWarp = kSumThreads / 32;    // the warp after them
constexpr int kSumAllThreads = kSumThreads + 32;

template <int DK, int DV>
struct SumSmem {
    static constexpr uint32_t kBlk = BC * 128;              // one 64-column block of a tile
    static constexpr uint32_t kGBytes = BC * DK * 4;        // staged log-gates, then prefix sums
    static constexpr uint32_t kABytes = BC * DK * 2;        // staged key-side rows
    static constexpr uint32_t kBBytes = BC * DV * 2;        // staged value-side rows
    static constexpr uint32_t kStage = kGBytes + kABytes + kBBytes;
    static constexpr uint32_t kSt = 0;                      // two staging buffers
    static constexpr uint32_t kA = 2 * kStage;              // A hi: two blocks (128 channels)
    static constexpr uint32_t kAlo = kA + 2 * kBlk;
    static constexpr uint32_t kB = kAlo + 2 * kBlk;         // B: DV / 64 blocks
    static constexpr uint32_t kBar = kB + (DV / 64) * kBlk;  // full[2], empty[2], done[2], drain
    static constexpr uint32_t kSlot = kBar + 8 * 8;
    static constexpr uint32_t kBytes = kSlot + 16 + 1024;   // + alignment slack
    static_assert(kStage % 1024 == 0, "operand tiles stay 1024-byte aligned");
    static_assert(kStage >= 8 * 32 * 32 * 4, "a staging buffer holds the 8 warps' store blocks");
    static_assert(kBytes <= 232448, "shared memory budget exceeded");
};

// Item w of the chunk sums: chunk fastest, then head, then which.
struct SumItem {
    long long g;   // chunk over all sequences (one head)
    int h, which;
};

__device__ __forceinline__ SumItem sum_item(const BwdLaunch &p, long long w) {
    SumItem it;
    it.g = w % p.chunks;
    const long long r = w / p.chunks;
    it.h = static_cast<int>(r % p.H);
    it.which = static_cast<int>(r / p.H);
    return it;
}

// AND of `pred` over the `n` threads of named barrier `id`.
__device__ __forceinline__ bool bar_and(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
        : "memory");
    return r != 0u;
}

template <int DK, int DV>
__global__ void __launch_bounds__(kSumAllThreads, 1) bwd_sums_kernel(BwdLaunch p, long long items) {
    constexpr int NTS = kSumThreads;
    using L = SumSmem<DK, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sA = sm + L::kA, *sAlo = sm + L::kAlo, *sB = sm + L::kB;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L::kBar);
    uint64_t *empty = full + 2, *done = full + 4, *drain = full + 6;
    uint32_t *slot = reinterpret_cast<uint32_t *>(sm + L::kSlot);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long first = blockIdx.x, stride = gridDim.x;
    const int nitems = first < items ? static_cast<int>((items - 1 - first) / stride + 1) : 0;

    if (warp == 0) tmem_alloc(slot, 2 * DV);   // two accumulators of DV columns
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&full[b], 1);
            mbar_init(&empty[b], NTS / 32);
            mbar_init(&done[b], 1);
        }
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;

    if (warp == kSumLoadWarp) {
        // ================================================= load warp
        int issued = 0;
        if (lane == 0) {
            for (int kk = 0; kk < nitems; ++kk) {
                const int s = kk & 1;
                // the compute warps are done with item kk - 2, which used this buffer
                if (kk >= 2 && !mbar_wait_bounded(&empty[s], ((kk - 2) >> 1) & 1, p.status)) break;
                const SumItem it = sum_item(p, first + kk * stride);
                const Chunk ck = chunk_at(p, it.g, it.h);
                const uint32_t n = static_cast<uint32_t>(ck.n);
                const size_t rk = static_cast<size_t>(ck.row) * DK;
                const size_t rv = static_cast<size_t>(ck.row) * DV;
                uint8_t *st = sm + L::kSt + s * L::kStage;
                mbar_arrive_expect_tx(&full[s], n * (DK * 4 + DK * 2 + DV * 2));
                bulk_load(st, p.log_alpha + rk, n * DK * 4, &full[s]);
                bulk_load(st + L::kGBytes, (it.which ? p.q : p.k) + rk, n * DK * 2, &full[s]);
                bulk_load(st + L::kGBytes + L::kABytes, (it.which ? p.d_o : p.v) + rv, n * DV * 2,
                          &full[s]);
                issued = kk + 1;
            }
            // every copy issued here lands before the shared memory is given up
            for (int c = issued > 2 ? issued - 2 : 0; c < issued; ++c)
                mbar_wait_bounded(&full[c & 1], (c >> 1) & 1, p.status);
        }
        __syncwarp();
    } else {
        // ================================================= compute warps
        bool ok = true;
        // the stores of item j's sums from TMEM accumulator j & 1.  A warp
        // reads key channels 32 (warp % 4) .. + 31 (its TMEM lanes, one row per
        // thread), warps 0-3 the first half of the value columns, warps 4-7 the
        // second, 32 columns at a time; each 32 x 32 block goes through the
        // warp's 4 KB of `xbuf` (16-byte pieces XOR-swizzled by row, so that
        // neither side has bank conflicts), and 8 threads then store one row's
        // 128 bytes: every store instruction writes 4 whole lines.
        auto store_sums = [&](int j, uint8_t *xbuf) {
            const SumItem it = sum_item(p, first + j * stride);
            const Chunk ck = chunk_at(p, it.g, it.h);
            const float mult = it.which ? p.scale : 1.f;
            float *dst = it.which ? p.adjoints : p.states;
            const long long base = it.which ? ck.w.rbase : ck.w.sbase;
            float *xw = reinterpret_cast<float *>(xbuf) + warp * 1024;
            const int i0 = 32 * (warp & 3);
            const uint32_t taddr = tmem + (j & 1) * DV + (static_cast<uint32_t>(i0) << 16);
            const int cbeg = warp < 4 ? 0 : DV / 2, cend = warp < 4 ? DV / 2 : DV;
#pragma unroll 1
            for (int c0 = cbeg; c0 < cend; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(taddr + c0, r);
                tmem_wait_ld();
#pragma unroll
                for (int x = 0; x < 8; ++x)
                    *reinterpret_cast<float4 *>(xw + lane * 32 + ((x ^ (lane & 7)) << 2)) =
                        make_float4(__uint_as_float(r[4 * x]) * mult, __uint_as_float(r[4 * x + 1]) * mult,
                                    __uint_as_float(r[4 * x + 2]) * mult, __uint_as_float(r[4 * x + 3]) * mult);
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int rr = 4 * k + (lane >> 3), x = lane & 7;
                    const float4 v = *reinterpret_cast<const float4 *>(xw + rr * 32 + ((x ^ (rr & 7)) << 2));
                    if (ok && i0 + rr < DK)
                        *reinterpret_cast<float4 *>(dst + slot_index<DK, DV>(base, i0 + rr, c0 + 4 * x, ck.c)) = v;
                }
                __syncwarp();
            }
        };
        int kk = 0;
#pragma unroll 1
        for (; kk < nitems; ++kk) {
            const int s = kk & 1;
            const SumItem it = sum_item(p, first + kk * stride);
            const Chunk ck = chunk_at(p, it.g, it.h);
            const int n = ck.n, which = it.which;
            uint8_t *st = sm + L::kSt + s * L::kStage;
            float *sG = reinterpret_cast<float *>(st);
            const uint8_t *sa = st + L::kGBytes, *sb = st + L::kGBytes + L::kABytes;
            ok = mbar_wait_bounded(&full[s], (kk >> 1) & 1, p.status) && ok;
            ok = bar_and(1, NTS, ok);   // one verdict for the compute warps
            if (!ok) break;
            // inclusive prefix sums of the log-gates (log2 units), in place, one
            // channel per thread; rows past the chunk's valid ones count as zero
            if (tid < DK) {
                float acc = 0.f;
#pragma unroll
                for (int t0 = 0; t0 < BC; t0 += 16) {
                    float x[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        x[j] = t0 + j < n ? sG[(t0 + j) * DK + tid] * kLog2e : 0.f;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        acc += x[j];
                        sG[(t0 + j) * DK + tid] = acc;
                    }
                }
            }
            // the operand tiles are free once item kk - 1's products are done
            if (kk >= 1) ok = mbar_wait_bounded(&done[(kk - 1) & 1], ((kk - 1) >> 1) & 1, p.status) && ok;
            named_barrier(1, NTS);   // the prefix sums
            tc_fence_after();
            // A: rows = tokens, columns = key channels, scaled and split
            constexpr int APER = BC * 64 / NTS;           // channel pairs per thread
#pragma unroll
            for (int m = 0; m < APER; ++m) {
                const int e = tid + m * NTS, t = e >> 6, i = (e & 63) * 2;
                uint32_t hi = 0u, lo = 0u;
                if (t < n && i < DK) {
                    const uint32_t a = *reinterpret_cast<const uint32_t *>(sa + (t * DK + i) * 2);
                    const float f0 = __uint_as_float(a << 16), f1 = __uint_as_float(a & 0xffff0000u);
                    const float g0 = sG[t * DK + i], g1 = sG[t * DK + i + 1];
                    const float e0 = which ? exp2f(g0) : exp2f(sG[(BC - 1) * DK + i] - g0);
                    const float e1 = which ? exp2f(g1) : exp2f(sG[(BC - 1) * DK + i + 1] - g1);
                    split_pair(f0 * e0, f1 * e1, hi, lo);
                }
                const uint32_t off = sw128_offset(t, i, L::kBlk);
                *reinterpret_cast<uint32_t *>(sA + off) = hi;
                *reinterpret_cast<uint32_t *>(sAlo + off) = lo;
            }
            // B: rows = tokens, columns = value columns (bf16 copied as is)
            constexpr int BPER = BC * DV / 8 / NTS;       // 16-byte value groups per thread
#pragma unroll
            for (int m = 0; m < BPER; ++m) {
                const int e = tid + m * NTS, t = e / (DV / 8), c = (e % (DV / 8)) * 8;
                const uint4 b = t < n ? *reinterpret_cast<const uint4 *>(sb + (t * DV + c) * 2)
                                      : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(sB + sw128_offset(t, c, L::kBlk)) = b;
            }
            if (which == 0 && warp < 4) {
                const int i = 32 * warp + lane;
                if (i < DK) p.decay[static_cast<size_t>(ck.w.rbase + ck.c) * DK + i] = exp2f(sG[(BC - 1) * DK + i]);
            }
            fence_proxy_async_smem();   // the tiles, before the tensor core reads them
            tc_fence_before();
            ok = bar_and(1, NTS, ok);   // the tiles, and the previous item's verdict
            tc_fence_after();
            if (!ok) break;
            if (tid == 0) {
                constexpr uint32_t id = idesc_bf16(128, DV, true, true);
                const uint32_t aA = smem_u32(sA), aAlo = smem_u32(sAlo), aB = smem_u32(sB);
                const uint32_t acc = tmem + s * DV;
#pragma unroll
                for (int ks = 0; ks < BC / 16; ++ks) {
                    const uint64_t db = sw128_desc(aB + ks * 2048, L::kBlk, 1024);
                    mma_bf16_ss(acc, sw128_desc(aA + ks * 2048, L::kBlk, 1024), db, id, ks > 0);
                    mma_bf16_ss(acc, sw128_desc(aAlo + ks * 2048, L::kBlk, 1024), db, id, 1);
                }
                mma_commit(&done[s]);
            }
            // the previous item's sums, while these products run, through this
            // item's staging buffer (every warp is done reading it: the barrier
            // above); then the buffer goes back to the load warp, the generic
            // writes to it ordered before the next bulk copy into it
            if (kk >= 1) store_sums(kk - 1, st);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            tc_fence_before();
        }
        // the last item's sums (after a full run of the loop)
        if (ok && kk == nitems && nitems > 0) {
            ok = mbar_wait_bounded(&done[(nitems - 1) & 1], ((nitems - 1) >> 1) & 1, p.status);
            tc_fence_after();
            store_sums(nitems - 1, sm + L::kSt + ((nitems - 1) & 1) * L::kStage);
        }
        // every product issued here completes before TMEM is given up
        if (tid == 0) {
            mma_commit(drain);
            mbar_wait_bounded(drain, 0, p.status);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * DV);
    }
}

// ---------------------------------------------------------------------------
// 2. scans over the chunks, one thread per state element (bh, i, c), value
//    columns fastest so that a warp covers 32 columns of one row (one
//    128-byte line of each chunk's block; the next chunk's is a block on).
//    States:    slot u holds dS_u on entry and S_u on exit, slot NC gets hT:
//               S_(u+1) = e^Gamma_C(u) S_u + dS_u, S_0 = h0.
//    Gradients: slot u holds dR_u on entry and R_u on exit, dh0 = R_(-1):
//               R_(u-1) = e^Gamma_C(u) R_u + dR_u, R_(NC-1) = dhT;
//               plus the log-gate carry rowsum(R_u * S_(u+1)) per 32 columns.
constexpr int kScanUnroll = 16;

template <int DK, int DV>
__global__ void __launch_bounds__(256, 3) bwd_state_scan_kernel(BwdLaunch p) {
    const size_t e = static_cast<size_t>(blockIdx.x) * 256 + threadIdx.x;
    const Unit w = unit_at(p, static_cast<int>(e / (DK * DV)));
    const int NCu = w.nch;
    const int rem = static_cast<int>(e % (DK * DV)), i = rem / DV;
    constexpr size_t kM = static_cast<size_t>(DK) * DV;   // one slot step
    float *buf = p.states + slot_index<DK, DV>(w.sbase, i, rem % DV, 0);
    const float *dec = p.decay + static_cast<size_t>(w.rbase) * DK + i;
    float S = p.h0 ? p.h0[e] : 0.f;
    float d[kScanUnroll], a[kScanUnroll];
    auto fetch = [&](int u0) {
#pragma unroll
        for (int j = 0; j < kScanUnroll; ++j) {
            if (u0 + j < NCu) {
                d[j] = buf[(u0 + j) * kM];
                a[j] = dec[static_cast<size_t>(u0 + j) * DK];
            }
        }
    };
    fetch(0);
    for (int u0 = 0; u0 < NCu; u0 += kScanUnroll) {
        float dn[kScanUnroll], an[kScanUnroll];
#pragma unroll
        for (int j = 0; j < kScanUnroll; ++j) {
            dn[j] = d[j];
            an[j] = a[j];
        }
        if (u0 + kScanUnroll < NCu) fetch(u0 + kScanUnroll);   // next group in flight
#pragma unroll
        for (int j = 0; j < kScanUnroll; ++j) {
            if (u0 + j < NCu) {
                buf[(u0 + j) * kM] = S;
                S = fmaf(an[j], S, dn[j]);
            }
        }
    }
    buf[static_cast<size_t>(NCu) * kM] = S;
}

template <int DK, int DV>
__global__ void __launch_bounds__(256, 2) bwd_adjoint_scan_kernel(BwdLaunch p) {
    constexpr int NTILE = DV / TW;
    const size_t e = static_cast<size_t>(blockIdx.x) * 256 + threadIdx.x;
    const Unit w = unit_at(p, static_cast<int>(e / (DK * DV)));
    const int NCu = w.nch;
    const int rem = static_cast<int>(e % (DK * DV)), i = rem / DV, c = rem % DV;
    const int lane = threadIdx.x & 31;
    constexpr size_t kM = static_cast<size_t>(DK) * DV;   // one slot step
    float *buf = p.adjoints + slot_index<DK, DV>(w.rbase, i, c, 0);
    const float *st = p.states + slot_index<DK, DV>(w.sbase, i, c, 0);
    const float *dec = p.decay + static_cast<size_t>(w.rbase) * DK + i;
    float *carry = p.carry + static_cast<size_t>(w.rbase) * NTILE * DK + (c / TW) * DK + i;
    float R = p.dhT ? p.dhT[e] : 0.f;
    float d[kScanUnroll], a[kScanUnroll], sn[kScanUnroll];
    auto fetch = [&](int u0) {
#pragma unroll
        for (int j = 0; j < kScanUnroll; ++j) {
            if (u0 - j >= 0) {
                d[j] = buf[(u0 - j) * kM];
                a[j] = dec[static_cast<size_t>(u0 - j) * DK];
                sn[j] = st[(u0 - j + 1) * kM];
            }
        }
    };
    fetch(NCu - 1);
    for (int u0 = NCu - 1; u0 >= 0; u0 -= kScanUnroll) {
        float dc[kScanUnroll], ac[kScanUnroll], sc[kScanUnroll];
#pragma unroll
        for (int j = 0; j < kScanUnroll; ++j) {
            dc[j] = d[j];
            ac[j] = a[j];
            sc[j] = sn[j];
        }
        if (u0 - kScanUnroll >= 0) fetch(u0 - kScanUnroll);   // next group in flight
#pragma unroll
        for (int j = 0; j < kScanUnroll; ++j) {
            const int u = u0 - j;
            if (u >= 0) {
                buf[u * kM] = R;
                float part = R * sc[j];
#pragma unroll
                for (int m = 16; m > 0; m >>= 1) part += __shfl_xor_sync(0xffffffffu, part, m);
                if (lane == 0) carry[static_cast<size_t>(u) * NTILE * DK] = part;
                R = fmaf(ac[j], R, dc[j]);
            }
        }
    }
    if (p.gh0) p.gh0[e] = R;
}

// ---------------------------------------------------------------------------
// 5. the state terms of the gradients on the tensor cores, one CTA per
//    flagged (chunk, head), written as fp32 partial gradients for bwd_grads:
//       pq = scale e^Gamma (dO S_u^T),  pk = e^(Gamma_C - Gamma) (V R_u^T),
//       pv = (K e^(Gamma_C - Gamma)) R_u.
//    Transposed so that every product has M = 128 (key channels or value
//    columns on the TMEM lanes) and N = the chunk's 64 tokens:
//       D1 = S_u dO^T, D2 = R_u V^T (K = value columns), D3 = R_u^T K'^T
//       (K = key channels).  The value columns go through in slabs of 128
//    (zero-padded when dv = 64).  S_u and R_u are split into bf16 pairs (hi +
//    lo): dlog_alpha takes the difference q dq - k dk, which cancels, so dq
//    and dk need more than one bf16 rounding of the states.
template <int DK, int DV>
struct InterSmem {
    static constexpr int kSlab = 128;
    static constexpr int kSlabs = DV > kSlab ? DV / kSlab : 1;
    static constexpr uint32_t kBlkI = 128 * 128;   // 64-column block of a 128-row tile
    static constexpr uint32_t kBlkT = BC * 128;    // 64-column block of a 64-row tile
    static constexpr uint32_t kS = 0;
    static constexpr uint32_t kSlo = kS + 2 * kBlkI;
    static constexpr uint32_t kR = kSlo + 2 * kBlkI;
    static constexpr uint32_t kRlo = kR + 2 * kBlkI;
    static constexpr uint32_t kDo = kRlo + 2 * kBlkI;
    static constexpr uint32_t kV = kDo + 2 * kBlkT;
    static constexpr uint32_t kKp = kV + 2 * kBlkT;
    static constexpr uint32_t kG = kKp + 2 * kBlkT;
    static constexpr uint32_t kBar = kG + BC * DK * 4;
    static constexpr uint32_t kSlot = kBar + 8;
    static constexpr uint32_t kBytes = kSlot + 8 + 1024;
    static constexpr uint32_t kCols = 256;         // D1 | D2 | D3 slab 0 | D3 slab 1
};

constexpr int kInterThreads = 256;

template <int DK, int DV>
__global__ void __launch_bounds__(kInterThreads, 1) bwd_inter_kernel(BwdLaunch p) {
    constexpr int NTI = kInterThreads;
    using L = InterSmem<DK, DV>;
    constexpr int SLAB = L::kSlab;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sS = sm + L::kS, *sR = sm + L::kR, *sDo = sm + L::kDo, *sV = sm + L::kV;
    uint8_t *sSlo = sm + L::kSlo, *sRlo = sm + L::kRlo;
    uint8_t *sKp = sm + L::kKp;
    float *sG = reinterpret_cast<float *>(sm + L::kG);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::kBar);
    uint32_t *slot = reinterpret_cast<uint32_t *>(sm + L::kSlot);
    const Chunk ck = chunk_at(p, blockIdx.x, blockIdx.y);
    const int u = ck.c, n = ck.n;
    if (!p.wide[ck.w.rbase + u]) return;   // done by bwd_intra
    const int tid = threadIdx.x, warp = tid >> 5;
    // first rows of the caller's tensors; the partials use the same offsets
    const size_t rk = static_cast<size_t>(ck.row) * DK, rv = static_cast<size_t>(ck.row) * DV;
    const size_t xk = rk, xv = rv;

    if (warp == 0) tmem_alloc(slot, L::kCols);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    // keys, loaded before the prefix sums; K' = k e^(Gamma_C - Gamma), one bf16
    constexpr int KPER = BC * DK / 2 / NTI;
    uint32_t kraw[KPER];
#pragma unroll
    for (int m = 0; m < KPER; ++m) {
        const int e = (tid + m * NTI) * 2, t = e / DK;
        kraw[m] = t < n ? *reinterpret_cast<const uint32_t *>(p.k + rk + e) : 0u;
    }
    load_prefix<DK, DK, NTI>(sG, p.log_alpha + rk, n);
#pragma unroll
    for (int m = 0; m < KPER; ++m) {
        const int e = (tid + m * NTI) * 2, t = e / DK, i = e % DK;
        const float k0 = __uint_as_float(kraw[m] << 16), k1 = __uint_as_float(kraw[m] & 0xffff0000u);
        const float f0 = exp2f(sG[(BC - 1) * DK + i] - sG[t * DK + i]);
        const float f1 = exp2f(sG[(BC - 1) * DK + i + 1] - sG[t * DK + i + 1]);
        *reinterpret_cast<uint32_t *>(sKp + sw128_offset(t, i, L::kBlkT)) = pack_bf16x2(k0 * f0, k1 * f1);
    }

    bool ok = true;
    for (int h = 0; h < L::kSlabs; ++h) {
        if (h > 0) {   // the previous slab's products must be done reading smem
            ok = ok && mbar_wait_bounded(bar, (h - 1) & 1, p.status);
            tc_fence_after();
        }
        const int cb = h * SLAB;
        // S_u and R_u rows (128, zero past dk) x 128 value columns -> bf16 pairs;
        // batches of 8 float4 per matrix in flight per thread
        constexpr int SPER = 128 * SLAB / 4 / NTI, SB = SPER;
#pragma unroll 1
        for (int mb = 0; mb < SPER; mb += SB) {
            float4 sv[SB], rr[SB];
#pragma unroll
            for (int m = 0; m < SB; ++m) {
                const int e = tid + (mb + m) * NTI, i = e / (SLAB / 4), cl = (e % (SLAB / 4)) * 4;
                sv[m] = make_float4(0.f, 0.f, 0.f, 0.f);
                rr[m] = sv[m];
                if (i < DK && cb + cl < DV) {
                    sv[m] = *reinterpret_cast<const float4 *>(
                        p.states + slot_index<DK, DV>(ck.w.sbase, i, cb + cl, u));
                    rr[m] = *reinterpret_cast<const float4 *>(
                        p.adjoints + slot_index<DK, DV>(ck.w.rbase, i, cb + cl, u));
                }
            }
#pragma unroll
            for (int m = 0; m < SB; ++m) {
                const int e = tid + (mb + m) * NTI, i = e / (SLAB / 4), cl = (e % (SLAB / 4)) * 4;
                const uint32_t off = sw128_offset(i, cl, L::kBlkI);
                uint32_t h0, l0, h1, l1;
                split_pair(sv[m].x, sv[m].y, h0, l0);
                split_pair(sv[m].z, sv[m].w, h1, l1);
                *reinterpret_cast<uint2 *>(sS + off) = make_uint2(h0, h1);
                *reinterpret_cast<uint2 *>(sSlo + off) = make_uint2(l0, l1);
                split_pair(rr[m].x, rr[m].y, h0, l0);
                split_pair(rr[m].z, rr[m].w, h1, l1);
                *reinterpret_cast<uint2 *>(sR + off) = make_uint2(h0, h1);
                *reinterpret_cast<uint2 *>(sRlo + off) = make_uint2(l0, l1);
            }
        }
        // dO and V rows (64 tokens) x 128 value columns
#pragma unroll
        for (int m = 0; m < BC * SLAB / 8 / NTI; ++m) {
            const int e = tid + m * NTI, t = e / (SLAB / 8), cl = (e % (SLAB / 8)) * 8;
            uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
            if (t < n && cb + cl < DV) {
                const size_t off = rv + static_cast<size_t>(t) * DV + cb + cl;
                a = *reinterpret_cast<const uint4 *>(p.d_o + off);
                b = *reinterpret_cast<const uint4 *>(p.v + off);
            }
            const uint32_t off = sw128_offset(t, cl, L::kBlkT);
            *reinterpret_cast<uint4 *>(sDo + off) = a;
            *reinterpret_cast<uint4 *>(sV + off) = b;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const uint32_t tmem = *slot;
            constexpr uint32_t id_kk = idesc_bf16(128, BC, false, false);
            constexpr uint32_t id_mk = idesc_bf16(128, BC, true, false);
            const uint32_t aS = smem_u32(sS), aR = smem_u32(sR), aDo = smem_u32(sDo);
            const uint32_t aSlo = smem_u32(sSlo), aRlo = smem_u32(sRlo);
            const uint32_t aV = smem_u32(sV), aKp = smem_u32(sKp);
#pragma unroll
            for (int kk = 0; kk < SLAB / 16; ++kk) {
                const uint32_t oi = (kk >> 2) * L::kBlkI + (kk & 3) * 32;
                const uint32_t ot = (kk >> 2) * L::kBlkT + (kk & 3) * 32;
                const uint32_t acc = (h > 0 || kk > 0) ? 1u : 0u;
                const uint64_t bdo = sw128_desc(aDo + ot, 16, 1024), bv = sw128_desc(aV + ot, 16, 1024);
                mma_bf16_ss(tmem, sw128_desc(aS + oi, 16, 1024), bdo, id_kk, acc);
                mma_bf16_ss(tmem, sw128_desc(aSlo + oi, 16, 1024), bdo, id_kk, 1u);
                mma_bf16_ss(tmem + BC, sw128_desc(aR + oi, 16, 1024), bv, id_kk, acc);
                mma_bf16_ss(tmem + BC, sw128_desc(aRlo + oi, 16, 1024), bv, id_kk, 1u);
            }
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                const uint32_t ot = (kk >> 2) * L::kBlkT + (kk & 3) * 32;
                const uint64_t bk = sw128_desc(aKp + ot, 16, 1024);
                mma_bf16_ss(tmem + 2 * BC + h * BC, sw128_desc(aR + kk * 2048, L::kBlkI, 1024), bk,
                            id_mk, kk > 0 ? 1u : 0u);
                mma_bf16_ss(tmem + 2 * BC + h * BC, sw128_desc(aRlo + kk * 2048, L::kBlkI, 1024), bk,
                            id_mk, 1u);
            }
            mma_commit(bar);
        }
    }
    ok = mbar_wait_bounded(bar, (L::kSlabs - 1) & 1, p.status) && ok;
    tc_fence_after();

    // epilogue: TMEM lane r = 32 (warp % 4) + lane; warps 0-3 take D1 and D2,
    // warps 4-7 the D3 slabs
    const uint32_t tmem = *slot;
    const int r = 32 * (warp & 3) + (tid & 31);
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const float gc = r < DK ? sG[(BC - 1) * DK + r] : 0.f;
    const int part0 = warp < 4 ? 0 : 2, part1 = warp < 4 ? 2 : 2 + L::kSlabs;
#pragma unroll 1
    for (int part = part0; part < part1; ++part) {
#pragma unroll 1
        for (int tb = 0; tb < BC; tb += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + part * BC + tb, v);
            tmem_wait_ld();
            if (!ok) continue;
            if (part < 2) {
                if (r >= DK) continue;
                float *dst = (part == 0 ? p.pq : p.pk) + xk + r;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int t = tb + j;
                    if (t < n) {
                        const float g = sG[t * DK + r];
                        const float f = part == 0 ? p.scale * exp2f(g) : exp2f(gc - g);
                        dst[static_cast<size_t>(t) * DK] = f * __uint_as_float(v[j]);
                    }
                }
            } else {
                const int c = (part - 2) * SLAB + r;
                if (c >= DV) continue;
                float *dst = p.pv + xv + c;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (tb + j < n) dst[static_cast<size_t>(tb + j) * DV] = __uint_as_float(v[j]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::kCols);
}

// ---------------------------------------------------------------------------
// 4. the gradients on the tensor cores, one CTA per (chunk, head), for every
//    chunk whose decay span allows the reference split (the others are
//    flagged for kernels 5 and 6).  With M = 64 rows per product (row m of an
//    M = 64 accumulator sits in TMEM lane 32 (m / 16) + m % 16):
//       A  = dO V^T                 (K = dv)      masked to j <= t
//       M  = Qh Kh^T                (K = dk)      masked to j <= t
//       dQ = A Kh + dO S~^T,  dK = A^T Qh + V R~^T,  dV = M^T dO + Kh R~
//       with Qh = Q e^(Gamma - r), Kh = K e^(r - Gamma), S~ = 2^r S_u and
//       R~ = 2^(Gamma_C - r) R_u / scale (the state terms, K = dv or dk,
//       accumulated onto the in-chunk products in TMEM).
//    Every fp32-valued operand (Qh, Kh, A, M, S~, R~) is a bf16 hi/lo pair;
//    products of two pairs take the hi.hi, hi.lo and lo.hi terms.  The
//    epilogue scales dQ by scale 2^(Gamma - r), dK by scale 2^(r - Gamma), dV
//    by scale, writes dq, dk, dv and takes dlog_alpha.
constexpr int kIntraThreads = 256;

template <int DK, int DV>
struct IntraSmem {
    static constexpr uint32_t kBlk = BC * 128;              // one 64-column block of a 64-row tile
    static constexpr uint32_t kQh = 0, kQl = kQh + (DK / 64) * kBlk;
    static constexpr uint32_t kKh = kQl + (DK / 64) * kBlk, kKl = kKh + (DK / 64) * kBlk;
    static constexpr uint32_t kDo = kKl + (DK / 64) * kBlk, kV = kDo + (DV / 64) * kBlk;
    static constexpr uint32_t kAh = kV + (DV / 64) * kBlk, kAl = kAh + kBlk;
    static constexpr uint32_t kMh = kAl + kBlk, kMl = kMh + kBlk;
    static constexpr int LG = DK + 4;                       // fp32 prefix sums [BC][LG]
    static constexpr uint32_t kG = kMl + kBlk;
    static constexpr uint32_t kRef = kG + BC * LG * 4;      // reference, Gamma_C, carry: 3 x DK
    static constexpr uint32_t kBar = kRef + 3 * DK * 4;
    static constexpr uint32_t kSlot = kBar + 16;
    static constexpr uint32_t kBytes = kSlot + 16 + 1024;
    static constexpr int LP = DK + 1;                       // q dq - k dk, fp32 [BC][LP], over Qh..Kl
    // the gradient epilogue's raw q and k rows, bf16 [BC][DK] each, over the
    // dO, V and A/M tiles (free once the state products are done)
    static constexpr uint32_t kQr = kDo, kKr = kQr + BC * DK * 2;
    // TMEM columns used: A, M / dV first half [0, 128), dQ, dK, then dV's second half
    static constexpr uint32_t kUsed = 128 + 2 * DK + (DV > 128 ? 128 : 0);
    static constexpr uint32_t kCols = kUsed <= 256 ? 256 : 512;
    static_assert(BC * LP * 4 <= 4 * (DK / 64) * kBlk, "P fits over the q/k tiles");
    static_assert(kKr + BC * DK * 2 <= kMl + kBlk, "raw q, k fit over the dO, V and A/M tiles");
    // epilogue 2's staging rows (bf16 dq, dk and dv): dq and dk after the raw
    // rows where the dO, V and A/M tiles have room, dv after them or else past
    // P in the q/k tiles; without room for dq and dk (dk 128 with dv 64) those
    // two are stored from the rows' own threads
    static constexpr uint32_t kRawEnd = kKr + BC * DK * 2;
    static constexpr bool kStageQK = kRawEnd + 2 * BC * DK * 2 <= kMl + kBlk;
    static constexpr uint32_t kXqk = kRawEnd;
    static constexpr uint32_t kAfterQK = kStageQK ? kRawEnd + 2 * BC * DK * 2 : kRawEnd;
    static constexpr uint32_t kPEnd = (kQh + BC * LP * 4 + 15) & ~15u;
    static constexpr uint32_t kXv = kAfterQK + BC * DV * 2 <= kMl + kBlk ? kAfterQK : kPEnd;
    static_assert(kXv != kPEnd || kPEnd + BC * DV * 2 <= kDo, "the dv rows of epilogue 2 have room");
};

// Columns: A [0, 64), M [64, 128) first; then dV over [0, 128) (+ [2 dk + 128, ...) for
// its second half), dQ [128, 128 + dk), dK [128 + dk, 128 + 2 dk).
template <int DK, int DV>
__global__ void __launch_bounds__(kIntraThreads, 1) bwd_intra_kernel(BwdLaunch p) {
    using L = IntraSmem<DK, DV>;
    constexpr int NTI = kIntraThreads, LG = L::LG, LP = L::LP;
    constexpr int NTILE = DV / TW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *sG = reinterpret_cast<float *>(sm + L::kG);
    float *sRef = reinterpret_cast<float *>(sm + L::kRef), *sGC = sRef + DK, *sCarry = sGC + DK;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::kBar);
    uint32_t *slot = reinterpret_cast<uint32_t *>(sm + L::kSlot);
    const Chunk ck = chunk_at(p, blockIdx.x, blockIdx.y);
    const int u = ck.c, n = ck.n;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t rk = static_cast<size_t>(ck.row) * DK;   // first row, key-side tensors
    const size_t rv = static_cast<size_t>(ck.row) * DV;   // first row, value-side tensors
    const float s = p.scale;

    // loads first: the gates and the log-gate carries (the prefix sums need them
    // first), then q, k pairs and dO, V 16-byte groups; then the prefix sums
    float4 gr[BC * DK / 4 / NTI];
    prefix_issue<DK, NTI>(gr, p.log_alpha + rk, n);
    float cr[NTILE];
#pragma unroll
    for (int x = 0; x < NTILE; ++x)
        cr[x] = tid < DK ? p.carry[(static_cast<size_t>(ck.w.rbase + u) * NTILE + x) * DK + tid] : 0.f;
    constexpr int QPER = BC * DK / 2 / NTI, VPER = BC * DV / 8 / NTI;
    uint32_t qr[QPER], kr[QPER];
    uint4 dor[VPER], vr[VPER];
#pragma unroll
    for (int m = 0; m < QPER; ++m) {
        const int e = (tid + m * NTI) * 2, t = e / DK;
        qr[m] = t < n ? *reinterpret_cast<const uint32_t *>(p.q + rk + e) : 0u;
        kr[m] = t < n ? *reinterpret_cast<const uint32_t *>(p.k + rk + e) : 0u;
    }
#pragma unroll
    for (int m = 0; m < VPER; ++m) {
        const int e = tid + m * NTI, t = e / (DV / 8), c = (e % (DV / 8)) * 8;
        const size_t off = rv + static_cast<size_t>(t) * DV + c;
        dor[m] = t < n ? *reinterpret_cast<const uint4 *>(p.d_o + off) : make_uint4(0u, 0u, 0u, 0u);
        vr[m] = t < n ? *reinterpret_cast<const uint4 *>(p.v + off) : make_uint4(0u, 0u, 0u, 0u);
    }
    prefix_finish<DK, LG, NTI>(sG, gr);
    int wide = 0;
    if (tid < DK) {
        const float g0 = sG[tid], gl = sG[(BC - 1) * LG + tid];
        sRef[tid] = 0.5f * (g0 + gl);
        sGC[tid] = gl;
        wide = (g0 - gl) > kMaxSpan;
        float c = 0.f;
#pragma unroll
        for (int x = 0; x < NTILE; ++x) c += cr[x];
        sCarry[tid] = c;
    }
    const bool exact = __syncthreads_or(wide) || p.force_exact;
    if (tid == 0) p.wide[ck.w.rbase + u] = exact ? 1 : 0;
    if (exact) return;   // the CUDA-core kernel takes this chunk

    if (warp == 0) tmem_alloc(slot, L::kCols);
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar + 1, 1);   // the raw q, k rows of the epilogue
        fence_mbar_init();
    }
    // Qh, Kh (hi/lo) as [t][i] tiles; dO, V as [t][c] tiles
#pragma unroll
    for (int m = 0; m < QPER; ++m) {
        const int e = (tid + m * NTI) * 2, t = e / DK, i = e % DK;
        const float d0 = sG[t * LG + i] - sRef[i], d1 = sG[t * LG + i + 1] - sRef[i + 1];
        const float q0 = __uint_as_float(qr[m] << 16), q1 = __uint_as_float(qr[m] & 0xffff0000u);
        const float k0 = __uint_as_float(kr[m] << 16), k1 = __uint_as_float(kr[m] & 0xffff0000u);
        uint32_t hi, lo;
        const uint32_t off = sw128_offset(t, i, L::kBlk);
        split_pair(q0 * exp2f(d0), q1 * exp2f(d1), hi, lo);
        *reinterpret_cast<uint32_t *>(sm + L::kQh + off) = hi;
        *reinterpret_cast<uint32_t *>(sm + L::kQl + off) = lo;
        split_pair(k0 * exp2f(-d0), k1 * exp2f(-d1), hi, lo);
        *reinterpret_cast<uint32_t *>(sm + L::kKh + off) = hi;
        *reinterpret_cast<uint32_t *>(sm + L::kKl + off) = lo;
    }
#pragma unroll
    for (int m = 0; m < VPER; ++m) {
        const int e = tid + m * NTI, t = e / (DV / 8), c = (e % (DV / 8)) * 8;
        const uint32_t off = sw128_offset(t, c, L::kBlk);
        *reinterpret_cast<uint4 *>(sm + L::kDo + off) = dor[m];
        *reinterpret_cast<uint4 *>(sm + L::kV + off) = vr[m];
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t a0 = smem_u32(sm);
    // group 1: A and M
    if (tid == 0) {
        constexpr uint32_t id_a = idesc_bf16(64, BC, false, false);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
            const uint32_t o = (kk >> 2) * L::kBlk + (kk & 3) * 32;
            mma_bf16_ss(tmem, sw128_desc(a0 + L::kDo + o, 16, 1024), sw128_desc(a0 + L::kV + o, 16, 1024),
                        id_a, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
            const uint32_t o = (kk >> 2) * L::kBlk + (kk & 3) * 32;
            const uint64_t qh = sw128_desc(a0 + L::kQh + o, 16, 1024), ql = sw128_desc(a0 + L::kQl + o, 16, 1024);
            const uint64_t kh = sw128_desc(a0 + L::kKh + o, 16, 1024), kl = sw128_desc(a0 + L::kKl + o, 16, 1024);
            mma_bf16_ss(tmem + 64, qh, kh, id_a, kk > 0 ? 1u : 0u);
            mma_bf16_ss(tmem + 64, qh, kl, id_a, 1u);
            mma_bf16_ss(tmem + 64, ql, kh, id_a, 1u);
        }
        mma_commit(bar);
    }
    bool ok = mbar_wait_bounded(bar, 0, p.status);
    tc_fence_after();

    // epilogue 1: mask A and M to j <= t, split into bf16 pairs, [t][j] tiles.
    // Warp q (= warp % 4) holds rows 16 q .. 16 q + 15 in lanes 0-15 of its
    // quarter, read with the half-split load: thread = row t and 16 columns of
    // each 32-column block.  Warps 0-3 take A, warps 4-7 take M.
    {
        const int q4 = warp & 3, t = 16 * q4 + (lane & 15), hc = (lane >> 4) * 16;
        const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
        const int col = warp < 4 ? 0 : 64;
        uint8_t *th = sm + (warp < 4 ? L::kAh : L::kMh), *tl = sm + (warp < 4 ? L::kAl : L::kMl);
#pragma unroll 1
        for (int jb = 0; jb < BC; jb += 32) {
            uint32_t r[16];
            tmem_ld16x2<16>(tmem + lane_off + col + jb, r);
            tmem_wait_ld();
#pragma unroll
            for (int j8 = 0; j8 < 16; j8 += 8) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int jj = jb + hc + j8 + 2 * x;
                    const float x0 = (jj <= t) ? __uint_as_float(r[j8 + 2 * x]) : 0.f;
                    const float x1 = (jj + 1 <= t) ? __uint_as_float(r[j8 + 2 * x + 1]) : 0.f;
                    split_pair(x0, x1, hi[x], lo[x]);
                }
                const uint32_t off = sw128_offset(t, jb + hc + j8, L::kBlk);
                *reinterpret_cast<uint4 *>(th + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(tl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // group 2: dQ, dK, dV
    if (tid == 0) {
        constexpr uint32_t id_q = idesc_bf16(64, DK, false, true);   // A [t][j] K-major, Kh [j][i] MN-major
        constexpr uint32_t id_k = idesc_bf16(64, DK, true, true);    // A^T (MN-major), Qh [t][i] MN-major
        constexpr int NV = DV > 128 ? 128 : DV;
        constexpr uint32_t id_v = idesc_bf16(64, NV, true, true);    // M^T (MN-major), dO [t][c] MN-major
#pragma unroll
        for (int kk = 0; kk < BC / 16; ++kk) {
            const uint32_t ok_ = (kk & 3) * 32;          // K-major step inside the 64-column block
            const uint32_t om = kk * 2048;               // MN-major step: 16 rows
            const uint64_t ah = sw128_desc(a0 + L::kAh + ok_, 16, 1024), al = sw128_desc(a0 + L::kAl + ok_, 16, 1024);
            const uint64_t kh = sw128_desc(a0 + L::kKh + om, L::kBlk, 1024), kl = sw128_desc(a0 + L::kKl + om, L::kBlk, 1024);
            mma_bf16_ss(tmem + 128, ah, kh, id_q, kk > 0 ? 1u : 0u);
            mma_bf16_ss(tmem + 128, al, kh, id_q, 1u);
            mma_bf16_ss(tmem + 128, ah, kl, id_q, 1u);
            const uint64_t ath = sw128_desc(a0 + L::kAh + om, L::kBlk, 1024), atl = sw128_desc(a0 + L::kAl + om, L::kBlk, 1024);
            const uint64_t qh = sw128_desc(a0 + L::kQh + om, L::kBlk, 1024), ql = sw128_desc(a0 + L::kQl + om, L::kBlk, 1024);
            mma_bf16_ss(tmem + 128 + DK, ath, qh, id_k, kk > 0 ? 1u : 0u);
            mma_bf16_ss(tmem + 128 + DK, atl, qh, id_k, 1u);
            mma_bf16_ss(tmem + 128 + DK, ath, ql, id_k, 1u);
            const uint64_t mth = sw128_desc(a0 + L::kMh + om, L::kBlk, 1024), mtl = sw128_desc(a0 + L::kMl + om, L::kBlk, 1024);
#pragma unroll
            for (int hv = 0; hv < DV / NV; ++hv) {
                const uint32_t dcol = hv == 0 ? 0u : 128u + 2u * DK;
                const uint64_t db = sw128_desc(a0 + L::kDo + om + hv * 2 * L::kBlk, L::kBlk, 1024);
                mma_bf16_ss(tmem + dcol, mth, db, id_v, kk > 0 ? 1u : 0u);
                mma_bf16_ss(tmem + dcol, mtl, db, id_v, 1u);
            }
        }
        mma_commit(bar);
    }
    // the first state slab's loads fly while group 2 runs (group 3 below)
    constexpr uint32_t kSB = DK * 128;
    constexpr int SPER = DK * 64 / 4 / NTI;
    float4 sv[SPER], rr[SPER];
    auto fetch = [&](int c0) {
#pragma unroll
        for (int m = 0; m < SPER; ++m) {
            const int e = tid + m * NTI, i = e / 16, cl = (e % 16) * 4;
            sv[m] = *reinterpret_cast<const float4 *>(
                p.states + slot_index<DK, DV>(ck.w.sbase, i, c0 + cl, u));
            rr[m] = *reinterpret_cast<const float4 *>(
                p.adjoints + slot_index<DK, DV>(ck.w.rbase, i, c0 + cl, u));
        }
    };
    fetch(0);
    ok = mbar_wait_bounded(bar, 1, p.status) && ok;
    tc_fence_after();

    // group 3: the state terms, accumulated onto dQ, dK and dV, 64 value
    // columns at a time:  dQ += dO S~^T,  dK += V R~^T,  dV += Kh R~  with
    // S~ = 2^r S_u and R~ = 2^(Gamma_C - r) R_u / scale (bf16 pairs, [dk][64]
    // tiles), so that the epilogue's factors s 2^(Gamma - r), s 2^(r - Gamma)
    // and s apply to both terms.  The slab tiles take the place of the Qh and
    // A / M tiles, which the products above have finished reading.
    {
        uint8_t *tSh = sm + L::kQh, *tSl = tSh + kSB, *tRh = sm + L::kAh, *tRl = tRh + kSB;
        // each row's two factors, the same for every slab
        float fsv[SPER], frv[SPER];
#pragma unroll
        for (int m = 0; m < SPER; ++m) {
            const int i = (tid + m * NTI) / 16;
            fsv[m] = exp2f(sRef[i]);
            frv[m] = exp2f(sGC[i] - sRef[i]) / s;
        }
#pragma unroll 1
        for (int sl = 0; sl < DV / 64; ++sl) {
            const int c0 = sl * 64;
#pragma unroll
            for (int m = 0; m < SPER; ++m) {
                const int e = tid + m * NTI, i = e / 16, cl = (e % 16) * 4;
                const float fs = fsv[m], fr = frv[m];
                const uint32_t off = sw128_offset(i, cl, kSB);
                uint32_t h0, l0, h1, l1;
                split_pair(sv[m].x * fs, sv[m].y * fs, h0, l0);
                split_pair(sv[m].z * fs, sv[m].w * fs, h1, l1);
                *reinterpret_cast<uint2 *>(tSh + off) = make_uint2(h0, h1);
                *reinterpret_cast<uint2 *>(tSl + off) = make_uint2(l0, l1);
                split_pair(rr[m].x * fr, rr[m].y * fr, h0, l0);
                split_pair(rr[m].z * fr, rr[m].w * fr, h1, l1);
                *reinterpret_cast<uint2 *>(tRh + off) = make_uint2(h0, h1);
                *reinterpret_cast<uint2 *>(tRl + off) = make_uint2(l0, l1);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (sl + 1 < DV / 64) fetch(c0 + 64);   // the next slab in flight during the products
            if (tid == 0) {
                constexpr uint32_t id_qk3 = idesc_bf16(64, DK, false, false);   // [t][c] x [i][c]
                constexpr uint32_t id_v3 = idesc_bf16(64, BC, false, true);     // Kh [t][i] x R~ [i][c]
                const uint32_t aSh = smem_u32(tSh), aSl = smem_u32(tSl);
                const uint32_t aRh = smem_u32(tRh), aRl = smem_u32(tRl);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t o = kk * 32;
                    const uint64_t ado = sw128_desc(a0 + L::kDo + sl * L::kBlk + o, 16, 1024);
                    const uint64_t av = sw128_desc(a0 + L::kV + sl * L::kBlk + o, 16, 1024);
                    mma_bf16_ss(tmem + 128, ado, sw128_desc(aSh + o, 16, 1024), id_qk3, 1u);
                    mma_bf16_ss(tmem + 128, ado, sw128_desc(aSl + o, 16, 1024), id_qk3, 1u);
                    mma_bf16_ss(tmem + 128 + DK, av, sw128_desc(aRh + o, 16, 1024), id_qk3, 1u);
                    mma_bf16_ss(tmem + 128 + DK, av, sw128_desc(aRl + o, 16, 1024), id_qk3, 1u);
                }
                const uint32_t dcol = c0 < 128 ? static_cast<uint32_t>(c0)
                                               : 128u + 2u * DK + static_cast<uint32_t>(c0 - 128);
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t o = (kk >> 2) * L::kBlk + (kk & 3) * 32;
                    const uint64_t kh = sw128_desc(a0 + L::kKh + o, 16, 1024);
                    const uint64_t kl = sw128_desc(a0 + L::kKl + o, 16, 1024);
                    const uint64_t rh = sw128_desc(aRh + kk * 2048, kSB, 1024);
                    const uint64_t rl = sw128_desc(aRl + kk * 2048, kSB, 1024);
                    mma_bf16_ss(tmem + dcol, kh, rh, id_v3, 1u);
                    mma_bf16_ss(tmem + dcol, kl, rh, id_v3, 1u);
                    mma_bf16_ss(tmem + dcol, kh, rl, id_v3, 1u);
                }
                mma_commit(bar);
            }
            ok = mbar_wait_bounded(bar, (2 + sl) & 1, p.status) && ok;
            tc_fence_after();
        }
    }
    // every state product is done: the chunk's raw q and k rows load over the
    // dO, V and A/M tiles for the gradient epilogue, while the epilogue starts
    if (tid == 0) {
        const uint32_t bytes = static_cast<uint32_t>(n) * DK * 2;
        mbar_arrive_expect_tx(bar + 1, 2 * bytes);
        bulk_load(sm + L::kQr, p.q + rk, bytes, bar + 1);
        bulk_load(sm + L::kKr, p.k + rk, bytes, bar + 1);
    }
    __syncthreads();   // every thread is past the tile reads; P may overwrite the q/k tiles

    // epilogue 2.  Warps 0-3: row t of dQ and dK, q dq - k dk into P.  Warps
    // 4-7: row j of dV.  Thread = row t and 16 columns of each 32-column block
    // (half-split loads, as in epilogue 1).  The bf16 rows go through shared
    // memory (the V and A/M tiles, free by now; each warp its own 16 rows,
    // 16-byte pieces XOR-swizzled by row), so that each warp then stores
    // whole rows: a store instruction writes 512 contiguous bytes.
    float *sP = reinterpret_cast<float *>(sm + L::kQh);
    {
        const int q4 = warp & 3, r16 = lane & 15, t = 16 * q4 + r16, hc = (lane >> 4) * 16;
        const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
        const bool row_ok = ok && t < n;
        // the warp's staging rows and the offset of row r's 16-byte piece c
        uint8_t *xq = sm + L::kXqk + q4 * (2 * 16 * DK * 2), *xk = xq + 16 * DK * 2;
        uint8_t *xv = sm + L::kXv + q4 * (16 * DV * 2);
        auto piece = [](int r, int c, int row_bytes) { return r * row_bytes + ((c ^ (r & 7)) << 4); };
        if (warp < 4) {
            const float *grow = sG + t * LG;
            // this thread's q and k columns from the rows loaded above (rows
            // past n were not loaded; their results are not used)
            const bool qk_ok = mbar_wait_bounded(bar + 1, 0, p.status);
            const uint8_t *qrow = sm + L::kQr + t * DK * 2, *krow = sm + L::kKr + t * DK * 2;
            // rolled loops: this code runs once per CTA, so a small body that
            // stays in the instruction cache beats unrolled straight-line code
#pragma unroll 1
            for (int b = 0; b < DK / 32; ++b) {
                const int ib = b * 32;
                uint32_t rq[16], rkk[16];
                tmem_ld16x2<16>(tmem + lane_off + 128 + ib, rq);
                tmem_ld16x2<16>(tmem + lane_off + 128 + DK + ib, rkk);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 q4 = *reinterpret_cast<const uint4 *>(qrow + (b * 32 + hc + h * 8) * 2);
                    const uint4 k4 = *reinterpret_cast<const uint4 *>(krow + (b * 32 + hc + h * 8) * 2);
                    const uint32_t qw[4] = {q4.x, q4.y, q4.z, q4.w};
                    const uint32_t kw[4] = {k4.x, k4.y, k4.z, k4.w};
                    uint32_t dqw[4], dkw[4];
                    float pr[8];
#pragma unroll
                    for (int x = 0; x < 8; x += 2) {
                        const int j = h * 8 + x, i = ib + hc + j;
                        float dqv[2], dkv[2];
#pragma unroll
                        for (int y = 0; y < 2; ++y) {
                            const float d = grow[i + y] - sRef[i + y];
                            dqv[y] = s * exp2f(d) * __uint_as_float(rq[j + y]);
                            dkv[y] = s * exp2f(-d) * __uint_as_float(rkk[j + y]);
                        }
                        const float q0 = __uint_as_float(qw[x / 2] << 16), q1 = __uint_as_float(qw[x / 2] & 0xffff0000u);
                        const float k0 = __uint_as_float(kw[x / 2] << 16), k1 = __uint_as_float(kw[x / 2] & 0xffff0000u);
                        pr[x] = q0 * dqv[0] - k0 * dkv[0];
                        pr[x + 1] = q1 * dqv[1] - k1 * dkv[1];
                        dqw[x / 2] = pack_bf16x2(dqv[0], dqv[1]);
                        dkw[x / 2] = pack_bf16x2(dkv[0], dkv[1]);
                    }
                    const int i0 = ib + hc + h * 8;
                    if constexpr (L::kStageQK) {
                        *reinterpret_cast<uint4 *>(xq + piece(r16, i0 >> 3, DK * 2)) =
                            make_uint4(dqw[0], dqw[1], dqw[2], dqw[3]);
                        *reinterpret_cast<uint4 *>(xk + piece(r16, i0 >> 3, DK * 2)) =
                            make_uint4(dkw[0], dkw[1], dkw[2], dkw[3]);
                    } else if (row_ok && qk_ok) {
                        const size_t off = rk + static_cast<size_t>(t) * DK + i0;
                        *reinterpret_cast<uint4 *>(p.gq + off) = make_uint4(dqw[0], dqw[1], dqw[2], dqw[3]);
                        *reinterpret_cast<uint4 *>(p.gk + off) = make_uint4(dkw[0], dkw[1], dkw[2], dkw[3]);
                    }
#pragma unroll
                    for (int x = 0; x < 8; ++x) sP[t * LP + i0 + x] = row_ok && qk_ok ? pr[x] : 0.f;
                }
            }
            __syncwarp();
            const bool wok = __all_sync(0xffffffffu, ok && qk_ok);
#pragma unroll
            for (int m = 0; m < (L::kStageQK ? 16 * DK / 8 / 32 : 0); ++m) {
                const int e = lane + 32 * m, r = e / (DK / 8), c = e % (DK / 8);
                if (wok && 16 * q4 + r < n) {
                    const size_t off = rk + static_cast<size_t>(16 * q4 + r) * DK + c * 8;
                    *reinterpret_cast<uint4 *>(p.gq + off) = *reinterpret_cast<const uint4 *>(xq + piece(r, c, DK * 2));
                    *reinterpret_cast<uint4 *>(p.gk + off) = *reinterpret_cast<const uint4 *>(xk + piece(r, c, DK * 2));
                }
            }
        } else {
#pragma unroll 1
            for (int cb = 0; cb < DV; cb += 32) {
                const uint32_t dcol = cb < 128 ? static_cast<uint32_t>(cb) : 128u + 2u * DK + (cb - 128);
                uint32_t rv_[16];
                tmem_ld16x2<16>(tmem + lane_off + dcol, rv_);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; j += 8) {
                    uint32_t w[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        w[x] = pack_bf16x2(s * __uint_as_float(rv_[j + 2 * x]), s * __uint_as_float(rv_[j + 2 * x + 1]));
                    *reinterpret_cast<uint4 *>(xv + piece(r16, (cb + hc + j) >> 3, DV * 2)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            __syncwarp();
            const bool wok = __all_sync(0xffffffffu, ok);
#pragma unroll
            for (int m = 0; m < 16 * DV / 8 / 32; ++m) {
                const int e = lane + 32 * m, r = e / (DV / 8), c = e % (DV / 8);
                if (wok && 16 * q4 + r < n)
                    *reinterpret_cast<uint4 *>(p.gv + rv + static_cast<size_t>(16 * q4 + r) * DV + c * 8) =
                        *reinterpret_cast<const uint4 *>(xv + piece(r, c, DV * 2));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::kCols);
    // dlog_alpha = carry + reverse in-chunk sum of q dq - k dk (16 rows' loads
    // in flight at a time; rows past n hold zeros and are not stored)
    if (tid < DK) {
        float acc = sCarry[tid];
#pragma unroll
        for (int t1 = BC; t1 > 0; t1 -= 16) {
            float x[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) x[j] = sP[(t1 - 1 - j) * LP + tid];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int t = t1 - 1 - j;
                if (t < n) {
                    acc += x[j];
                    p.ga[rk + static_cast<size_t>(t) * DK + tid] = acc;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// 6. per-chunk gradients on CUDA cores, for the chunks the tensor-core kernel
//    leaves (decay span beyond the reference split, or force_exact): every
//    in-chunk decay factor e^(Gamma_t - Gamma_j) is its own exponential.
//    Thread (ty, tx) = (tid / 16, tid % 16) owns rows 4 ty .. 4 ty + 3 and
//    columns tx, tx + 16, ... of every C x C, C x dk and C x 32 block it
//    computes.  (Kernels appear in this file in the order 1, 2, 5, 4, 6; the
//    numbers are the launch order.)
template <int DK>
struct GradSmem {
    static constexpr int LD = DK + 1;      // odd strides: conflict-free column walks
    static constexpr int LA = BC + 1;
    static constexpr int LS = TW + 1;
    static constexpr int kG = 0, kQ = kG + BC * LD, kK = kQ + BC * LD, kP = kK + BC * LD;
    static constexpr int kAM = kP + BC * LD;
    static constexpr int kDo = kAM + BC * LA, kV = kDo + BC * LS;
    static constexpr int kCarry = kV + BC * LS;
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
    float *sCarry = smem + L::kCarry;

    const Chunk ck = chunk_at(p, blockIdx.x, blockIdx.y);
    const int u = ck.c, n = ck.n;
    if (!p.wide[ck.w.rbase + u]) return;   // done by the tensor-core kernel
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    // first rows of the caller's tensors; the partials use the same offsets
    const size_t rk = static_cast<size_t>(ck.row) * DK, rv = static_cast<size_t>(ck.row) * DV;
    const size_t xk = rk, xv = rv;
    const float s = p.scale;

    // the state terms of dq and dk (bwd_inter), fetched early for phase 2
    float pq[4][NB], pk[4][NB];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int t = 4 * ty + a;
            const size_t off = xk + static_cast<size_t>(t) * DK + tx + 16 * b;
            pq[a][b] = t < n ? p.pq[off] : 0.f;
            pk[a][b] = t < n ? p.pk[off] : 0.f;
        }

    // prefix sums and the log-gate carry
    load_prefix<DK, LD>(sG, p.log_alpha + rk, n);
    if (tid < DK) {
        float c = 0.f;
        for (int x = 0; x < NTILE; ++x)
            c += p.carry[(static_cast<size_t>(ck.w.rbase + u) * NTILE + x) * DK + tid];
        sCarry[tid] = c;
    }

    // q and k as they are: every decay factor below is its own exponential
    {
        constexpr int PER = BC * DK / 2 / NT;
        uint32_t qr[PER], kr[PER];
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            const int e = (tid + m * NT) * 2, t = e / DK;
            const size_t off = rk + static_cast<size_t>(e);
            qr[m] = t < n ? *reinterpret_cast<const uint32_t *>(p.q + off) : 0u;
            kr[m] = t < n ? *reinterpret_cast<const uint32_t *>(p.k + off) : 0u;
        }
#pragma unroll
        for (int m = 0; m < PER; ++m) {
            const int e = (tid + m * NT) * 2, t = e / DK, i = e % DK;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                sQ[t * LD + i + h] = __uint_as_float(h ? (qr[m] & 0xffff0000u) : (qr[m] << 16));
                sK[t * LD + i + h] = __uint_as_float(h ? (kr[m] & 0xffff0000u) : (kr[m] << 16));
            }
        }
    }

    // phase 1: A = dO V^T, streaming the value columns; the next slice's loads
    // are in flight while the current slice is multiplied
    float accA[4][4] = {};
    {
        constexpr int PV = BC * TW / NT;
        float dov[PV], vv[PV];
        auto fetch = [&](int c0) {
#pragma unroll
            for (int m = 0; m < PV; ++m) {
                const int e = tid + m * NT, t = e / TW, c = e % TW;
                const size_t off = rv + static_cast<size_t>(t) * DV + c0 + c;
                dov[m] = t < n ? bf(p.d_o, off) : 0.f;
                vv[m] = t < n ? bf(p.v, off) : 0.f;
            }
        };
        fetch(0);
        for (int c0 = 0; c0 < DV; c0 += TW) {
            __syncthreads();
#pragma unroll
            for (int m = 0; m < PV; ++m) {
                const int e = tid + m * NT, t = e / TW, c = e % TW;
                sDo[t * LS + c] = dov[m];
                sV[t * LS + c] = vv[m];
            }
            __syncthreads();
            if (c0 + TW < DV) fetch(c0 + TW);
#pragma unroll 4
            for (int c = 0; c < TW; ++c) {
                float dr[4], vj[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    dr[a] = sDo[(4 * ty + a) * LS + c];
                    vj[a] = sV[(tx + 16 * a) * LS + c];
                }
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) accA[a][b] = fmaf(dr[a], vj[b], accA[a][b]);
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
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int i = tx + 16 * b;
            const float dq = s * iq[b] + pq[a][b];
            const float dk = s * ik[b] + pk[a][b];
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
                for (int i = 0; i < DK; ++i)
                    m = fmaf(sQ[t * LD + i] * sK[j * LD + i], exp2f(sG[t * LD + i] - sG[j * LD + i]), m);
            }
            accA[a][b] = s * m;
        }
    }
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) sAM[(4 * ty + a) * LA + tx + 16 * b] = accA[a][b];
    // phase 4: dV = M^T dO + the state term (bwd_inter), a slice of value
    // columns at a time, the next slice's loads in flight
    {
        constexpr int PV = BC * TW / NT;
        float dov[PV], pvv[4][2];
        auto fetch = [&](int c0) {
#pragma unroll
            for (int m = 0; m < PV; ++m) {
                const int e = tid + m * NT, t = e / TW, c = e % TW;
                dov[m] = t < n ? bf(p.d_o, rv + static_cast<size_t>(t) * DV + c0 + c) : 0.f;
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int j = 4 * ty + a;
                const size_t off = xv + static_cast<size_t>(j) * DV + c0 + tx;
                pvv[a][0] = j < n ? p.pv[off] : 0.f;
                pvv[a][1] = j < n ? p.pv[off + 16] : 0.f;
            }
        };
        fetch(0);
        for (int c0 = 0; c0 < DV; c0 += TW) {
            __syncthreads();
#pragma unroll
            for (int m = 0; m < PV; ++m) {
                const int e = tid + m * NT;
                sDo[(e / TW) * LS + e % TW] = dov[m];
            }
            float acc[4][2];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                acc[a][0] = pvv[a][0];
                acc[a][1] = pvv[a][1];
            }
            __syncthreads();
            if (c0 + TW < DV) fetch(c0 + TW);
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int j = 4 * ty + a;
                for (int x = j; x < BC; ++x) {
                    const float mxj = sAM[x * LA + j];
                    acc[a][0] = fmaf(mxj, sDo[x * LS + tx], acc[a][0]);
                    acc[a][1] = fmaf(mxj, sDo[x * LS + tx + 16], acc[a][1]);
                }
                if (j < n) {
                    const size_t off = rv + static_cast<size_t>(j) * DV + c0;
                    p.gv[off + tx] = __float2bfloat16_rn(acc[a][0]);
                    p.gv[off + tx + 16] = __float2bfloat16_rn(acc[a][1]);
                }
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

// ---------------------------------------------------------------------------
// One gate per token and head: the backward runs on the gate broadcast to
// every key channel, and the head gate's gradient is the sum of the channel
// gates' gradients (each channel's gate is the same input).
template <int DK>
__global__ void __launch_bounds__(256) bwd_gate_broadcast_kernel(const float *__restrict__ g,
                                                                 float *__restrict__ full,
                                                                 long long rows) {
    const long long e = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;   // float4 index
    if (e >= rows * (DK / 4)) return;
    const float x = g[e / (DK / 4)];
    reinterpret_cast<float4 *>(full)[e] = make_float4(x, x, x, x);
}

template <int DK>
__global__ void __launch_bounds__(256) bwd_gate_sum_kernel(const float *__restrict__ full,
                                                           float *__restrict__ g, long long rows) {
    const long long r = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
    if (r >= rows) return;
    const float4 *src = reinterpret_cast<const float4 *>(full + r * DK);
    float acc = 0.f;
#pragma unroll 8
    for (int m = 0; m < DK / 4; ++m) {
        const float4 v = src[m];
        acc += (v.x + v.y) + (v.z + v.w);
    }
    g[r] = acc;
}

template <int DK, int DV>
int launch_bwd_dims(const BwdLaunch &p, cudaStream_t stream) {
    const size_t sum_bytes = SumSmem<DK, DV>::kBytes;
    const size_t grad_bytes = GradSmem<DK>::kBytes;
    const size_t inter_bytes = InterSmem<DK, DV>::kBytes;
    const size_t intra_bytes = IntraSmem<DK, DV>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(bwd_sums_kernel<DK, DV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sum_bytes));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_intra_kernel<DK, DV>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(intra_bytes));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_inter_kernel<DK, DV>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(inter_bytes));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_grads_kernel<DK, DV>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(grad_bytes));
    if (e != cudaSuccess) return static_cast<int>(e);
    const unsigned scan_blocks =
        static_cast<unsigned>(static_cast<size_t>(p.N) * p.H * DK * DV / 256);
    const unsigned nchunks = static_cast<unsigned>(p.chunks);
    if (nchunks == 0) {   // only empty sequences: dh0 = dhT (the scans walk no chunk)
        bwd_state_scan_kernel<DK, DV><<<scan_blocks, 256, 0, stream>>>(p);
        bwd_adjoint_scan_kernel<DK, DV><<<scan_blocks, 256, 0, stream>>>(p);
        return static_cast<int>(cudaGetLastError());
    }
    // chunk sums: persistent CTAs, as many as fit on the GPU at once
    const long long items = 2LL * p.chunks * p.H;
    int dev = 0, sms = 0, per_sm = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bwd_sums_kernel<DK, DV>,
                                                          kSumAllThreads, sum_bytes);
    if (e != cudaSuccess) return static_cast<int>(e);
    const long long slots = static_cast<long long>(sms) * (per_sm > 0 ? per_sm : 1);
    const unsigned sum_grid = static_cast<unsigned>(items < slots ? items : slots);
    bwd_sums_kernel<DK, DV><<<sum_grid, kSumAllThreads, sum_bytes, stream>>>(p, items);
    bwd_state_scan_kernel<DK, DV><<<scan_blocks, 256, 0, stream>>>(p);
    bwd_adjoint_scan_kernel<DK, DV><<<scan_blocks, 256, 0, stream>>>(p);
    bwd_intra_kernel<DK, DV><<<dim3(nchunks, p.H), kIntraThreads, intra_bytes, stream>>>(p);
    bwd_inter_kernel<DK, DV><<<dim3(nchunks, p.H), kInterThreads, inter_bytes, stream>>>(p);
    bwd_grads_kernel<DK, DV><<<dim3(nchunks, p.H), NT, grad_bytes, stream>>>(p);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace

int bwd_chunk_tokens() { return BC; }
int bwd_value_tiles(int dv) { return dv / TW; }

int launch_gate_broadcast(const float *g, float *full, long long rows, int dk, cudaStream_t stream) {
    const long long n = rows * (dk / 4);
    const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
    if (dk == 64) bwd_gate_broadcast_kernel<64><<<blocks, 256, 0, stream>>>(g, full, rows);
    else bwd_gate_broadcast_kernel<128><<<blocks, 256, 0, stream>>>(g, full, rows);
    return static_cast<int>(cudaGetLastError());
}

int launch_gate_sum(const float *full, float *g, long long rows, int dk, cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>((rows + 255) / 256);
    if (dk == 64) bwd_gate_sum_kernel<64><<<blocks, 256, 0, stream>>>(full, g, rows);
    else bwd_gate_sum_kernel<128><<<blocks, 256, 0, stream>>>(full, g, rows);
    return static_cast<int>(cudaGetLastError());
}

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
