// gla_decode.cu — one recurrent decode step for many independent heads.
//
// Per head (source: "Gated Linear Attention (GLA): Mathematical Foundations,
// ..." (llms.blog), section "The Gated Recurrent Update"):
//     h <- diag(exp(log_alpha)) h + k^T v,     o = scale * q h   (updated h)
//
// The step is a pure stream of the fp32 state: 8*dk*dv bytes per head (read +
// write) against 5*dk*dv flops, so it is HBM-bound.  One CTA per head; each
// thread owns one 16-byte column group of `rows_per_thread` state rows chosen
// so that every warp-wide load covers whole 512-byte runs of a row (fully
// coalesced).  All of a thread's state loads are issued before any use so a
// CTA keeps its whole 64 KB head in flight.  The dk-reduction of q*h runs in
// registers, then across the lanes that share a column group with warp
// shuffles, then across warps through shared memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gla_internal.h"

namespace gla {
namespace {

template <int DK, int DV>
struct DecodeShape {
    static constexpr int kThreads = DV > 128 ? 512 : 256;
    static constexpr int kGroups = DV / 4;                   // float4 column groups per row
    static constexpr int kRowBases = kThreads / kGroups;     // threads sharing one column group
    static constexpr int kRowsPerThread = DK / kRowBases;
    static constexpr int kWarps = kThreads / 32;
    static_assert(DK % kRowBases == 0, "rows must divide evenly");
};

template <int DK, int DV>
__global__ void __launch_bounds__(DecodeShape<DK, DV>::kThreads)
    recurrent_step_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                          const __nv_bfloat16 *__restrict__ v, const float *__restrict__ log_alpha,
                          float scale, float *__restrict__ h, __nv_bfloat16 *__restrict__ o) {
    using Sh = DecodeShape<DK, DV>;
    constexpr int G = Sh::kGroups, RB = Sh::kRowBases, RPT = Sh::kRowsPerThread;
    const int bh = blockIdx.x;
    const int tid = threadIdx.x;
    const int cg = tid % G;   // column group: columns 4cg .. 4cg+3
    const int rb = tid / G;   // rows rb, rb + RB, rb + 2 RB, ...

    float4 *hs = reinterpret_cast<float4 *>(h + static_cast<size_t>(bh) * DK * DV);

    // 1. put the whole state tile of this thread in flight.
    float4 s[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m) s[m] = __ldcs(hs + (rb + m * RB) * G + cg);

    // 2. the small per-head vectors.
    __shared__ float s_q[DK], s_k[DK], s_a[DK];
    __shared__ float4 s_red[Sh::kWarps][G < 32 ? G : 32];
    if (tid < DK) {
        const size_t i = static_cast<size_t>(bh) * DK + tid;
        s_q[tid] = __bfloat162float(q[i]);
        s_k[tid] = __bfloat162float(k[i]);
        s_a[tid] = expf(log_alpha[i]);
    }
    const uint2 vraw = *reinterpret_cast<const uint2 *>(v + static_cast<size_t>(bh) * DV + 4 * cg);
    const __nv_bfloat162 v01 = *reinterpret_cast<const __nv_bfloat162 *>(&vraw.x);
    const __nv_bfloat162 v23 = *reinterpret_cast<const __nv_bfloat162 *>(&vraw.y);
    const float4 vv = make_float4(__low2float(v01), __high2float(v01), __low2float(v23),
                                  __high2float(v23));
    __syncthreads();

    // 3. update in registers, write back, and accumulate q * h' over this thread's rows.
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int d = rb + m * RB;
        const float a = s_a[d], kd = s_k[d], qd = s_q[d];
        float4 t = s[m];
        t.x = fmaf(a, t.x, kd * vv.x);
        t.y = fmaf(a, t.y, kd * vv.y);
        t.z = fmaf(a, t.z, kd * vv.z);
        t.w = fmaf(a, t.w, kd * vv.w);
        __stcs(hs + d * G + cg, t);
        acc.x = fmaf(qd, t.x, acc.x);
        acc.y = fmaf(qd, t.y, acc.y);
        acc.z = fmaf(qd, t.z, acc.z);
        acc.w = fmaf(qd, t.w, acc.w);
    }

    // 4. reduce over the rows: lanes of a warp that share a column group first ...
    const int lane = tid & 31, warp = tid >> 5;
    if constexpr (G < 32) {
#pragma unroll
        for (int off = G; off < 32; off <<= 1) {
            acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
            acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
            acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
            acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
        }
        if (lane < G) s_red[warp][lane] = acc;
    } else {
        s_red[warp][lane] = acc;  // warp covers columns groups (warp % (G/32))*32 + lane
    }
    __syncthreads();

    // ... then across warps.
    if (tid < G) {
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        constexpr int kWarpsPerGroupSet = (G < 32) ? Sh::kWarps : Sh::kWarps / (G / 32);
#pragma unroll
        for (int w = 0; w < kWarpsPerGroupSet; ++w) {
            const float4 x = (G < 32) ? s_red[w][tid] : s_red[w * (G / 32) + tid / 32][tid % 32];
            r.x += x.x;
            r.y += x.y;
            r.z += x.z;
            r.w += x.w;
        }
        uint2 out;
        out.x = [&] {
            __nv_bfloat162 p = __floats2bfloat162_rn(scale * r.x, scale * r.y);
            return *reinterpret_cast<uint32_t *>(&p);
        }();
        out.y = [&] {
            __nv_bfloat162 p = __floats2bfloat162_rn(scale * r.z, scale * r.w);
            return *reinterpret_cast<uint32_t *>(&p);
        }();
        *reinterpret_cast<uint2 *>(o + static_cast<size_t>(bh) * DV + 4 * tid) = out;
    }
}

template <int DK, int DV>
int launch_dk_dv(const DecodeLaunch &p, cudaStream_t stream) {
    using Sh = DecodeShape<DK, DV>;
    recurrent_step_kernel<DK, DV><<<p.BH, Sh::kThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(p.q), static_cast<const __nv_bfloat16 *>(p.k),
        static_cast<const __nv_bfloat16 *>(p.v), p.log_alpha, p.scale, p.h,
        static_cast<__nv_bfloat16 *>(p.o));
    return static_cast<int>(cudaGetLastError());
}

}  // namespace

int launch_recurrent_step(const DecodeLaunch &p, cudaStream_t stream) {
    if (p.dk == 64) {
        if (p.dv == 64) return launch_dk_dv<64, 64>(p, stream);
        if (p.dv == 128) return launch_dk_dv<64, 128>(p, stream);
        if (p.dv == 256) return launch_dk_dv<64, 256>(p, stream);
    } else if (p.dk == 128) {
        if (p.dv == 64) return launch_dk_dv<128, 64>(p, stream);
        if (p.dv == 128) return launch_dk_dv<128, 128>(p, stream);
        if (p.dv == 256) return launch_dk_dv<128, 256>(p, stream);
    }
    return static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace gla
