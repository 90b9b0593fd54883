// gla_api.cu — the C ABI declared in include/gla.h: host-side validation,
// device checks, TMA tensor-map encoding and kernel dispatch.
//
// Nothing here computes any part of the method; every step of the forward
// and of the decode step runs in the kernels of gla_chunk.cu / gla_decode.cu.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <algorithm>
#include <mutex>
#include <vector>

#include "gla.h"
#include "gla_internal.h"

namespace gla {

__device__ unsigned int g_device_status = 0u;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int sm_count = 1;
    unsigned int *status = nullptr;  // device address of g_device_status
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Current device, checked to be sm_103 (GB300).  Returns a GLA status.
int current_device(DeviceInfo **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GLA_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &info = g_devices[dev];
    if (!info.probed) {
        info.probed = true;
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
            cudaGetLastError();
            return GLA_ERR_DEVICE;
        }
        info.supported = (prop.major == 10 && prop.minor == 3);
        info.sm_count = prop.multiProcessorCount;
        if (info.supported) {
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) {
                cudaGetLastError();
                info.supported = false;
            } else {
                info.status = static_cast<unsigned int *>(addr);
            }
        }
    }
    if (!info.supported) return GLA_ERR_DEVICE;
    *out = &info;
    return GLA_OK;
}

int encode_fn(EncodeTiledFn *fn) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p) {
            cudaGetLastError();
            return GLA_ERR_DEVICE;
        }
        g_encode = reinterpret_cast<EncodeTiledFn>(p);
    }
    *fn = g_encode;
    return GLA_OK;
}

// 3-D tensor map over a [BH, T, C] row-major tensor: dims (C, T, BH).
bool make_map(EncodeTiledFn enc, CUtensorMap *m, const void *ptr, CUtensorMapDataType dt,
              int elem_bytes, int C, int T, int BH, int box_c, int box_t,
              CUtensorMapSwizzle swz) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(T),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(C) * elem_bytes,
                             static_cast<cuuint64_t>(C) * elem_bytes * static_cast<cuuint64_t>(T)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_c), static_cast<cuuint32_t>(box_t), 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Plan {
    int dv_tile;
    bool pair;      // the two value-column tiles of a head run as a 2-CTA cluster
    int NC;         // chunks (of 128 tokens) per sequence
    int L;          // chunks per range of the work split
    int W;          // ranges: CTAs (clusters, for pairs) of the FULL pass per tile column
    int seg_max;    // most segments a sequence is cut into
};

constexpr int kMinRange = 16;   // shortest automatic range, in chunks

// Segments of sequence u when ranges of L chunks tile all sequences' chunks
// (the same arithmetic as the kernel's).
int nseg_host(long long u, int NC, int L) {
    const long long a = u * NC;
    return 1 + static_cast<int>((a + NC - 1) / L - a / L);
}

// Launch plan of gla_chunk_fwd: value-column tile, CTA pairs, work split.
// Pairs: with dk = 128 and exactly two value-column tiles, the tiles of a head
// share the key-side preparation (each CTA prepares one half of the channels).
// Work split: when there are fewer sequences than CTAs that can run at once,
// the chunks of all sequences, one after another, are cut into equal ranges,
// one per resident CTA (or cluster), so that every SM has the same work; a
// cut inside a sequence makes a new segment of it, joined by the state
// correction.  Ranges stay at least kMinRange chunks long, so that the
// correction windows stay a small part of the work.
size_t scratch_needed(const Plan &pl, int B, int H, int dk, int dv);

// scratch_cap: bytes of segment scratch available (SIZE_MAX: allocated to
// fit).  An automatic plan whose segments would need more takes longer
// ranges, down to one range per sequence (no scratch).
Plan make_plan(int B, int H, int T, int dk, int dv, const gla_chunk_options &op, int sm_count,
               size_t scratch_cap = SIZE_MAX) {
    Plan pl;
    pl.dv_tile = op.dv_tile ? op.dv_tile : (dv >= 128 ? 128 : 64);
    pl.pair = dk == 128 && dv == 2 * pl.dv_tile && op.cta_pair >= 0;
    const long long BH = static_cast<long long>(B) * H;
    pl.NC = (T + 127) / 128;
    const long long total = BH * pl.NC;
    long long L;
    if (op.segments > 0) {
        L = (pl.NC + op.segments - 1) / op.segments;
    } else {
        const int n_dvt = dv / pl.dv_tile;
        int resident = gla::chunk_fwd_max_resident(dk, pl.dv_tile, pl.pair ? 1 : 0);
        if (resident <= 0) resident = pl.pair ? sm_count / 2 : sm_count;
        const long long ranges = pl.pair ? resident : resident / n_dvt;
        if (ranges <= BH) {
            L = pl.NC;   // enough sequences: one per CTA, none cut
        } else if (pl.pair) {
            // CTA pairs: whole-number segments per sequence.  Measured on the
            // GB300, a pair kernel's chunk rate does not grow with more
            // clusters than that (the extra clusters only add correction work).
            const long long per = ranges / BH;
            L = (pl.NC + per - 1) / per;
            if (L < kMinRange) L = std::min<long long>(kMinRange, pl.NC);
        } else {
            L = (total + ranges - 1) / ranges;
            if (L < kMinRange) L = kMinRange;
            if (L > pl.NC) L = pl.NC;
        }
    }
    if (L < 1) L = 1;
    while (true) {
        pl.L = static_cast<int>(L);
        pl.W = static_cast<int>((total + L - 1) / L);
        pl.seg_max = 1;
        if (pl.L < pl.NC)
            for (long long u = 0; u < BH; ++u)
                pl.seg_max = std::max(pl.seg_max, nseg_host(u, pl.NC, pl.L));
        if (op.segments > 0 || pl.seg_max == 1 || scratch_needed(pl, B, H, dk, dv) <= scratch_cap)
            return pl;
        L = std::min<long long>(2 * L, pl.NC);
    }
}

bool options_ok(int dv, const gla_chunk_options &op) {
    if (op.dv_tile != 0 && op.dv_tile != 64 && op.dv_tile != 128) return false;
    if (op.dv_tile > dv || op.segments < 0) return false;
    if (op.gate_per_head != 0 && op.gate_per_head != 1) return false;
    return op.cta_pair >= -1 && op.cta_pair <= 1;
}

size_t scratch_needed(const Plan &pl, int B, int H, int dk, int dv) {
    return pl.seg_max > 1
               ? static_cast<size_t>(pl.seg_max) * B * H * dk * (dv + 1) * sizeof(float)
               : 0;
}

bool dk_ok(int dk) { return dk == 64 || dk == 128; }
bool dv_ok(int dv) { return dv == 64 || dv == 128 || dv == 256; }

}  // namespace

int chunk_fwd_with_scratch(const void *q, const void *k, const void *v, const float *log_alpha,
                           float scale, const float *h0, void *o, float *hT, int B, int H, int T,
                           int dk, int dv, const gla_chunk_options *opts, cudaStream_t stream,
                           void *scratch, size_t scratch_bytes, const gla_chunk_debug *dbg) {
    if (!q || !k || !v || !log_alpha || !o) return GLA_ERR_ARG;
    if (B <= 0 || H <= 0 || T <= 0) return GLA_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) ||
        !aligned16(o) || (h0 && !aligned16(h0)) || (hT && !aligned16(hT)))
        return GLA_ERR_ARG;
    if (!dk_ok(dk) || !dv_ok(dv)) return GLA_ERR_SHAPE;
    gla_chunk_options o_def = {};
    const gla_chunk_options &op = opts ? *opts : o_def;
    if (!options_ok(dv, op)) return GLA_ERR_ARG;
    if (static_cast<long long>(B) * H > 0x7fffffffLL) return GLA_ERR_ARG;
    if (scratch && !aligned16(scratch)) return GLA_ERR_ARG;
    if (dbg && (dbg->withhold_v < 0 || (dbg->gamma && !aligned16(dbg->gamma)))) return GLA_ERR_ARG;
    // the instrumented kernel build covers one gate per key channel only
    if (dbg && opts && opts->gate_per_head) return GLA_ERR_ARG;

    DeviceInfo *dev = nullptr;
    int st = current_device(&dev);
    if (st != GLA_OK) return st;
    EncodeTiledFn enc = nullptr;
    st = encode_fn(&enc);
    if (st != GLA_OK) return st;

    const int BH = B * H;
    const Plan pl =
        make_plan(B, H, T, dk, dv, op, dev->sm_count, scratch ? scratch_bytes : SIZE_MAX);
    const size_t state_bytes =
        pl.seg_max > 1 ? static_cast<size_t>(pl.seg_max) * BH * dk * dv * sizeof(float) : 0;
    const size_t decay_bytes =
        pl.seg_max > 1 ? static_cast<size_t>(pl.seg_max) * BH * dk * sizeof(float) : 0;
    if (state_bytes + decay_bytes > (scratch ? scratch_bytes : 0)) return GLA_ERR_SCRATCH;

    ChunkLaunch p = {};
    // with one gate per token the kernel reads the gates itself (no A map)
    if (!make_map(enc, &p.tm_q, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dk, T, BH, 64, 128,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(enc, &p.tm_k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dk, T, BH, 64, 128,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        (!op.gate_per_head &&
         !make_map(enc, &p.tm_a, log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dk, T, BH,
                   pl.pair ? dk / 2 : dk, 128, CU_TENSOR_MAP_SWIZZLE_NONE)) ||
        !make_map(enc, &p.tm_v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dv, T, BH, 64, 128,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(enc, &p.tm_o32, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dv, T, BH, 64, 32,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return GLA_ERR_LAUNCH;
    p.q = q;
    p.k = k;
    p.log_alpha = log_alpha;
    p.h0 = h0;
    p.hT = hT;
    p.o = o;
    // Every scratch entry a launch reads is written earlier in the same call,
    // so nothing in it needs to start at zero.
    p.ws_state = pl.seg_max > 1 ? static_cast<float *>(scratch) : nullptr;
    p.ws_decay = pl.seg_max > 1
                     ? reinterpret_cast<float *>(static_cast<char *>(scratch) + state_bytes)
                     : nullptr;
    p.scale = scale;
    p.B = B;
    p.H = H;
    p.T = T;
    p.dk = dk;
    p.dv = dv;
    p.dv_tile = pl.dv_tile;
    p.pair = pl.pair ? 1 : 0;
    p.NC = pl.NC;
    p.L = pl.L;
    p.W = pl.W;
    p.seg_max = pl.seg_max;
    p.total = static_cast<long long>(BH) * pl.NC;
    p.seqs = nullptr;
    p.NS = 0;
    p.gate_per_head = op.gate_per_head;
    p.force_exact = op.force_exact ? 1 : 0;
    // two segments per sequence, each range one whole segment: the first
    // segment's CTA pair corrects the second segment's window itself
    p.fuse = (pl.pair && pl.seg_max == 2 && pl.NC % pl.L == 0 && pl.NC / pl.L == 2) ? 1 : 0;
    p.status = dev->status;
    if (dbg) {
        p.debug = 1;
        p.wait_ns = static_cast<unsigned long long>(dbg->wait_limit_us) * 1000ull;
        p.dbg_gamma = dbg->gamma;
        p.dbg_blk = dbg->block_len;
        p.withhold_v = dbg->withhold_v;
    }
    return launch_chunk_fwd(p, stream) == 0 ? GLA_OK : GLA_ERR_LAUNCH;
}

// ---------------------------------------------------------------- packed batches

namespace {

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Packed variable-length batch: per sequence n, {first row, length, chunks,
// chunk offset}, and the chunks of one head in all.
struct Packed {
    std::vector<int4> seqs;
    long long chunks = 0;
    int max_chunks = 0;
};

// Checks cu_seqlens (N + 1 offsets, from 0 to T_total, nondecreasing) and
// builds the sequence table.  Returns a GLA status.
int packed_layout(const int *cu_seqlens, int N, int T_total, Packed *pk) {
    if (!cu_seqlens || N <= 0 || T_total < 0) return GLA_ERR_ARG;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T_total) return GLA_ERR_ARG;
    pk->seqs.resize(N);
    long long off = 0;
    for (int n = 0; n < N; ++n) {
        const int len = cu_seqlens[n + 1] - cu_seqlens[n];
        if (len < 0) return GLA_ERR_ARG;
        const int nch = (len + 127) / 128;
        if (off > 0x7fffffffLL) return GLA_ERR_ARG;
        pk->seqs[n] = make_int4(cu_seqlens[n], len, nch, static_cast<int>(off));
        off += nch;
        pk->max_chunks = std::max(pk->max_chunks, nch);
    }
    pk->chunks = off;
    return GLA_OK;
}

// Launch plan for a packed batch: ranges of equal chunk counts over all
// sequences' chunks (the sequences differ in length, so cuts follow the
// chunk count, not the sequences), at least kMinRange chunks long.
Plan make_plan_packed(const Packed &pk, int H, int dk, int dv, const gla_chunk_options &op,
                      int sm_count) {
    Plan pl;
    pl.dv_tile = op.dv_tile ? op.dv_tile : (dv >= 128 ? 128 : 64);
    pl.pair = dk == 128 && dv == 2 * pl.dv_tile && op.cta_pair >= 0;
    pl.NC = pk.max_chunks;
    const long long total = static_cast<long long>(H) * pk.chunks;
    long long L;
    if (op.segments > 0) {
        L = (pk.max_chunks + op.segments - 1) / op.segments;
    } else {
        const int n_dvt = dv / pl.dv_tile;
        int resident = gla::chunk_fwd_max_resident(dk, pl.dv_tile, pl.pair ? 1 : 0);
        if (resident <= 0) resident = pl.pair ? sm_count / 2 : sm_count;
        const long long ranges = std::max<long long>(1, pl.pair ? resident : resident / n_dvt);
        L = (total + ranges - 1) / ranges;
        if (L < kMinRange) L = kMinRange;
        if (L > pk.max_chunks) L = pk.max_chunks;
    }
    if (L < 1) L = 1;
    pl.L = static_cast<int>(L);
    pl.W = static_cast<int>((total + L - 1) / L);
    pl.seg_max = 1;
    for (size_t n = 0; n < pk.seqs.size(); ++n) {
        const int4 e = pk.seqs[n];
        if (e.z == 0) continue;
        for (int h = 0; h < H; ++h) {
            const long long a = static_cast<long long>(H) * e.w + static_cast<long long>(h) * e.z;
            pl.seg_max = std::max(pl.seg_max, 1 + static_cast<int>((a + e.z - 1) / L - a / L));
        }
    }
    return pl;
}

}  // namespace

int chunk_fwd_packed(const void *q, const void *k, const void *v, const float *log_alpha,
                     float scale, const float *h0, void *o, float *hT, const int *cu_seqlens,
                     int N, int H, int T_total, int dk, int dv, const gla_chunk_options *opts,
                     cudaStream_t stream) {
    if (!q || !k || !v || !log_alpha || !o) return GLA_ERR_ARG;
    if (N <= 0 || H <= 0 || T_total < 0) return GLA_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) ||
        !aligned16(o) || (h0 && !aligned16(h0)) || (hT && !aligned16(hT)))
        return GLA_ERR_ARG;
    if (!dk_ok(dk) || !dv_ok(dv)) return GLA_ERR_SHAPE;
    gla_chunk_options o_def = {};
    const gla_chunk_options &op = opts ? *opts : o_def;
    if (!options_ok(dv, op) || op.gate_per_head) return GLA_ERR_ARG;
    if (static_cast<long long>(N) * H > 0x7fffffffLL) return GLA_ERR_ARG;
    Packed pk;
    int st = packed_layout(cu_seqlens, N, T_total, &pk);
    if (st != GLA_OK) return st;

    DeviceInfo *dev = nullptr;
    st = current_device(&dev);
    if (st != GLA_OK) return st;
    EncodeTiledFn enc = nullptr;
    st = encode_fn(&enc);
    if (st != GLA_OK) return st;

    // empty sequences: hT = h0 (zero without h0); nothing else to do for them
    const size_t state_elems = static_cast<size_t>(H) * dk * dv;
    if (hT && hT != h0) {
        for (int n = 0; n < N; ++n) {
            if (pk.seqs[n].y != 0) continue;
            float *dst = hT + n * state_elems;
            const cudaError_t e =
                h0 ? cudaMemcpyAsync(dst, h0 + n * state_elems, state_elems * sizeof(float),
                                     cudaMemcpyDeviceToDevice, stream)
                   : cudaMemsetAsync(dst, 0, state_elems * sizeof(float), stream);
            if (e != cudaSuccess) {
                cudaGetLastError();
                return GLA_ERR_LAUNCH;
            }
        }
    }
    if (pk.chunks == 0) return GLA_OK;

    const long long NH = static_cast<long long>(N) * H;
    const Plan pl = make_plan_packed(pk, H, dk, dv, op, dev->sm_count);
    const size_t table_bytes = align256(pk.seqs.size() * sizeof(int4));
    const size_t state_bytes =
        pl.seg_max > 1 ? static_cast<size_t>(pl.seg_max) * NH * dk * dv * sizeof(float) : 0;
    const size_t decay_bytes =
        pl.seg_max > 1 ? static_cast<size_t>(pl.seg_max) * NH * dk * sizeof(float) : 0;
    void *scratch = nullptr;
    if (cudaMallocAsync(&scratch, table_bytes + state_bytes + decay_bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_ALLOC;
    }
    int result = GLA_OK;
    // the table goes up with the launch; a copy from pageable memory has
    // taken the host data by the time the call returns
    if (cudaMemcpyAsync(scratch, pk.seqs.data(), pk.seqs.size() * sizeof(int4),
                        cudaMemcpyHostToDevice, stream) != cudaSuccess) {
        cudaGetLastError();
        result = GLA_ERR_LAUNCH;
    }
    ChunkLaunch p = {};
    if (result == GLA_OK &&
        (!make_map(enc, &p.tm_q, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dk, T_total, H, 64, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
         !make_map(enc, &p.tm_k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dk, T_total, H, 64, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
         !make_map(enc, &p.tm_a, log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dk, T_total, H,
                   pl.pair ? dk / 2 : dk, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
         !make_map(enc, &p.tm_v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dv, T_total, H, 64, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
         !make_map(enc, &p.tm_o32, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dv, T_total, H, 64, 32,
                   CU_TENSOR_MAP_SWIZZLE_128B)))
        result = GLA_ERR_LAUNCH;
    if (result == GLA_OK) {
        char *ws = static_cast<char *>(scratch) + table_bytes;
        p.q = q;
        p.k = k;
        p.log_alpha = log_alpha;
        p.h0 = h0;
        p.hT = hT;
        p.o = o;
        p.ws_state = pl.seg_max > 1 ? reinterpret_cast<float *>(ws) : nullptr;
        p.ws_decay = pl.seg_max > 1 ? reinterpret_cast<float *>(ws + state_bytes) : nullptr;
        p.scale = scale;
        p.B = N;
        p.H = H;
        p.T = T_total;
        p.dk = dk;
        p.dv = dv;
        p.dv_tile = pl.dv_tile;
        p.pair = pl.pair ? 1 : 0;
        p.NC = pl.NC;
        p.L = pl.L;
        p.W = pl.W;
        p.seg_max = pl.seg_max;
        p.total = static_cast<long long>(H) * pk.chunks;
        p.seqs = static_cast<const int4 *>(scratch);
        p.NS = N;
        p.force_exact = op.force_exact ? 1 : 0;
        p.status = dev->status;
        if (launch_chunk_fwd(p, stream) != 0) result = GLA_ERR_LAUNCH;
    }
    cudaFreeAsync(scratch, stream);
    return result;
}

}  // namespace gla

extern "C" {

int gla_version(void) { return 100; }

const char *gla_status_string(int status) {
    switch (status) {
        case GLA_OK: return "ok";
        case GLA_ERR_ARG: return "invalid argument (null pointer, non-positive size or misaligned pointer)";
        case GLA_ERR_SHAPE: return "unsupported head dimensions (dk in {64,128}, dv in {64,128,256})";
        case GLA_ERR_DEVICE: return "no usable CUDA device (this library needs an sm_103 GB300)";
        case GLA_ERR_LAUNCH: return "a CUDA call failed while enqueuing work";
        case GLA_ERR_TIMEOUT: return "a bounded device-side wait expired";
        case GLA_ERR_ALLOC: return "stream-ordered scratch allocation failed";
        case GLA_ERR_SCRATCH: return "the launch plan needs more scratch than the fixed no-allocation scratch holds";
        default: return "unknown status";
    }
}

int gla_chunk_fwd_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                     float scale, const float *h0, void *o, float *hT, int B, int H, int T,
                     int dk, int dv, const gla_chunk_options *opts, cudaStream_t stream) {
    return gla_chunk_fwd_debug(q, k, v, log_alpha, scale, h0, o, hT, B, H, T, dk, dv, opts,
                               nullptr, stream);
}

int gla_chunk_fwd_debug(const void *q, const void *k, const void *v, const float *log_alpha,
                        float scale, const float *h0, void *o, float *hT, int B, int H, int T,
                        int dk, int dv, const gla_chunk_options *opts, const gla_chunk_debug *dbg,
                        cudaStream_t stream) {
    using namespace gla;
    if (!q || !k || !v || !log_alpha || !o) return GLA_ERR_ARG;
    if (B <= 0 || H <= 0 || T <= 0) return GLA_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) ||
        !aligned16(o) || (h0 && !aligned16(h0)) || (hT && !aligned16(hT)))
        return GLA_ERR_ARG;
    if (!dk_ok(dk) || !dv_ok(dv)) return GLA_ERR_SHAPE;
    gla_chunk_options o_def = {};
    const gla_chunk_options &op = opts ? *opts : o_def;
    if (!options_ok(dv, op)) return GLA_ERR_ARG;
    if (static_cast<long long>(B) * H > 0x7fffffffLL) return GLA_ERR_ARG;
    // the instrumentation's own arguments; its kernel build covers one gate per
    // key channel only
    if (dbg && (dbg->withhold_v < 0 || (dbg->gamma && !aligned16(dbg->gamma)) || op.gate_per_head))
        return GLA_ERR_ARG;

    DeviceInfo *dev = nullptr;
    const int st = current_device(&dev);
    if (st != GLA_OK) return st;
    // the segment workspace (summaries S*, total decays) is stream-ordered
    const size_t ws_bytes = scratch_needed(make_plan(B, H, T, dk, dv, op, dev->sm_count), B, H,
                                           dk, dv);
    void *ws = nullptr;
    if (ws_bytes) {
        if (cudaMallocAsync(&ws, ws_bytes, stream) != cudaSuccess) {
            cudaGetLastError();
            return GLA_ERR_ALLOC;
        }
    }
    const int r = chunk_fwd_with_scratch(q, k, v, log_alpha, scale, h0, o, hT, B, H, T, dk, dv,
                                         &op, stream, ws, ws_bytes, dbg);
    if (ws) cudaFreeAsync(ws, stream);
    return r;
}

int gla_chunk_fwd_plan(int B, int H, int T, int dk, int dv, const gla_chunk_options *opts,
                       int *n_segments, int *dv_tile, int *launches, unsigned long *scratch_bytes) {
    using namespace gla;
    if (B <= 0 || H <= 0 || T <= 0) return GLA_ERR_ARG;
    if (static_cast<long long>(B) * H > 0x7fffffffLL) return GLA_ERR_ARG;
    if (!dk_ok(dk) || !dv_ok(dv)) return GLA_ERR_SHAPE;
    gla_chunk_options o_def = {};
    const gla_chunk_options &op = opts ? *opts : o_def;
    if (!options_ok(dv, op)) return GLA_ERR_ARG;
    DeviceInfo *dev = nullptr;
    const int st = current_device(&dev);
    if (st != GLA_OK) return st;
    const Plan pl = make_plan(B, H, T, dk, dv, op, dev->sm_count);
    if (n_segments) *n_segments = pl.seg_max;
    if (dv_tile) *dv_tile = pl.dv_tile;
    if (launches) *launches = pl.seg_max > 1 ? 2 : 1;
    if (scratch_bytes) *scratch_bytes = scratch_needed(pl, B, H, dk, dv);
    return GLA_OK;
}

int gla_chunk_fwd_varlen_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                            float scale, const float *h0, void *o, float *hT,
                            const int *cu_seqlens, int N, int H, int T_total, int dk, int dv,
                            const gla_chunk_options *opts, cudaStream_t stream) {
    return gla::chunk_fwd_packed(q, k, v, log_alpha, scale, h0, o, hT, cu_seqlens, N, H, T_total,
                                 dk, dv, opts, stream);
}

int gla_chunk_fwd_varlen_plan(const int *cu_seqlens, int N, int H, int T_total, int dk, int dv,
                              const gla_chunk_options *opts, int *n_segments, int *dv_tile,
                              int *launches, unsigned long *scratch_bytes) {
    using namespace gla;
    if (N <= 0 || H <= 0 || T_total < 0) return GLA_ERR_ARG;
    if (static_cast<long long>(N) * H > 0x7fffffffLL) return GLA_ERR_ARG;
    if (!dk_ok(dk) || !dv_ok(dv)) return GLA_ERR_SHAPE;
    gla_chunk_options o_def = {};
    const gla_chunk_options &op = opts ? *opts : o_def;
    if (!options_ok(dv, op)) return GLA_ERR_ARG;
    Packed pk;
    int st = packed_layout(cu_seqlens, N, T_total, &pk);
    if (st != GLA_OK) return st;
    DeviceInfo *dev = nullptr;
    st = current_device(&dev);
    if (st != GLA_OK) return st;
    if (pk.chunks == 0) {
        if (n_segments) *n_segments = 0;
        if (dv_tile) *dv_tile = 0;
        if (launches) *launches = 0;
        if (scratch_bytes) *scratch_bytes = 0;
        return GLA_OK;
    }
    const Plan pl = make_plan_packed(pk, H, dk, dv, op, dev->sm_count);
    const size_t NH = static_cast<size_t>(N) * H;
    if (n_segments) *n_segments = pl.seg_max;
    if (dv_tile) *dv_tile = pl.dv_tile;
    if (launches) *launches = pl.seg_max > 1 ? 2 : 1;
    if (scratch_bytes)
        *scratch_bytes = align256(pk.seqs.size() * sizeof(int4)) +
                         (pl.seg_max > 1 ? static_cast<size_t>(pl.seg_max) * NH * dk * (dv + 1) *
                                               sizeof(float)
                                         : 0);
    return GLA_OK;
}

int gla_chunk_fwd_varlen(const void *q, const void *k, const void *v, const float *log_alpha,
                         float scale, const float *h0, void *o, float *hT, const int *cu_seqlens,
                         int N, int H, int T_total, int dk, int dv, cudaStream_t stream) {
    return gla::chunk_fwd_packed(q, k, v, log_alpha, scale, h0, o, hT, cu_seqlens, N, H, T_total,
                                 dk, dv, nullptr, stream);
}

int gla_chunk_fwd(const void *q, const void *k, const void *v, const float *log_alpha,
                  float scale, const float *h0, void *o, float *hT, int B, int H, int T, int dk,
                  int dv, cudaStream_t stream) {
    return gla_chunk_fwd_ex(q, k, v, log_alpha, scale, h0, o, hT, B, H, T, dk, dv, nullptr,
                            stream);
}

int gla_recurrent_step(const void *q, const void *k, const void *v, const float *log_alpha,
                       float scale, float *h, void *o, int B, int H, int dk, int dv,
                       cudaStream_t stream) {
    using namespace gla;
    if (!q || !k || !v || !log_alpha || !h || !o) return GLA_ERR_ARG;
    if (B <= 0 || H <= 0) return GLA_ERR_ARG;
    if (static_cast<long long>(B) * H > 0x7fffffffLL) return GLA_ERR_ARG;
    if (!aligned16(h) || (reinterpret_cast<uintptr_t>(v) & 7u) ||
        (reinterpret_cast<uintptr_t>(o) & 7u) || (reinterpret_cast<uintptr_t>(q) & 1u) ||
        (reinterpret_cast<uintptr_t>(k) & 1u) || (reinterpret_cast<uintptr_t>(log_alpha) & 3u))
        return GLA_ERR_ARG;
    if (!dk_ok(dk) || !dv_ok(dv)) return GLA_ERR_SHAPE;
    DeviceInfo *dev = nullptr;
    int st = current_device(&dev);
    if (st != GLA_OK) return st;
    DecodeLaunch p{q, k, v, log_alpha, h, o, scale, B * H, dk, dv};
    return launch_recurrent_step(p, stream) == 0 ? GLA_OK : GLA_ERR_LAUNCH;
}

namespace {

// Scratch of the chunkwise backward for `units` (sequence, head) pairs whose
// chunks number `chunks` in all, over `rows` rows of the caller's tensors:
// chunk states (chunks + units slots) and state gradients (chunks slots) of
// dk x dv fp32 each, per-chunk carries and decays, the partial gradients and
// the path flags, each piece 256-byte aligned.
struct BwdScratch {
    size_t states, adjoints, carry, decay, partials, flags;
    size_t total() const { return states + adjoints + carry + decay + partials + flags; }
};

BwdScratch bwd_layout(long long units, long long chunks, long long rows, int dk, int dv) {
    const auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    BwdScratch s;
    s.states = al(sizeof(float) * static_cast<size_t>(chunks + units) * dk * dv);
    s.adjoints = al(sizeof(float) * static_cast<size_t>(chunks) * dk * dv);
    s.carry = al(sizeof(float) * static_cast<size_t>(chunks) * gla::bwd_value_tiles(dv) * dk);
    s.decay = al(sizeof(float) * static_cast<size_t>(chunks) * dk);
    s.partials = al(sizeof(float) * static_cast<size_t>(rows) * (2 * dk + dv));
    s.flags = al(static_cast<size_t>(chunks));
    return s;
}

// Points the scratch fields of p into ws, laid out as `s`.
void bwd_bind_scratch(gla::BwdLaunch &p, char *ws, const BwdScratch &s, long long rows, int dk) {
    p.states = reinterpret_cast<float *>(ws);
    ws += s.states;
    p.adjoints = reinterpret_cast<float *>(ws);
    ws += s.adjoints;
    p.carry = reinterpret_cast<float *>(ws);
    ws += s.carry;
    p.decay = reinterpret_cast<float *>(ws);
    ws += s.decay;
    p.pq = reinterpret_cast<float *>(ws);
    p.pk = p.pq + static_cast<size_t>(rows) * dk;
    p.pv = p.pk + static_cast<size_t>(rows) * dk;
    ws += s.partials;
    p.wide = reinterpret_cast<unsigned char *>(ws);
}

int bwd_chunks(int len) { return (len + gla::bwd_chunk_tokens() - 1) / gla::bwd_chunk_tokens(); }

int bwd_shape_ok(int B, int H, int T, int dk, int dv) {
    if (B <= 0 || H <= 0 || T <= 0) return GLA_ERR_ARG;
    if (H > 65535 || static_cast<long long>(B) * H > 0x7fffffffLL) return GLA_ERR_ARG;
    if (static_cast<long long>(B) * bwd_chunks(T) > 0x7fffffffLL) return GLA_ERR_ARG;
    if (!gla::dk_ok(dk) || !gla::dv_ok(dv)) return GLA_ERR_SHAPE;
    return GLA_OK;
}

BwdScratch bwd_layout_fixed(int B, int H, int T, int dk, int dv) {
    const long long units = static_cast<long long>(B) * H;
    return bwd_layout(units, units * bwd_chunks(T), units * T, dk, dv);
}

bool bwd_pointers_ok(const void *q, const void *k, const void *v, const float *log_alpha,
                     const void *d_o, const void *grad_q, const void *grad_k, const void *grad_v,
                     const float *grad_log_alpha, const float *h0, const float *dhT,
                     const float *grad_h0) {
    using gla::aligned16;
    if (!q || !k || !v || !log_alpha || !d_o || !grad_q || !grad_k || !grad_v || !grad_log_alpha)
        return false;
    return aligned16(q) && aligned16(k) && aligned16(v) && aligned16(d_o) && aligned16(grad_q) &&
           aligned16(grad_k) && aligned16(grad_v) && aligned16(log_alpha) &&
           aligned16(grad_log_alpha) && (!h0 || aligned16(h0)) && (!dhT || aligned16(dhT)) &&
           (!grad_h0 || aligned16(grad_h0));
}

void bwd_bind_tensors(gla::BwdLaunch &p, const void *q, const void *k, const void *v,
                      const float *log_alpha, const float *h0, const void *d_o,
                      const float *dhT, void *grad_q, void *grad_k, void *grad_v,
                      float *grad_log_alpha, float *grad_h0) {
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.d_o = static_cast<const __nv_bfloat16 *>(d_o);
    p.log_alpha = log_alpha;
    p.h0 = h0;
    p.dhT = dhT;
    p.gq = static_cast<__nv_bfloat16 *>(grad_q);
    p.gk = static_cast<__nv_bfloat16 *>(grad_k);
    p.gv = static_cast<__nv_bfloat16 *>(grad_v);
    p.ga = grad_log_alpha;
    p.gh0 = grad_h0;
}

}  // namespace

int gla_chunk_bwd_plan(int B, int H, int T, int dk, int dv, int *chunk, int *launches,
                       unsigned long *scratch_bytes) {
    const int st = bwd_shape_ok(B, H, T, dk, dv);
    if (st != GLA_OK) return st;
    if (chunk) *chunk = gla::bwd_chunk_tokens();
    if (launches) *launches = 6;
    if (scratch_bytes)
        *scratch_bytes = static_cast<unsigned long>(bwd_layout_fixed(B, H, T, dk, dv).total());
    return GLA_OK;
}

int gla_chunk_bwd_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                     float scale, const float *h0, const void *d_o, const float *dhT,
                     void *grad_q, void *grad_k, void *grad_v, float *grad_log_alpha,
                     float *grad_h0, int B, int H, int T, int dk, int dv,
                     const gla_chunk_options *opts, cudaStream_t stream) {
    using namespace gla;
    if (!bwd_pointers_ok(q, k, v, log_alpha, d_o, grad_q, grad_k, grad_v, grad_log_alpha, h0,
                         dhT, grad_h0))
        return GLA_ERR_ARG;
    const int shape = bwd_shape_ok(B, H, T, dk, dv);
    if (shape != GLA_OK) return shape;
    gla_chunk_options o_def = {};
    const gla_chunk_options &op = opts ? *opts : o_def;
    if ((op.gate_per_head != 0 && op.gate_per_head != 1) ||
        (op.force_exact != 0 && op.force_exact != 1))
        return GLA_ERR_ARG;
    const BwdScratch sl = bwd_layout_fixed(B, H, T, dk, dv);
    const long long rows = static_cast<long long>(B) * H * T;
    // one gate per head: the gate broadcast to every channel and its gradient, fp32 [BH, T, dk]
    const size_t gate_b = op.gate_per_head
                              ? ((sizeof(float) * static_cast<size_t>(rows) * dk + 255) &
                                 ~static_cast<size_t>(255))
                              : 0;

    DeviceInfo *dev = nullptr;
    const int st = current_device(&dev);
    if (st != GLA_OK) return st;
    char *ws = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void **>(&ws), sl.total() + 2 * gate_b, stream) !=
        cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_ALLOC;
    }
    BwdLaunch p = {};
    bwd_bind_tensors(p, q, k, v, log_alpha, h0, d_o, dhT, grad_q, grad_k, grad_v,
                     grad_log_alpha, grad_h0);
    bwd_bind_scratch(p, ws, sl, rows, dk);
    p.status = dev->status;
    p.scale = scale;
    p.seqs = nullptr;
    p.N = B;
    p.H = H;
    p.T = T;
    p.NC = bwd_chunks(T);
    p.chunks = static_cast<long long>(B) * p.NC;
    p.dk = dk;
    p.dv = dv;
    p.force_exact = op.force_exact;
    int r = GLA_OK;
    if (op.gate_per_head) {
        float *full = reinterpret_cast<float *>(ws + sl.total());
        float *gfull = reinterpret_cast<float *>(ws + sl.total() + gate_b);
        if (launch_gate_broadcast(log_alpha, full, rows, dk, stream) != 0) r = GLA_ERR_LAUNCH;
        p.log_alpha = full;
        p.ga = gfull;
    }
    if (r == GLA_OK && launch_chunk_bwd(p, stream) != 0) r = GLA_ERR_LAUNCH;
    if (r == GLA_OK && op.gate_per_head &&
        launch_gate_sum(p.ga, grad_log_alpha, rows, dk, stream) != 0)
        r = GLA_ERR_LAUNCH;
    cudaFreeAsync(ws, stream);
    return r;
}

int gla_chunk_bwd(const void *q, const void *k, const void *v, const float *log_alpha,
                  float scale, const float *h0, const void *d_o, const float *dhT,
                  void *grad_q, void *grad_k, void *grad_v, float *grad_log_alpha,
                  float *grad_h0, int B, int H, int T, int dk, int dv, cudaStream_t stream) {
    return gla_chunk_bwd_ex(q, k, v, log_alpha, scale, h0, d_o, dhT, grad_q, grad_k, grad_v,
                            grad_log_alpha, grad_h0, B, H, T, dk, dv, nullptr, stream);
}

int gla_chunk_bwd_varlen_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                            float scale, const float *h0, const void *d_o, const float *dhT,
                            void *grad_q, void *grad_k, void *grad_v, float *grad_log_alpha,
                            float *grad_h0, const int *cu_seqlens, int N, int H, int T_total,
                            int dk, int dv, const gla_chunk_options *opts, cudaStream_t stream) {
    using namespace gla;
    if (!bwd_pointers_ok(q, k, v, log_alpha, d_o, grad_q, grad_k, grad_v, grad_log_alpha, h0,
                         dhT, grad_h0) || !cu_seqlens)
        return GLA_ERR_ARG;
    if (N <= 0 || H <= 0 || T_total < 0 || H > 65535 ||
        static_cast<long long>(N) * H > 0x7fffffffLL)
        return GLA_ERR_ARG;
    if (!dk_ok(dk) || !dv_ok(dv)) return GLA_ERR_SHAPE;
    gla_chunk_options o_def = {};
    const gla_chunk_options &op = opts ? *opts : o_def;
    if (op.gate_per_head != 0 || (op.force_exact != 0 && op.force_exact != 1)) return GLA_ERR_ARG;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T_total) return GLA_ERR_ARG;
    // the sequence table {first row, length, chunks, first chunk}, 64-token chunks
    std::vector<int4> seqs(N);
    long long chunks = 0;
    for (int n = 0; n < N; ++n) {
        const int len = cu_seqlens[n + 1] - cu_seqlens[n];
        if (len < 0) return GLA_ERR_ARG;
        seqs[n] = make_int4(cu_seqlens[n], len, bwd_chunks(len), static_cast<int>(chunks));
        chunks += bwd_chunks(len);
        if (chunks > 0x7fffffffLL) return GLA_ERR_ARG;
    }
    DeviceInfo *dev = nullptr;
    const int st = current_device(&dev);
    if (st != GLA_OK) return st;
    const long long units = static_cast<long long>(N) * H, rows = static_cast<long long>(H) * T_total;
    const BwdScratch sl = bwd_layout(units, chunks * H, rows, dk, dv);
    const size_t table_b = (sizeof(int4) * static_cast<size_t>(N) + 255) & ~static_cast<size_t>(255);
    char *ws = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void **>(&ws), table_b + sl.total(), stream) !=
        cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_ALLOC;
    }
    int r = GLA_OK;
    // a copy from pageable memory has taken the host table by the time it returns
    if (cudaMemcpyAsync(ws, seqs.data(), sizeof(int4) * static_cast<size_t>(N),
                        cudaMemcpyHostToDevice, stream) != cudaSuccess) {
        cudaGetLastError();
        r = GLA_ERR_LAUNCH;
    }
    if (r == GLA_OK) {
        BwdLaunch p = {};
        bwd_bind_tensors(p, q, k, v, log_alpha, h0, d_o, dhT, grad_q, grad_k, grad_v,
                         grad_log_alpha, grad_h0);
        bwd_bind_scratch(p, ws + table_b, sl, rows, dk);
        p.status = dev->status;
        p.scale = scale;
        p.seqs = reinterpret_cast<const int4 *>(ws);
        p.N = N;
        p.H = H;
        p.T = T_total;
        p.NC = 0;
        p.chunks = chunks;
        p.dk = dk;
        p.dv = dv;
        p.force_exact = op.force_exact;
        if (launch_chunk_bwd(p, stream) != 0) r = GLA_ERR_LAUNCH;
    }
    cudaFreeAsync(ws, stream);
    return r;
}

int gla_chunk_bwd_varlen(const void *q, const void *k, const void *v, const float *log_alpha,
                         float scale, const float *h0, const void *d_o, const float *dhT,
                         void *grad_q, void *grad_k, void *grad_v, float *grad_log_alpha,
                         float *grad_h0, const int *cu_seqlens, int N, int H, int T_total, int dk,
                         int dv, cudaStream_t stream) {
    return gla_chunk_bwd_varlen_ex(q, k, v, log_alpha, scale, h0, d_o, dhT, grad_q, grad_k, grad_v,
                                   grad_log_alpha, grad_h0, cu_seqlens, N, H, T_total, dk, dv,
                                   nullptr, stream);
}

int gla_gdn_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                      const float *beta, float scale, const float *h0, void *o, float *hT, int B,
                      int H, int T, int dk, int dv, cudaStream_t stream) {
    using namespace gla;
    if (!q || !k || !v || !g || !beta || !o) return GLA_ERR_ARG;
    if (B <= 0 || H <= 0 || T <= 0) return GLA_ERR_ARG;
    if (dk != 128 || !dv_ok(dv)) return GLA_ERR_SHAPE;
    if (static_cast<long long>(B) * H > 65535) return GLA_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (hT && !aligned16(hT)) || (reinterpret_cast<uintptr_t>(g) & 3u) ||
        (reinterpret_cast<uintptr_t>(beta) & 3u) || (h0 && (reinterpret_cast<uintptr_t>(h0) & 3u)))
        return GLA_ERR_ARG;
    const long long BH = static_cast<long long>(B) * H;
    // the scratch rows are addressed by 32-bit TMA coordinates
    if (BH * ((static_cast<long long>(T) + 63) / 64) * 64 > 0x7fffffffLL) return GLA_ERR_ARG;
    DeviceInfo *dev = nullptr;
    const int st = current_device(&dev);
    if (st != GLA_OK) return st;
    const size_t bytes = gdn_chunk_scratch_bytes(BH, T, dk);
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_ALLOC;
    }
    const size_t rows = static_cast<size_t>(BH) * ((T + 63) / 64) * 64;
    GdnChunkLaunch p = {};
    p.q = q;
    p.k = k;
    p.v = v;
    p.g = g;
    p.beta = beta;
    p.scale = scale;
    p.h0 = h0;
    p.o = o;
    p.hT = hT;
    p.BH = static_cast<int>(BH);
    p.T = T;
    p.dk = dk;
    p.dv = dv;
    p.W = static_cast<__nv_bfloat16 *>(ws);
    p.Tm = reinterpret_cast<__nv_bfloat16 *>(static_cast<char *>(ws) + rows * dk * 2);
    p.status = dev->status;
    EncodeTiledFn enc = nullptr;
    int r = encode_fn(&enc);
    if (r == GLA_OK &&
        (!make_map(enc, &p.tm_q, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dk, T, p.BH, 64, 64,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
         !make_map(enc, &p.tm_k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dk, T, p.BH, 64, 64,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
         !make_map(enc, &p.tm_v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dv, T, p.BH, 64, 64,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
         !make_map(enc, &p.tm_w, p.W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dk,
                   static_cast<int>(rows), 1, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
         !make_map(enc, &p.tm_t, p.Tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64,
                   static_cast<int>(rows), 1, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)))
        r = GLA_ERR_LAUNCH;
    if (r != GLA_OK) {
        cudaFreeAsync(ws, stream);
        return r;
    }
    r = launch_gdn_chunk(p, stream);
    cudaFreeAsync(ws, stream);
    return r == 0 ? GLA_OK : GLA_ERR_LAUNCH;
}

int gla_last_device_status(cudaStream_t stream) {
    using namespace gla;
    DeviceInfo *dev = nullptr;
    int st = current_device(&dev);
    if (st != GLA_OK) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_LAUNCH;
    }
    unsigned int word = 0;
    if (cudaMemcpy(&word, dev->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_LAUNCH;
    }
    if (word != 0) {
        const unsigned int zero = 0;
        cudaMemcpy(dev->status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        return GLA_ERR_TIMEOUT;
    }
    return GLA_OK;
}

}  // extern "C"
