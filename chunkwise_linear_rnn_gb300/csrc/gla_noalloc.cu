// gla_noalloc.cu — gla_chunk_fwd_noalloc: the chunked forward for callers that
// cannot let the library allocate device memory (runtimes that reserve and
// account for all of HBM themselves, or run without the stream-ordered pool).
//
// The segment scratch of the sequence-split path comes from one fixed array
// in this file instead of cudaMallocAsync.  Host code never uses the array's
// name as an address (on the host it names a host-side stand-in); the device
// address is looked up per device with cudaGetSymbolAddress and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "gla.h"
#include "gla_internal.h"

namespace gla {
namespace {

constexpr size_t kNoAllocScratchBytes = GLA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxNoAllocDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
void *g_noalloc_addr[kMaxNoAllocDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once
// per device, with that device current).  Returns a GLA status.
int noalloc_scratch(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxNoAllocDevices) {
        cudaGetLastError();
        return GLA_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&ptr), g_noalloc_scratch) !=
                cudaSuccess ||
            !ptr) {
            cudaGetLastError();
            return GLA_ERR_DEVICE;
        }
        g_noalloc_addr[dev] = ptr;
    }
    *out = g_noalloc_addr[dev];
    return GLA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace gla

extern "C" int gla_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                     const float *log_alpha, float scale, const float *h0,
                                     void *o, float *hT, int B, int H, int T, int dk, int dv,
                                     const gla_chunk_options *opts, cudaStream_t stream) {
    using namespace gla;
    // Host-side argument checks first, as for every other entry point.
    if (!q || !k || !v || !log_alpha || !o) return GLA_ERR_ARG;
    if (B <= 0 || H <= 0 || T <= 0) return GLA_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) ||
        !aligned16(o) || (h0 && !aligned16(h0)) || (hT && !aligned16(hT)))
        return GLA_ERR_ARG;
    if (!(dk == 64 || dk == 128) || !(dv == 64 || dv == 128 || dv == 256)) return GLA_ERR_SHAPE;
    void *scratch = nullptr;
    const int st = noalloc_scratch(&scratch);
    if (st != GLA_OK) return st;
    return chunk_fwd_with_scratch(q, k, v, log_alpha, scale, h0, o, hT, B, H, T, dk, dv, opts,
                                  stream, scratch, kNoAllocScratchBytes);
}
