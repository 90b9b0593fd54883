// gla_chunk.cu — the chunked forward's fixed-length instantiations, its
// dispatch, and the occupancy query the launch plans use.  The kernel itself
// is in gla_chunk_kernel.cuh.
#include <mutex>

#include "gla_chunk_kernel.cuh"

namespace gla {


int chunk_fwd_max_resident(int dk, int dv_tile, int pair) {
    // cached per device and kernel variant (the query is a driver round trip)
    constexpr int kDevs = 64;
    static std::mutex mu;
    static int cache[kDevs][6];
    static bool init = false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) {
        cudaGetLastError();
        return 0;
    }
    const int variant = (dk == 128 ? 2 : 0) + (dv_tile == 64 ? 0 : 1) + (dk == 128 && pair ? 2 : 0);
    std::lock_guard<std::mutex> lock(mu);
    if (!init) {
        for (auto &row : cache)
            for (int &x : row) x = -1;
        init = true;
    }
    int &slot = cache[dev][variant];
    if (slot < 0) {
        if (dk == 128 && pair)
            slot = dv_tile == 64 ? max_resident<128, 64, true>() : max_resident<128, 128, true>();
        else if (dk == 128)
            slot = dv_tile == 64 ? max_resident<128, 64, false>() : max_resident<128, 128, false>();
        else
            slot = dv_tile == 64 ? max_resident<64, 64, false>() : max_resident<64, 128, false>();
    }
    return slot;
}

int launch_chunk_fwd(const ChunkLaunch &p, cudaStream_t stream) {
    if (p.debug) return launch_chunk_fwd_debug(p, stream);
    if (p.seqs) return launch_chunk_fwd_packed(p, stream);
    if (p.gate_per_head) return launch_chunk_fwd_scalar(p, stream);
    if (p.dk == 64) {
        if (p.dv_tile == 64) return launch_tiles<64, 64, false, false, false>(p, stream);
        if (p.dv_tile == 128) return launch_tiles<64, 128, false, false, false>(p, stream);
    } else if (p.dk == 128 && p.pair) {
        if (p.dv != 2 * p.dv_tile) return static_cast<int>(cudaErrorInvalidValue);
        if (p.dv_tile == 64) return launch_tiles<128, 64, true, false, false>(p, stream);
        if (p.dv_tile == 128) return launch_tiles<128, 128, true, false, false>(p, stream);
    } else if (p.dk == 128) {
        if (p.dv_tile == 64) return launch_tiles<128, 64, false, false, false>(p, stream);
        if (p.dv_tile == 128) return launch_tiles<128, 128, false, false, false>(p, stream);
    }
    return static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace gla
