// gla_chunk_scalar.cu — the chunked forward's instantiations for one gate per
// token and head (log_alpha [B, H, T]: the per-head decays of RetNet and
// Mamba-2 style models, a special case of GLA's per-channel gate).  The prep
// threads read the chunk's gates themselves and use each for every channel;
// no A tile is loaded.  Its own translation unit, compiled in parallel.
#include "gla_chunk_kernel.cuh"

namespace gla {

int launch_chunk_fwd_scalar(const ChunkLaunch &p, cudaStream_t stream) {
    if (p.dk == 64) {
        if (p.dv_tile == 64) return launch_tiles<64, 64, false, false, true>(p, stream);
        if (p.dv_tile == 128) return launch_tiles<64, 128, false, false, true>(p, stream);
    } else if (p.dk == 128 && p.pair) {
        if (p.dv != 2 * p.dv_tile) return static_cast<int>(cudaErrorInvalidValue);
        if (p.dv_tile == 64) return launch_tiles<128, 64, true, false, true>(p, stream);
        if (p.dv_tile == 128) return launch_tiles<128, 128, true, false, true>(p, stream);
    } else if (p.dk == 128) {
        if (p.dv_tile == 64) return launch_tiles<128, 64, false, false, true>(p, stream);
        if (p.dv_tile == 128) return launch_tiles<128, 128, false, false, true>(p, stream);
    }
    return static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace gla
