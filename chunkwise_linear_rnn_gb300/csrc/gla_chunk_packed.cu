// gla_chunk_packed.cu — the chunked forward's instantiations for packed
// variable-length batches (sequence table, tail rows masked inside the
// kernel).  Kept apart from the fixed-length ones so that those compile
// without any of it, and so that the two translation units build in parallel.
#include "gla_chunk_kernel.cuh"

namespace gla {

int launch_chunk_fwd_packed(const ChunkLaunch &p, cudaStream_t stream) {
    if (p.dk == 64) {
        if (p.dv_tile == 64) return launch_tiles<64, 64, false, true, false>(p, stream);
        if (p.dv_tile == 128) return launch_tiles<64, 128, false, true, false>(p, stream);
    } else if (p.dk == 128 && p.pair) {
        if (p.dv != 2 * p.dv_tile) return static_cast<int>(cudaErrorInvalidValue);
        if (p.dv_tile == 64) return launch_tiles<128, 64, true, true, false>(p, stream);
        if (p.dv_tile == 128) return launch_tiles<128, 128, true, true, false>(p, stream);
    } else if (p.dk == 128) {
        if (p.dv_tile == 64) return launch_tiles<128, 64, false, true, false>(p, stream);
        if (p.dv_tile == 128) return launch_tiles<128, 128, false, true, false>(p, stream);
    }
    return static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace gla
