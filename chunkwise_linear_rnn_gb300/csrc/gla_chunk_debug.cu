// gla_chunk_debug.cu — the chunked forward's instrumented build, for
// gla_chunk_fwd_debug only: the kernel with its test hooks compiled in (the
// prefix-sum and block-length dumps, a caller-set wait limit, a withheld
// value tile).  The production instantiations (gla_chunk.cu and the packed
// and per-head-gate files) are compiled without them.
#include "gla_chunk_kernel.cuh"

namespace gla {

int launch_chunk_fwd_debug(const ChunkLaunch &p, cudaStream_t stream) {
    if (p.seqs || p.gate_per_head) return static_cast<int>(cudaErrorInvalidValue);
    if (p.dk == 64) {
        if (p.dv_tile == 64) return launch_tiles<64, 64, false, false, false, true>(p, stream);
        if (p.dv_tile == 128) return launch_tiles<64, 128, false, false, false, true>(p, stream);
    } else if (p.dk == 128 && p.pair) {
        if (p.dv != 2 * p.dv_tile) return static_cast<int>(cudaErrorInvalidValue);
        if (p.dv_tile == 64) return launch_tiles<128, 64, true, false, false, true>(p, stream);
        if (p.dv_tile == 128) return launch_tiles<128, 128, true, false, false, true>(p, stream);
    } else if (p.dk == 128) {
        if (p.dv_tile == 64) return launch_tiles<128, 64, false, false, false, true>(p, stream);
        if (p.dv_tile == 128) return launch_tiles<128, 128, false, false, false, true>(p, stream);
    }
    return static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace gla
