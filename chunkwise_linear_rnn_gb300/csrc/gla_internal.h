// gla_internal.h — launchers shared between the C-ABI translation unit and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace gla {

struct ChunkLaunch {
    // Tensor maps (3-D: channel, token, batch*head) for q, k, v, log_alpha.
    CUtensorMap tm_q, tm_k, tm_v, tm_a;
    const float *h0;          // [BH, dk, dv] or null (zero state)
    float *hT;                // [BH, dk, dv] or null
    void *o;                  // bf16 [BH, T, dv]
    float scale;
    int B, H, T, dk, dv;
    int dv_tile;              // 64 or 128
    int force_exact;
    unsigned int *status;     // device status word
};

// Returns a cudaError_t value (0 on success).
int launch_chunk_fwd(const ChunkLaunch &p, cudaStream_t stream);

struct DecodeLaunch {
    const void *q, *k, *v;
    const float *log_alpha;
    float *h;
    void *o;
    float scale;
    int BH, dk, dv;
};

int launch_recurrent_step(const DecodeLaunch &p, cudaStream_t stream);

}  // namespace gla
