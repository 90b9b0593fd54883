// gla_internal.h — launchers shared between the C-ABI translation unit and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>

#include "gla.h"

namespace gla {

struct ChunkLaunch {
    // 3-D tensor maps (channel, token, batch*head): q, k, log_alpha, v, and o
    // (32-token boxes: each TMEM warp stores its own rows)
    CUtensorMap tm_q, tm_k, tm_a, tm_v, tm_o32;
    const void *q, *k;        // bf16 [BH, T, dk] (packed: [H, T, dk])
    const float *log_alpha;   // fp32 [BH, T, dk]
    const float *h0;          // [BH, dk, dv] or null (zero state)
    float *hT;                // [BH, dk, dv] or null
    void *o;                  // bf16 [BH, T, dv]
    float *ws_state;          // segment summaries [seg_max, BH, dk, dv] (seg_max > 1)
    float *ws_decay;          // segment total decays [seg_max, BH, dk]   (seg_max > 1)
    float scale;
    int B, H, T, dk, dv;
    int dv_tile;              // 64 or 128
    int pair;                 // 1: the two value tiles of a head run as a 2-CTA cluster
    // Work split: the chunks of all sequences, one after another, cut into W
    // ranges of L chunks (the last may be short); NC chunks per sequence;
    // seg_max = most segments any sequence is cut into (1: no sequence is cut).
    int NC, L, W, seg_max;
    long long total;          // chunks of all sequences
    // Packed variable-length batches (B = NS sequences per head, T = the
    // packed rows): device table of NS entries {first row, length, chunks,
    // chunk offset}, sequence u = n H + h.  Null for fixed-length batches.
    const int4 *seqs;
    int NS;
    int gate_per_head;        // 1: log_alpha is [BH, T], one gate per token (fixed length only)
    int force_exact;          // process every chunk in rescaled sub-chunks
    // two-segment plan of CTA pairs whose ranges are whole segments: the first
    // segment's CTA corrects the second segment's window itself, and a small
    // kernel forms hT (no correction pass)
    int fuse;
    unsigned int *status;     // device status word
    // test instrumentation (gla_chunk_fwd_debug; zero / null otherwise).  A
    // call with `debug` set runs the instrumented kernel build, which alone
    // reads the fields below; production calls run a build without them.
    int debug;
    unsigned long long wait_ns;   // bounded-wait limit (0 = the default, 2 s)
    float *dbg_gamma;         // [rows, dk] in-chunk prefix sums the preparation used, or null
    int *dbg_blk;             // block length of every chunk (global chunk index), or null
    int withhold_v;           // n > 0: each FULL-pass CTA withholds its n-th value tile
};

// Returns a cudaError_t value (0 on success).
int launch_chunk_fwd(const ChunkLaunch &p, cudaStream_t stream);

// launch_chunk_fwd with the instrumented kernel build (p.debug set; fixed-length
// batches, one gate per key channel); gla_chunk_debug.cu.
int launch_chunk_fwd_debug(const ChunkLaunch &p, cudaStream_t stream);

// launch_chunk_fwd for a packed batch (p.seqs set); gla_chunk_packed.cu.
int launch_chunk_fwd_packed(const ChunkLaunch &p, cudaStream_t stream);

// launch_chunk_fwd with one gate per token and head (p.gate_per_head);
// gla_chunk_scalar.cu.
int launch_chunk_fwd_scalar(const ChunkLaunch &p, cudaStream_t stream);

// How many CTAs (clusters, for a CTA pair) of the chunked forward for these
// head dimensions can run at once on the current device; 0 if unknown.
int chunk_fwd_max_resident(int dk, int dv_tile, int pair);

// gla_chunk_fwd_ex with the segment scratch supplied by the caller instead of
// allocated (`scratch_bytes` bytes of device memory, 16-byte aligned; may be
// null when the plan needs none).  Returns a GLA status; GLA_ERR_SCRATCH when
// the launch plan needs more scratch than given.
// `dbg`: test instrumentation (gla_chunk_fwd_debug), or null.
int chunk_fwd_with_scratch(const void *q, const void *k, const void *v, const float *log_alpha,
                           float scale, const float *h0, void *o, float *hT, int B, int H, int T,
                           int dk, int dv, const gla_chunk_options *opts, cudaStream_t stream,
                           void *scratch, size_t scratch_bytes,
                           const gla_chunk_debug *dbg = nullptr);

// The chunked forward over a packed variable-length batch (see
// gla_chunk_fwd_varlen_ex).  Returns a GLA status.
int chunk_fwd_packed(const void *q, const void *k, const void *v, const float *log_alpha,
                     float scale, const float *h0, void *o, float *hT, const int *cu_seqlens,
                     int N, int H, int T_total, int dk, int dv, const gla_chunk_options *opts,
                     cudaStream_t stream);

struct DecodeLaunch {
    const void *q, *k, *v;
    const float *log_alpha;
    float *h;
    void *o;
    float scale;
    int BH, dk, dv;
};

int launch_recurrent_step(const DecodeLaunch &p, cudaStream_t stream);

// The chunkwise backward (gla_backward.cu).
struct BwdLaunch {
    const __nv_bfloat16 *q, *k, *v, *d_o;   // [BH, T, dk] / [BH, T, dv]
    const float *log_alpha;                  // [BH, T, dk]
    const float *h0, *dhT;                   // [BH, dk, dv] or null (zero)
    __nv_bfloat16 *gq, *gk, *gv;             // gradients of q, k, v
    float *ga;                               // gradient of log_alpha [BH, T, dk]
    float *gh0;                              // gradient of h0 [BH, dk, dv] or null
    // Scratch.  Per unit, chunk states (nch + 1 slots) and state gradients
    // (nch slots) of dk x dv fp32 each; per unit and chunk, the log-gate
    // carry (dv / 32 x dk), the chunk decay (dk) and the path flag; partial
    // gradients laid out like the caller's q / v rows.
    float *states, *adjoints, *carry, *decay;
    float *pq, *pk, *pv;
    unsigned char *wide;                     // 1 = chunk left to the exact-path kernels
    unsigned int *status;                    // device status word (bounded waits)
    float scale;
    // Work: N sequences of H heads; unit n H + h indexes h0, dhT and dh0.
    // Fixed length (seqs == null): the caller's tensors are [N, H, T, .] and
    // every sequence has NC chunks.  Packed (seqs set): the tensors are
    // [H, T, .] with T the packed length, and seqs[n] = {first row, length,
    // chunks, first chunk} describes sequence n.  `chunks` counts the chunks
    // of all sequences (one head).
    const int4 *seqs;
    int N, H, T, NC, dk, dv;
    long long chunks;
    int force_exact;
};

// Tokens per backward chunk, and value-column tiles of the state passes.
int bwd_chunk_tokens();
int bwd_value_tiles(int dv);

// One gate per token and head: full[r][i] = g[r] for every key channel, and
// g[r] = sum_i full[r][i] (rows = B * H * T).  Return cudaError_t values.
int launch_gate_broadcast(const float *g, float *full, long long rows, int dk, cudaStream_t stream);
int launch_gate_sum(const float *full, float *g, long long rows, int dk, cudaStream_t stream);

// Enqueues the six backward kernels; returns a cudaError_t value.
int launch_chunk_bwd(const BwdLaunch &p, cudaStream_t stream);

// The gated delta rule forward by chunks (gla_gdn_chunk.cu): dk = 128.
struct GdnChunkLaunch {
    const void *q, *k, *v;         // bf16 [BH, T, dk] / [BH, T, dv]
    const float *g, *beta;         // fp32 [BH, T]
    float scale;
    const float *h0;               // [BH, dk, dv] or null (zero state)
    void *o;                       // bf16 [BH, T, dv]
    float *hT;                     // [BH, dk, dv] or null
    int BH, T, dk, dv;
    // scratch of the pre-pass, rows = BH * ceil(T / 64) * 64:
    // W bf16 [rows, dk] and the chunks' inverses T bf16 [rows, 64]
    __nv_bfloat16 *W;
    __nv_bfloat16 *Tm;
    // tensor maps, 64 x 64 boxes, 128-byte swizzle: q, k (128, T, BH), v (dv, T, BH),
    // W (128, rows, 1), T (64, rows, 1)
    CUtensorMap tm_q, tm_k, tm_v, tm_w, tm_t;
    unsigned int *status;          // device status word (bounded waits)
};

// Bytes of pre-pass scratch for these sizes (W and T).
inline size_t gdn_chunk_scratch_bytes(long long BH, int T, int dk) {
    const long long rows = BH * ((T + 63) / 64) * 64;
    return static_cast<size_t>(rows) * (static_cast<size_t>(dk) * 2 + 64 * 2);
}

// Enqueues the WY pre-pass and the sequential chunk kernel; returns a cudaError_t value.
int launch_gdn_chunk(const GdnChunkLaunch &p, cudaStream_t stream);

}  // namespace gla
