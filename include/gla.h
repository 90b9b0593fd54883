/*
 * gla.h — C ABI of the GB300 (sm_103a) gated linear attention library: the
 * chunked forward, its backward, and the decode step.
 *
 * The operation (from "Gated Linear Attention (GLA): Mathematical Foundations,
 * Data-Dependent Gating, Chunkwise Parallel Forms, and Sub-Quadratic Sequence
 * Modeling", llms.blog, section "The Gated Recurrent Update"):
 *
 *     S_t = diag(alpha_t) S_{t-1} + k_t^T v_t,      o_t = scale * q_t S_t,
 *
 * per (batch, head), with S in R^{dk x dv} and the gate given in log space,
 * log_alpha_t = log(alpha_t) (the page's A, section "Sequence Partitioning and
 * State Factorization").  The output reads the state after the token's own
 * update; `scale` multiplies the output only, never the state.
 *
 * Layouts: row-major, contiguous, head-first.
 *     q, k       bf16  [B, H, T, dk]
 *     v          bf16  [B, H, T, dv]
 *     log_alpha  fp32  [B, H, T, dk]
 *     o          bf16  [B, H, T, dv]      (round-to-nearest-even from fp32)
 *     h0, hT     fp32  [B, H, dk, dv]     (row index = key channel)
 *
 * Every pointer is a DEVICE pointer on the current CUDA device.  The caller
 * owns every buffer; the library keeps no pointer after a call returns.
 * All calls are asynchronous on `stream` (0 = the legacy default stream) and
 * return once the work is enqueued.
 *
 * Supported shapes: dk in {64, 128}; dv in {64, 128, 256}; B, H >= 1;
 * T >= 1 (any value: a ragged last chunk is handled inside the kernel).
 * Pointers must be 16-byte aligned.
 *
 * Domain: log_alpha finite and <= 0 (alpha in (0, 1], the page's range in
 * "Data-Dependent Forget Gate Parametrization").  Results for other gate
 * values are computed but not covered by the accuracy claim.
 *
 * Accuracy: o and hT match the token-by-token recurrence evaluated in fp64 on
 * the same inputs to relative L2 error <= 1e-2 and max-abs error <=
 * 2e-2 * RMS(reference), for every finite input in the domain.
 *
 * Error behaviour: every entry point validates its arguments on the host
 * before touching the GPU and returns a GLA_* status; nothing is enqueued
 * when the status is not GLA_OK.  Device-side bounded waits that expire set a
 * device status word, read (and cleared) by gla_last_device_status().
 */
#ifndef GLA_H_
#define GLA_H_

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *cudaStream_t;

enum gla_status {
    GLA_OK = 0,
    GLA_ERR_ARG = 1,         /* null pointer, non-positive size, misaligned pointer   */
    GLA_ERR_SHAPE = 2,       /* dk / dv outside the supported set                      */
    GLA_ERR_DEVICE = 3,      /* no CUDA device, or the device is not sm_103            */
    GLA_ERR_LAUNCH = 4,      /* a CUDA call failed while enqueuing the work            */
    GLA_ERR_TIMEOUT = 5,     /* a bounded device-side wait expired (from the status word) */
    GLA_ERR_ALLOC = 6,       /* stream-ordered scratch allocation failed               */
    GLA_ERR_SCRATCH = 7      /* plan needs more than gla_chunk_fwd_noalloc's fixed scratch */
};

/*
 * gla_chunk_fwd — chunkwise-parallel forward over whole sequences (prefill).
 *
 * Computes o for every token and, when hT != NULL, the state after the last
 * token, for the recurrence above started from h0 (zero when h0 == NULL).
 * The method is the chunkwise form of the same page, sections "Cumulative
 * Decay Representation", "Intra-Chunk Matrix Multiplications" and
 * "Inter-Chunk Recurrence and Output Projection": per chunk of tokens the
 * causal decayed Q K^T block times V, plus the decayed query times the state
 * entering the chunk, with the state carried on chip from chunk to chunk.
 *
 * hT may alias h0 (in-place state update).  o must not overlap any input.
 * When B * H is small the library splits each sequence into segments and
 * joins them with an exact state correction; that path allocates its scratch
 * with cudaMallocAsync / cudaFreeAsync on `stream`.
 */
int gla_chunk_fwd(const void *q, const void *k, const void *v, const float *log_alpha,
                  float scale, const float *h0, void *o, float *hT, int B, int H, int T,
                  int dk, int dv, cudaStream_t stream);

/* Tuning and test knobs for gla_chunk_fwd_ex.  Zero-initialise; 0 = automatic. */
typedef struct gla_chunk_options {
    int segments;      /* sequence segments per (batch, head); 0 = automatic, 1 = no split */
    int dv_tile;       /* value columns per CTA: 0 = automatic, else 64 or 128             */
    int force_exact;   /* 1 = process every chunk as rescaled sub-chunks (test knob)          */
    int cta_pair;      /* dk = 128 with two value-column tiles: 0 = run the tiles of a head as
                          a 2-CTA cluster sharing the key-side preparation (default),
                          -1 = independent CTAs; other values are GLA_ERR_ARG              */
    int gate_per_head; /* 1 = log_alpha is [B, H, T] fp32: one gate per token and head, the
                          same for every key channel (RetNet's fixed decay, the GLA page's
                          "The Retention and Recall Degradation Problem"; Mamba-2's scalar
                          gate, its "Structural Comparison Across Sub-Quadratic
                          Architectures"); the result is that of the [B, H, T, dk] gate
                          with every channel equal.  Fixed-length calls only
                          (gla_chunk_fwd_varlen_ex returns GLA_ERR_ARG); 0 = per channel */
    int reserved[3];
} gla_chunk_options;

/* gla_chunk_fwd with explicit options (opts may be NULL = all automatic). */
int gla_chunk_fwd_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                     float scale, const float *h0, void *o, float *hT, int B, int H, int T,
                     int dk, int dv, const gla_chunk_options *opts, cudaStream_t stream);

/*
 * gla_chunk_fwd_varlen — the chunked forward over a packed batch of N
 * sequences of different lengths: the chunkwise form above (the GLA page's
 * sections "Cumulative Decay Representation" to "Inter-Chunk Recurrence and
 * Output Projection") applied to each sequence on its own.  The FlashQLA
 * page, section "Application Scenarios and Outlook", lists variable-length
 * sequences among the cases such a kernel serves.
 *
 * Sequence n holds the token rows [cu_seqlens[n], cu_seqlens[n+1]) of every
 * head; its recurrence starts from its own initial state and ends in its own
 * final state, exactly as gla_chunk_fwd with B = 1 on that slice.
 *
 *   q, k       : [H, T_total, dk] bf16, device (head-first, sequences packed
 *                along the token axis)
 *   v          : [H, T_total, dv] bf16, device
 *   log_alpha  : [H, T_total, dk] fp32, device
 *   h0         : [N, H, dk, dv] fp32, device, or NULL (zero initial states)
 *   o          : [H, T_total, dv] bf16, device, written
 *   hT         : [N, H, dk, dv] fp32, device, or NULL; may alias h0
 *   cu_seqlens : HOST array of N + 1 ints: 0 = cu_seqlens[0] <= ... <=
 *                cu_seqlens[N] = T_total.  Read during the call only; the
 *                library keeps no pointer to it.  Empty sequences are
 *                allowed: their hT is their h0 (zero without h0).
 *
 * Device pointers must be 16-byte aligned.  Stream-ordered like
 * gla_chunk_fwd: the call allocates a small per-sequence table (plus the
 * segment scratch when sequences are split) with cudaMallocAsync on `stream`
 * and frees it on the same stream.  Returns GLA_ERR_ARG for null required
 * pointers, N or H <= 0, T_total < 0, cu_seqlens that do not run from 0 to
 * T_total without decreasing, or misaligned pointers; GLA_ERR_SHAPE for
 * unsupported dk/dv; GLA_ERR_ALLOC if the scratch cannot be allocated.
 */
int gla_chunk_fwd_varlen(const void *q, const void *k, const void *v, const float *log_alpha,
                         float scale, const float *h0, void *o, float *hT, const int *cu_seqlens,
                         int N, int H, int T_total, int dk, int dv, cudaStream_t stream);

/* gla_chunk_fwd_varlen with explicit options (opts may be NULL).  With a packed
 * batch, opts->segments caps the chunks of one range at ceil(longest
 * sequence's chunks / segments). */
int gla_chunk_fwd_varlen_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                            float scale, const float *h0, void *o, float *hT,
                            const int *cu_seqlens, int N, int H, int T_total, int dk, int dv,
                            const gla_chunk_options *opts, cudaStream_t stream);

/* The launch plan gla_chunk_fwd_varlen_ex would use for this packed batch
 * (no GPU work): most segments of any sequence, value-column tile, kernel
 * launches (0 when every sequence is empty) and stream-ordered scratch bytes
 * (sequence table included).  Output pointers may be NULL; cu_seqlens is a
 * host array as for gla_chunk_fwd_varlen. */
int gla_chunk_fwd_varlen_plan(const int *cu_seqlens, int N, int H, int T_total, int dk, int dv,
                              const gla_chunk_options *opts, int *n_segments, int *dv_tile,
                              int *launches, unsigned long *scratch_bytes);

/*
 * gla_chunk_fwd_plan — the launch plan gla_chunk_fwd_ex would use on the
 * current device for these sizes and options (no GPU work is enqueued):
 * the number of sequence segments, the value-column tile, the number of
 * kernel launches (1, or 2 when segments > 1) and the bytes of stream-ordered
 * scratch it allocates.  Any output pointer may be NULL.
 */
int gla_chunk_fwd_plan(int B, int H, int T, int dk, int dv, const gla_chunk_options *opts,
                       int *n_segments, int *dv_tile, int *launches, unsigned long *scratch_bytes);

/*
 * gla_chunk_fwd_debug — gla_chunk_fwd_ex with test instrumentation.  Not for
 * production use: the library's own tests call it to look inside the chunked
 * forward.  With dbg == NULL, or every field zero, it is gla_chunk_fwd_ex.
 *
 *   gamma         : nullable, device [B, H, T, dk] fp32, written: for every
 *                   token and key channel, the in-chunk prefix sum of
 *                   log_alpha that the preparation rescaled Q and K with (the
 *                   GLA page's "Cumulative Decay Representation"), in
 *                   natural-log units, relative to the reference of the
 *                   token's block: the chunk start when the chunk is one
 *                   block, else the start of its rescaled sub-chunk, whose
 *                   gates are clamped to [-30, 30].
 *   block_len     : nullable, device [B * H * ceil(T / 128)] int32, written:
 *                   the block length each chunk was processed with (128: one
 *                   block; less: the rescaled sub-chunk length).  Index
 *                   (b * H + h) * ceil(T / 128) + chunk.
 *   wait_limit_us : 0 = the production limit of every bounded device wait
 *                   (2 s); else that limit in microseconds.
 *   withhold_v    : 0 = off; n > 0: in the first launch every CTA's loader
 *                   never loads, nor announces, the value tile of the n-th
 *                   chunk it serves, so that the waits for it expire.  This
 *                   makes a timeout on purpose with no copy or product in
 *                   flight on the withheld barrier: the waiting threads give
 *                   up, the CTA frees its TMEM and returns.  The call returns
 *                   GLA_OK (it was enqueued); gla_last_device_status then
 *                   reports GLA_ERR_TIMEOUT, and the outputs are undefined.
 *
 * With dbg non-NULL the call runs an instrumented build of the kernel (the
 * production entry points run a build without any of this); it covers one
 * gate per key channel, so opts->gate_per_head must be 0.
 *
 * Returns as gla_chunk_fwd_ex, and GLA_ERR_ARG for a negative withhold_v or
 * gate_per_head set.
 */
typedef struct gla_chunk_debug {
    float *gamma;
    int *block_len;
    unsigned int wait_limit_us;
    int withhold_v;
} gla_chunk_debug;
int gla_chunk_fwd_debug(const void *q, const void *k, const void *v, const float *log_alpha,
                        float scale, const float *h0, void *o, float *hT, int B, int H, int T,
                        int dk, int dv, const gla_chunk_options *opts, const gla_chunk_debug *dbg,
                        cudaStream_t stream);

/*
 * gla_chunk_fwd_noalloc — gla_chunk_fwd_ex that allocates no device memory.
 *
 * The pages describe no counterpart: this is a service to callers that cannot
 * let a library allocate, such as serving runtimes that reserve all of HBM up
 * front and account for every byte themselves, or that run with the
 * stream-ordered memory pool disabled.  For them the cudaMallocAsync that
 * gla_chunk_fwd_ex makes when it splits sequences into segments is not an
 * option.  This entry point computes exactly what gla_chunk_fwd_ex computes,
 * with the segment scratch taken from one fixed array of
 * GLA_NOALLOC_SCRATCH_BYTES (16 MiB) that lives in the library and is held
 * on every GPU that loads it, until the process exits.  The caller still
 * passes every input and output buffer.
 *
 * Limit: an automatic plan (opts->segments == 0) whose segments would need
 * more scratch than the array holds cuts the sequences into fewer, longer
 * segments (down to none), so it always fits; the results stay within the
 * accuracy bar either way.  An explicit opts->segments that needs more
 * returns GLA_ERR_SCRATCH and enqueues nothing.  gla_chunk_fwd_plan reports
 * the allocating entry point's plan.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (with that device current) and caches it; make that first call before any
 * stream capture begins.
 *
 * Sharing: every call uses the same array and leaves the last call's contents
 * in it.  Calls whose GPU work overlaps (different streams, or several host
 * threads without ordering between their streams) race on the array; order
 * such calls on one stream.  Nothing in the array needs to start at zero.
 */
#define GLA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int gla_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *log_alpha,
                          float scale, const float *h0, void *o, float *hT, int B, int H, int T,
                          int dk, int dv, const gla_chunk_options *opts, cudaStream_t stream);

/*
 * gla_chunk_fwd_host — gla_chunk_fwd on buffers in host memory, end to end.
 *
 * Computes what gla_chunk_fwd computes (the same page and sections), for
 * q, k, v, log_alpha, h0 (nullable), o and hT (nullable) that live in host
 * memory, with gla_chunk_fwd's layouts.  The inputs are copied to the device,
 * the chunked forward runs, and the outputs are copied back.  The work is
 * pipelined over up to 8 groups of consecutive (batch, head) rows: while one
 * group computes, the next group's inputs travel host->device and the
 * previous group's outputs travel device->host on two internal streams.
 *
 * Ordering: the call is asynchronous and ordered on `stream`.  Once `stream`
 * has completed the work enqueued here, o and hT hold the results.
 * Copies overlap only when the host buffers are page-locked (cudaHostAlloc
 * or cudaHostRegister); pageable buffers give the same results, more slowly.
 * hT may alias h0.
 *
 * Device memory: two input slots and two output slots of one group each
 * (about 2/8 of the whole problem's device footprint, plus segment scratch).
 * They are allocated with cudaMallocAsync on `stream` and freed with
 * cudaFreeAsync once the call's work is done.  The internal streams and
 * events are created and destroyed inside each call, so the call cannot be
 * captured into a CUDA graph.
 *
 * Errors are those of gla_chunk_fwd: GLA_ERR_ARG / GLA_ERR_SHAPE before any
 * CUDA call; GLA_ERR_ALLOC when the slots cannot be allocated; GLA_ERR_LAUNCH
 * when a copy, event or kernel launch fails.  After an error, no further work
 * is enqueued.  Work already enqueued completes before the slots are freed;
 * outputs are then incomplete.
 */
int gla_chunk_fwd_host(const void *q, const void *k, const void *v, const float *log_alpha,
                       float scale, const float *h0, void *o, float *hT, int B, int H, int T,
                       int dk, int dv, cudaStream_t stream);

/*
 * gla_recurrent_step — one decode token for B * H independent heads.
 *
 * h (fp32 [B, H, dk, dv]) is read and overwritten in place with
 * diag(exp(log_alpha)) h + k^T v; o (bf16 [B, H, dv]) receives scale * q h
 * with the updated h.  q, k, log_alpha are [B, H, dk]; v is [B, H, dv].
 * Source: the recurrence above, one step (the same page, "The Gated Recurrent
 * Update"; constant-memory decoding in its "Training and Inference
 * Throughput" section).
 */
int gla_recurrent_step(const void *q, const void *k, const void *v, const float *log_alpha,
                       float scale, float *h, void *o, int B, int H, int dk, int dv,
                       cudaStream_t stream);

/*
 * gla_chunk_bwd — gradients of the chunked forward, for training.
 *
 * With the forward above (same q, k, v, log_alpha, scale, h0) and the loss
 * L = sum_t <d_o_t, o_t> + <dhT, hT>, writes
 *     grad_q, grad_k    bf16 [B, H, T, dk]    dL/dq, dL/dk
 *     grad_v            bf16 [B, H, T, dv]    dL/dv
 *     grad_log_alpha    fp32 [B, H, T, dk]    dL/dlog_alpha
 *     grad_h0           fp32 [B, H, dk, dv]   dL/dh0 (nullable: not written)
 * from d_o (bf16 [B, H, T, dv], the gradient of o) and dhT (fp32
 * [B, H, dk, dv], the gradient of hT; NULL = zero).  h0 NULL = zero state.
 * No output may alias an input.
 *
 * The states are recomputed from the inputs (no forward activations are
 * needed): every chunk's own state and state-gradient sums in parallel, two
 * scans over the chunks for the chunk-start states and the state gradients,
 * then every chunk's gradients
 * independently.  Source: the recurrence and chunk equations of the page
 * named above (sections "The Gated Recurrent Update", "Cumulative Decay
 * Representation", "Intra-Chunk Matrix Multiplications", "Inter-Chunk
 * Recurrence and Output Projection"), differentiated; its section "I/O-Aware
 * Kernel Design in FlashLinearAttention" has the backward recompute the chunk
 * states rather than cache them, as this call does.
 *
 * Scratch: (2 NC + 1) * B * H * dk * dv fp32 plus per-chunk decays and
 * log-gate carries, NC = ceil(T / 64), taken stream-ordered (cudaMallocAsync) and released on
 * `stream` (GLA_ERR_ALLOC when the pool cannot supply it).
 *
 * Shapes as for gla_chunk_fwd, with H <= 65535; pointers 16-byte aligned.
 * A bounded device wait that expires leaves the gradients unspecified and is
 * reported by gla_last_device_status (GLA_ERR_TIMEOUT).  Accuracy: each gradient matches the fp64 reverse-mode
 * differentiation of the recurrence to relative L2 error <= 1e-2 and max-abs
 * error <= 2e-2 * RMS(reference).
 */
int gla_chunk_bwd(const void *q, const void *k, const void *v, const float *log_alpha,
                  float scale, const float *h0, const void *d_o, const float *dhT,
                  void *grad_q, void *grad_k, void *grad_v, float *grad_log_alpha,
                  float *grad_h0, int B, int H, int T, int dk, int dv, cudaStream_t stream);

/*
 * gla_chunk_bwd with options.  `force_exact`: every chunk takes each
 * in-chunk decay factor as its own exponential (the path chunks whose decay
 * spans more than 2^120 always take).  `gate_per_head` = 1: log_alpha and
 * grad_log_alpha are fp32 [B, H, T], one gate per token and head used for
 * every key channel; the gradient of a head gate is the sum of its channels'
 * (two more launches and 2 * B * H * T * dk fp32 of scratch).  The other
 * fields are ignored.  opts NULL = defaults.
 */
int gla_chunk_bwd_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                     float scale, const float *h0, const void *d_o, const float *dhT,
                     void *grad_q, void *grad_k, void *grad_v, float *grad_log_alpha,
                     float *grad_h0, int B, int H, int T, int dk, int dv,
                     const gla_chunk_options *opts, cudaStream_t stream);

/*
 * The launch plan gla_chunk_bwd uses for a shape (host only, no GPU work):
 * tokens per chunk, kernel launches per call and scratch bytes.  Any output
 * pointer may be NULL.  Returns GLA_OK, GLA_ERR_ARG or GLA_ERR_SHAPE.
 */
int gla_chunk_bwd_plan(int B, int H, int T, int dk, int dv, int *chunk, int *launches,
                       unsigned long *scratch_bytes);

/*
 * gla_chunk_bwd_varlen — the backward of gla_chunk_fwd_varlen: gradients for
 * a packed batch of N sequences of different lengths, each its own
 * recurrence (layouts as for gla_chunk_fwd_varlen):
 *   q, k, log_alpha, grad_q, grad_k, grad_log_alpha : [H, T_total, dk]
 *   v, d_o, grad_v                                   : [H, T_total, dv]
 *   h0, dhT, grad_h0                                 : [N, H, dk, dv] (each nullable)
 *   cu_seqlens : HOST array of N + 1 ints, from 0 to T_total, nondecreasing.
 * One set of launches covers every chunk of every sequence (a table of the
 * sequences goes up to stream-ordered scratch with the call); an empty
 * sequence gets grad_h0 = dhT (zero without dhT).  Per-head gates are not
 * supported here (GLA_ERR_ARG).
 * Errors as for gla_chunk_bwd and gla_chunk_fwd_varlen.
 */
int gla_chunk_bwd_varlen(const void *q, const void *k, const void *v, const float *log_alpha,
                         float scale, const float *h0, const void *d_o, const float *dhT,
                         void *grad_q, void *grad_k, void *grad_v, float *grad_log_alpha,
                         float *grad_h0, const int *cu_seqlens, int N, int H, int T_total, int dk,
                         int dv, cudaStream_t stream);

/* gla_chunk_bwd_varlen with options (force_exact only; opts may be NULL). */
int gla_chunk_bwd_varlen_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                            float scale, const float *h0, const void *d_o, const float *dhT,
                            void *grad_q, void *grad_k, void *grad_v, float *grad_log_alpha,
                            float *grad_h0, const int *cu_seqlens, int N, int H, int T_total,
                            int dk, int dv, const gla_chunk_options *opts, cudaStream_t stream);

/*
 * gla_gdn_fwd — the gated delta rule (Gated DeltaNet), forward, per (batch,
 * head), with S in R^{dk x dv} and row vectors:
 *     S_t = alpha_t (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t,
 *     o_t = scale * q_t S_t,
 * from the FlashQLA page ("Qwen Team Releases FlashQLA for High-Performance
 * Linear Attention", "Core Technical Principles": scalar alpha, beta in
 * (0, 1), L2-normalised keys), in the standard gated-delta-rule reading.
 *   q, k    bf16 [B, H, T, dk] (k as given: the caller normalises it)
 *   v, o    bf16 [B, H, T, dv]
 *   g       fp32 [B, H, T]     log alpha (finite, <= 0)
 *   beta    fp32 [B, H, T]     in [0, 1]
 *   h0, hT  fp32 [B, H, dk, dv] (nullable; zero initial state / not written)
 * No output may overlap an input (hT must not alias h0).  The call is
 * asynchronous on `stream`; the caller owns every buffer.
 * Token-recurrent: the exact recurrence, one step per token, the state in
 * registers.  Shapes: dk in {64, 128}, dv in {64, 128, 256}, B * H <= 65535.
 * q, k and v must be 16-byte aligned (the next 32 tokens are fetched in
 * 16-byte pieces while the current ones compute; GLA_ERR_ARG otherwise); the
 * other pointers need their element alignment.  Errors as for gla_chunk_fwd.
 */
int gla_gdn_fwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                float scale, const float *h0, void *o, float *hT, int B, int H, int T, int dk,
                int dv, cudaStream_t stream);

/*
 * gla_gdn_chunk_fwd — the same gated delta rule forward as gla_gdn_fwd (same
 * arguments, layouts and results), computed by chunks of 64 tokens on the
 * tensor cores with the FlashQLA page's four-step chunk algorithm ("Qwen Team
 * Releases FlashQLA for High-Performance Linear Attention", "Core Technical
 * Principles"): per chunk, with gamma the in-chunk products of the gates,
 *   1. T = (I + L)^-1, L_ti = beta_t (gamma_t / gamma_i) k_t.k_i for i < t;
 *   2. W = T diag(beta gamma) K and U = T diag(beta) V;
 *   3. S_end = gamma_C S + (diag(gamma_C / gamma) K)^T (U - W S);
 *   4. O = scale (diag(gamma) Q S + tril(Q K^T gamma_t / gamma_i) (U - W S)).
 * Step 1 and W run for all chunks at once and leave W and (T - I) diag(beta)
 * (bf16) in stream-ordered scratch (cudaMallocAsync / cudaFreeAsync on
 * `stream`): ceil(T / 64) * 64 * B * H * (2 dk + 128) bytes.  U and steps 3-4
 * run as each head's chunks are walked in order with the state on chip.
 * dk = 128 only (GLA_ERR_SHAPE otherwise); dv in {64, 128, 256};
 * B * H <= 65535 and B * H * ceil(T / 64) * 64 < 2^31 (the scratch rows'
 * tensor-map coordinates).  q, k, v, o and hT must be 16-byte aligned, g, beta
 * and h0 4-byte aligned.  GLA_ERR_ARG for a violated bound or alignment, found
 * on the host before any device call.  hT may alias h0.  GLA_ERR_ALLOC if the
 * scratch cannot be allocated.
 */
int gla_gdn_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                      const float *beta, float scale, const float *h0, void *o, float *hT, int B,
                      int H, int T, int dk, int dv, cudaStream_t stream);

/* Static text for a status code (never NULL). */
const char *gla_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word on the current device.  Returns GLA_ERR_TIMEOUT if any kernel since
 * the last call gave up a bounded wait, GLA_ERR_LAUNCH if the stream reports
 * a CUDA error, else GLA_OK.
 */
int gla_last_device_status(cudaStream_t stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int gla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GLA_H_ */
