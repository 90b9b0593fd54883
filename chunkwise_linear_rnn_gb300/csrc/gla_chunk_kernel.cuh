// gla_chunk_kernel.cuh — chunkwise-parallel GLA forward on sm_103a tensor cores:
// the kernel template and its launcher, instantiated by gla_chunk.cu
// (fixed-length batches) and gla_chunk_packed.cu (packed variable-length
// batches: PACKED = true), which compile in parallel.
//
// Method ("Gated Linear Attention (GLA): Mathematical Foundations, ..."
// (llms.blog), sections "Sequence Partitioning and State Factorization",
// "Cumulative Decay Representation", "Intra-Chunk Matrix Multiplications",
// "Inter-Chunk Recurrence and Output Projection", "I/O-Aware Kernel Design"):
// per chunk of C tokens with A = log alpha and Gamma = in-chunk inclusive
// prefix sum of A (per key channel),
//     O     = scale * ( M V + (Q * e^Gamma) S_prev ),
//             M_ij = sum_d Q_id K_jd e^(Gamma_id - Gamma_jd)  for j <= i, else 0
//     S_new = diag(e^Gamma_C) S_prev + (K * e^(Gamma_C - Gamma))^T V,
// with the state S held on chip (TMEM, fp32) across the whole chunk loop.
//
// Rescaling (bounded exponents).  With a reference r (the Gamma value just
// before the first token of a block of tokens), Qh = Q e^(Gamma - r) <= |Q| and
// Kh = K e^(r - Gamma): the decayed score block factorises as P = Qh Kh^T and
// the state update as S_new = diag(e^(Gamma_end - r)) (S_prev + Kh^T V).  Both
// are plain tensor-core products.  A chunk is processed as one block when
// every |Gamma - r| <= kExpBound over it (the common case); otherwise it is
// cut into equal power-of-two sub-chunks, each with its own reference, small
// enough that the bound holds in each (sub-chunk rescaling).  A single token
// whose own |log alpha| exceeds the bound is clamped to it: the state term
// that changes is below e^-30 ~ 9e-14 of the state, under fp32 resolution.
// Masked score entries are selected away, never multiplied by zero.
//
// A CTA pair folds the read-out scale into Qh (scale Q e^Gamma): both of an
// output's products then arrive scaled, and the epilogue of the TMEM warps,
// on the pair's critical path, only rounds.  A single CTA, whose preparation
// is the longer path, scales in the epilogue.
//
// Precision.  bf16 operands carry 8 significant bits; the two roundings that
// dominate the output error are removed by splitting the operand into a bf16
// pair x = hi + lo: the rescaled keys Kh (score and state products) and the
// score block P (the A operand of P V, kept in TMEM).
//
// CTA organisation (one CTA per (batch, head, value-column tile, sequence
// segment); 448 threads):
//   warp 13 "tma": streams each chunk's A (fp32), Q, K (bf16, 128-byte swizzle,
//     already in the K-major operand layout) and V (MN-major) tiles with TMA,
//     each as soon as the tile it replaces has been consumed.
//   warps 0-7 "prep": two channels x 32 tokens per thread (dk = 128).  As
//     soon as the A tile lands (before Q and K): the fp32 prefix sum per token
//     part, written in place of A, the exponent-bound check that picks one
//     block or rescaled sub-chunks, and the state factor and correction-window
//     bookkeeping.  When Q and K land: Gamma = part offset + local sum, and the
//     elementwise in-place rescale to Qh and Kh_hi plus Kh_lo.
//   warp 12 "mma": one thread issues every tcgen05.mma and commit.
//   warps 8-11 "tmem": thread i owns TMEM lane i — causal mask and hi/lo split
//     of P, the per-row state scale and its bf16 copy for the next chunk's
//     Qh S product, and the output epilogue.
// The O accumulator is double-buffered so the next chunk's products overlap
// the current chunk's epilogue; the next chunk's Q/K/A loads overlap the
// current chunk's P V product and epilogue.
//
// Sequence segments (when B*H*tiles is too small to fill the GPU): segment
// s > 0 first runs from a zero state (FULL mode), storing its end state and
// total decay.  Its outputs depend on the true start state only through
// (Q * e^Gamma_seg) S_start, where Gamma_seg is the decay since the segment
// start; once every channel has decayed past e^-20.8 = 2^-30 that term is
// below 2^-30 of the start state's read-out, far below the bf16 resolution of
// the output, and the FULL outputs are stored as they are.
// The chunks before that point are recomputed by a second launch (CORRECT
// mode) from the exact start state, obtained by scanning the segment summaries
// S_start(s+1) = diag(e^G_s) S_start(s) + S*_s.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "gla_internal.h"
#include "gla_ptx.cuh"

namespace gla {
namespace {

constexpr int kChunk = 128;
constexpr int kPrepWarps = 8;           // warps 0-7
constexpr int kPrepThreads = 32 * kPrepWarps;
constexpr int kTmemWarp0 = 8;           // warps 8-11
constexpr int kMmaWarp = 12;
constexpr int kTmaWarp = 13;
constexpr int kThreads = 448;           // 14 warps
constexpr float kExpBound = 30.f;
constexpr float kWindowCut = 20.79441542f;  // 30 ln 2
// The fast path keeps in-chunk prefix sums in log2 units (Gamma log2 e), so
// that every exponential is one ex2.
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kExpBound2 = kExpBound * kLog2e;
constexpr uint32_t kBlk = kChunk * 128;     // one 64-column block of a 128-row tile

constexpr int kItemLast = 1;      // last item of its chunk: releases the chunk's V stage
constexpr int kItemStore = 2;     // store this item's output rows
constexpr int kItemEnd = 4;       // end of the item stream
constexpr int kItemPieceEnd = 8;  // last item of a piece (FULL pass): its end state is stored
// with kItemPieceEnd: the state is stored and kept, because the CTA goes on
// into the next segment's decay window with it (two-segment plans)
constexpr int kItemKeep = 16;

constexpr int kModeFull = 0, kModeCorrect = 1;

// One MMA work item: sequence bh, chunk start t0, token rows [r0, r1), flags,
// chunk counter lc, and (CTA pair) the index of the operand exchange it
// needs, or -1.
struct ItemInfo {
    int t0, r0, r1, flags, lc, xi, bh, pad;
};

// A chunk load request (t0 of sequence bh), or the end of the requests.
struct ChunkReq {
    int t0, first_item, end, bh;
};


enum Bar {
    kBarQkFull = 0, kBarQkEmpty, kBarItem0, kBarItem1, kBarPFull, kBarPSplit, kBarSDone, kBarSReady,
    kBarOFull0, kBarOFull1, kBarOFree0, kBarOFree1, kBarVFull0, kBarVFull1, kBarVEmpty0,
    kBarVEmpty1, kBarAFull, kBarQkRaw, kBarReq, kBarXchg0, kBarXchg1, kBarVerd0, kBarVerd1,
    kBarDrain, kNumBars
};
// arrival counts, in enum order (a CTA pair doubles kBarQkEmpty: both MMAs commit to it)
__device__ constexpr uint32_t kBarCounts[kNumBars] = {kPrepWarps, 1, 1, 1, 1, 4, 1, 4, 1, 1, 4, 4,
                                                      1, 1, 4, 4, 1, 1, 1, 1, 1, 1, 1, 1};

template <int DK, int DVT, bool PAIR>
struct Smem {
    static constexpr int kDKA = PAIR ? DK / 2 : DK;       // key channels prepared here
    static constexpr uint32_t kQBytes = kChunk * DK * 2;
    static constexpr uint32_t kQ = 0;                     // Qh (rescaled in place when single)
    static constexpr uint32_t kK = kQ + kQBytes;          // Kh_hi
    static constexpr uint32_t kKlo = kK + kQBytes;        // Kh_lo
    static constexpr uint32_t kA = kKlo + kQBytes;        // fp32 log gates [128][kDKA]
    static constexpr uint32_t kABytes = kChunk * kDKA * 4;
    static constexpr uint32_t kRaw = kA + kABytes;        // pair: raw Q, K of this CTA's channels
    static constexpr uint32_t kRawBytes = PAIR ? 2 * kBlk : 0;
    static constexpr uint32_t kVBytes = kChunk * DVT * 2;
    static constexpr uint32_t kSBlk = DK * 128;
    static constexpr uint32_t kSBytes = DK * DVT * 2;
    // V tiles: two slots where they fit (the next chunk's V loads while this
    // chunk's products read the other slot), else one
    static constexpr uint32_t kRest = 2 * DK * 4 + 64 + 16 + 16 + 8 * kNumBars + 16 + 1024;
    static constexpr int kVSlots =
        (kRaw + kRawBytes + 2 * kVBytes + kSBytes + kRest) <= 232448u ? 2 : 1;
    static constexpr uint32_t kV = kRaw + kRawBytes;      // V slots
    static constexpr uint32_t kS = kV + kVSlots * kVBytes;
    static constexpr uint32_t kG = kS + kSBytes;          // float [2][DK]: state scale per item
    static constexpr uint32_t kItem = kG + 2 * DK * 4;    // ItemInfo[2]
    static constexpr uint32_t kReq = kItem + 64;          // ChunkReq
    static constexpr uint32_t kVerd = kReq + 16;          // pair: the peer's verdicts [2]
    static constexpr uint32_t kBar = kVerd + (PAIR ? 16 : 0);  // mbarriers
    static constexpr uint32_t kMisc = kBar + 8 * kNumBars;  // tmem slot
    static constexpr uint32_t kTotal = kMisc + 16;
    // At least 120 KB so that only one CTA fits on an SM: each CTA allocates
    // all 512 TMEM columns.
    static constexpr uint32_t kAlloc = (kTotal + 1024) > 122880u ? (kTotal + 1024) : 122880u;
    static_assert(kAlloc <= 232448, "shared memory budget exceeded");
    static_assert(!PAIR || DK == 128, "CTA pairs split 128 key channels into two 64-channel blocks");
    static_assert(kG % 16 == 0, "bulk copies move 16-byte units");
};

// TMEM columns: P [0,128), O0 [128,128+DVT), O1, S after them.  P holds the
// fp32 scores of key tokens j = column; each 16-column piece (tokens 16 p ..
// 16 p + 15) is then replaced in place by its bf16 hi pairs (first 8 columns)
// and lo pairs (last 8), the A operand of the P V products.
template <int DVT>
struct Tmem {
    static constexpr uint32_t kP = 0, kO0 = 128, kO1 = 128 + DVT, kS = 128 + 2 * DVT;
    static constexpr uint32_t kCols = 512;
};

struct KParams {
    CUtensorMap tm_q, tm_k, tm_a, tm_v, tm_o32;
    const uint32_t *q;  // bf16 pairs
    const uint32_t *k;
    const float2 *a;
    const float *g;     // one gate per (sequence, token), [BH][T] (SCALAR kernels), else null
    const float *h0;
    float *hT;
    __nv_bfloat16 *o;
    float *ws_state;    // [seg_max][BH][DK][dv]: segment end states S*
    float *ws_decay;    // [seg_max][BH][DK]: segment total log-decays G
    float scale;
    int BH, T, dv;   // sequences, token rows per tensor head, value columns
    // Work split: the chunks of all BH sequences, one after another, cut into
    // ranges of L chunks, one range per CTA (per cluster for a CTA pair) of
    // the FULL pass.  A cut inside a sequence starts a new segment of it.
    int NC;        // chunks per sequence (fixed-length batches)
    int L;         // chunks per range
    int seg_max;   // most segments any sequence has
    long long total;   // chunks of all sequences
    // Packed variable-length batches: per packed sequence n, {first token row,
    // length, chunks, chunk offset (the chunks of the sequences before it)};
    // sequence u = n H + h.  Null for fixed-length batches, where sequence u
    // is tensor head u, rows [0, T).
    const int4 *seqs;
    int NS, H;
    int mode, force_sub;
    // Two-segment plans (CTA pairs): the CTA of a sequence's first segment,
    // whose start state is exact, goes on through the second segment's decay
    // window, storing its outputs, in place of the correction pass.
    int fuse;
    long long n_units;   // CTAs (clusters) per tile column in this launch
    unsigned int *status;
    unsigned long long wait_ns;   // limit of every bounded wait
    // Test instrumentation (null / 0 in production): the in-chunk prefix sums
    // of log_alpha the preparation used ([rows][DK] fp32, natural-log units,
    // relative to the reference of the token's block), the block length of
    // every chunk (by global chunk index), and a value tile the TMA thread
    // withholds (n > 0: the n-th chunk each CTA of the FULL pass serves gets
    // no V load, so that the waits for it expire).
    float *dbg_gamma;
    int *dbg_blk;
    int withhold_v;
};

// Where sequence u lives: tensor head z, token rows [y0, y0 + len), nch
// chunks, which are global chunks [a, a + nch) of the work split.
struct Seq {
    int z, y0, len, nch;
    long long a;
};

template <bool PACKED>
__device__ __forceinline__ Seq seq_of(const KParams &p, int u) {
    Seq s;
    if constexpr (!PACKED) {
        s.z = u;
        s.y0 = 0;
        s.len = p.T;
        s.nch = p.NC;
        s.a = static_cast<long long>(u) * p.NC;
    } else {
        const int n = u / p.H, h = u - n * p.H;
        const int4 e = p.seqs[n];
        s.z = h;
        s.y0 = e.x;
        s.len = e.y;
        s.nch = e.z;
        s.a = static_cast<long long>(p.H) * e.w + static_cast<long long>(h) * e.z;
    }
    return s;
}

// Segment geometry of the work split (identical on the host): cuts fall at
// multiples of L.
template <bool PACKED>
__device__ __forceinline__ int nseg_of(const KParams &p, int u) {
    const Seq q = seq_of<PACKED>(p, u);
    return 1 + static_cast<int>((q.a + q.nch - 1) / p.L - q.a / p.L);
}
template <bool PACKED>
__device__ __forceinline__ int seg_start(const KParams &p, int u, int s) {
    if (s == 0) return 0;
    const long long a = seq_of<PACKED>(p, u).a;
    return static_cast<int>((a / p.L + s) * p.L - a);
}

// End (global chunk) of this CTA's FULL-pass range, recomputed from the block
// index where needed instead of being held in registers.
__device__ __forceinline__ long long full_range_end(const KParams &p) {
    const long long unit = blockIdx.y + static_cast<long long>(blockIdx.z) * gridDim.y;
    return min((unit + 1) * p.L, p.total);
}

// One piece of a CTA's range: chunks [c0, c1) of sequence u, its segment seg.
struct Piece {
    int u, c0, c1, seg;
};

// The piece that starts at global chunk g of a range ending at g_end.
template <bool PACKED>
__device__ __forceinline__ Piece piece_at(const KParams &p, long long g, long long g_end) {
    int u;
    if constexpr (!PACKED) {
        u = static_cast<int>(g / p.NC);
    } else {
        // the packed sequence whose chunks (all heads) hold g: the last n with
        // H * offset(n) <= g, which has chunks (an empty one is always followed
        // by one that qualifies too)
        int lo = 0, hi = p.NS - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (static_cast<long long>(p.H) * p.seqs[mid].w <= g) lo = mid;
            else hi = mid - 1;
        }
        const int4 e = p.seqs[lo];
        u = lo * p.H + static_cast<int>((g - static_cast<long long>(p.H) * e.w) / e.z);
    }
    const Seq q = seq_of<PACKED>(p, u);
    Piece pc;
    pc.u = u;
    pc.c0 = static_cast<int>(g - q.a);
    pc.c1 = static_cast<int>(min(static_cast<long long>(q.nch), pc.c0 + (g_end - g)));
    pc.seg = static_cast<int>(g / p.L - q.a / p.L);
    return pc;
}

// Valid token rows of the chunk starting at row t0 of sequence u (the rest of
// the tile belongs past its end: zero gates and operands there).
template <bool PACKED>
__device__ __forceinline__ int valid_rows(const KParams &p, int u, int t0) {
    if constexpr (!PACKED) return kChunk;   // rows past T are the tensor maps' zero fill
    return min(kChunk, seq_of<PACKED>(p, u).len - t0);
}

__device__ __forceinline__ bool bar_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) { return pack_bf16x2(lo, hi); }

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Split (x, y) into a bf16 hi pair and a bf16 lo pair, x = hi + lo to 16
// significant bits.  Two packed conversions; the hi halves are widened back
// to fp32 by bit shifts.
__device__ __forceinline__ void split_pair(float x, float y, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16x2(x, y);
    const float2 h = unpack_bf16x2(hi);
    lo = pack_bf16x2(x - h.x, y - h.y);
}

__device__ __forceinline__ float clamp_gate(float a) {
    return fminf(fmaxf(a, -kExpBound), kExpBound);
}

// Causal split of one 32-column block of P (key tokens j0 .. j0 + 31) for
// row i, from its fp32 scores r: both 16-column pieces are stored back in
// place as 8 columns of bf16 hi pairs followed by 8 of lo pairs, with the
// entries j > i zeroed where the block holds the diagonal (`diag`, uniform
// over the warp).  One piece is stored before the next is split.
__device__ __forceinline__ void split_p_block(uint32_t taddr, const uint32_t (&r)[32], int j0, int i,
                                              bool diag) {
#pragma unroll
    for (int pc = 0; pc < 2; ++pc) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float x0 = __uint_as_float(r[16 * pc + 2 * e]);
            float x1 = __uint_as_float(r[16 * pc + 2 * e + 1]);
            if (diag) {
                const int j = j0 + 16 * pc + 2 * e;
                x0 = j <= i ? x0 : 0.f;
                x1 = j + 1 <= i ? x1 : 0.f;
            }
            split_pair(x0, x1, w[e], w[8 + e]);
        }
        tmem_st16(taddr + 16 * pc, w);
    }
}

// A 32-column block of P past the diagonal for every row of the warp: zeros.
__device__ __forceinline__ void zero_p_block(uint32_t taddr) {
    uint32_t z[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) z[e] = 0u;
    tmem_st16(taddr, z);
    tmem_st16(taddr + 16, z);
}

// Test instrumentation: the in-chunk prefix sums of token t (of sequence u)
// for channels ch and ch + 1, given in log2 units, stored in natural-log units.
// The limit of every bounded wait: the library's, or (instrumented builds
// only) the caller's shorter one.
template <bool DBG>
__device__ __forceinline__ unsigned long long wait_limit(const KParams &p) {
    if constexpr (DBG) return p.wait_ns;
    return kWaitLimitNs;
}

template <bool PACKED>
__device__ __forceinline__ void dbg_gamma_pair(const KParams &p, int u, int t, int ch, float g0,
                                               float g1, int dk) {
    const Seq sq = seq_of<PACKED>(p, u);
    if (t >= sq.len) return;
    const size_t row = static_cast<size_t>(sq.z) * p.T + sq.y0 + t;
    *reinterpret_cast<float2 *>(p.dbg_gamma + row * dk + ch) = make_float2(g0 * kLn2, g1 * kLn2);
}

// Sub-chunk rescaling of one chunk (prep threads): the largest power-of-two
// block length cs whose every block keeps |Gamma - r_block| <= kExpBound
// (clamped gates); each block becomes one item, written to the operand tiles
// with its own reference.  Gates, Q and K are read from global memory.
// Thread pt owns the channel pair 2*(pt % (DK/2)) of token part pt / (DK/2).
// `n` counts items; `last_flags` go to the chunk's last item; gtot0/gtot1
// return the chunk's clamped Gamma at its end for the thread's channels (valid
// in the last token part).  Returns false if a bounded wait expired.
template <int DK, bool PACKED, bool SCALAR, bool FOLD, bool DBG, typename BeforeEmptyWait>
__device__ __forceinline__ bool sub_chunk_items(const KParams &p, int dbg_block, int bh, int t0,
                                                int lc, bool store, int last_flags, int pt,
                                                uint8_t *sQ,
                                                uint8_t *sK,
                                                uint8_t *sKlo, float *sG, ItemInfo *sItem,
                                                uint64_t *bars, int &n, float &gtot0,
                                                float &gtot1, BeforeEmptyWait &&before_empty_wait) {
    constexpr int NP = DK / 2;
    constexpr int NQ = kPrepThreads / NP;
    constexpr int TP = kChunk / NQ;
    constexpr int kStride = DK / 2;     // row stride in bf16 pairs
    const int pr = pt % NP, part = pt / NP;
    const int ch = 2 * pr;
    const bool last_part = part == NQ - 1;
    const int lane = pt & 31;
    const Seq sq = seq_of<PACKED>(p, bh);
    const int T = sq.len;                        // rows past it are zero
    const size_t row0 = static_cast<size_t>(sq.z) * p.T + sq.y0;
    const uint32_t *qb = p.q + (row0 * DK + ch) / 2;
    const uint32_t *kb = p.k + (row0 * DK + ch) / 2;
    auto raw_gate = [&](int i) {
        const int t = t0 + i;
        if constexpr (SCALAR) {
            const float g = t < T ? p.g[row0 + t] : 0.f;
            return make_float2(g, g);
        } else {
            const float2 *ab = p.a + (row0 * DK + ch) / 2;
            return t < T ? ab[static_cast<size_t>(t) * kStride] : make_float2(0.f, 0.f);
        }
    };
    float bnd0[NQ], bnd1[NQ];  // clamped Gamma just before each part start
    {
        float c0 = 0.f, c1 = 0.f;
        bnd0[0] = 0.f;
        bnd1[0] = 0.f;
        for (int qq = 1; qq < NQ; ++qq) {
            for (int i = (qq - 1) * TP; i < qq * TP; ++i) {
                const float2 a = raw_gate(i);
                c0 += clamp_gate(a.x);
                c1 += clamp_gate(a.y);
            }
            bnd0[qq] = c0;
            bnd1[qq] = c1;
        }
    }
    int cs = 64;
    for (; cs > 1; cs >>= 1) {
        float c0 = bnd0[part], c1 = bnd1[part];
        const int s_first = (part * TP) / cs * cs;
        float r0 = (s_first >= part * TP) ? c0 : bnd0[s_first / TP];
        float r1 = (s_first >= part * TP) ? c1 : bnd1[s_first / TP];
        bool viol = false;
        for (int ii = 0; ii < TP; ++ii) {
            const int i = part * TP + ii;
            if (i % cs == 0) {
                r0 = c0;
                r1 = c1;
            }
            const float2 a = raw_gate(i);
            c0 += clamp_gate(a.x);
            c1 += clamp_gate(a.y);
            viol |= fabsf(c0 - r0) > kExpBound || fabsf(c1 - r1) > kExpBound;
        }
        if (!bar_or(3, kPrepThreads, viol)) break;
    }
    // cs == 1 always satisfies the bound: a single clamped gate is within it.
    const int n_sub = kChunk / cs;
    const bool dbg = DBG && p.dbg_gamma != nullptr && (dbg_block == -1 || (ch >> 6) == dbg_block);
    if (DBG && p.dbg_blk != nullptr && dbg_block != -2 && pt == 0) p.dbg_blk[sq.a + t0 / kChunk] = cs;
    bool ok = true;
    for (int sidx = 0; sidx < n_sub; ++sidx) {
        const int sa = sidx * cs, sb = sa + cs;
        bool okw = true;
        if (sidx > 0) {
            before_empty_wait();
            okw = mbar_wait_bounded(&bars[kBarQkEmpty], (n - 1) & 1, p.status, wait_limit<DBG>(p));
        }
        ok = !bar_or(4, kPrepThreads, !okw);
        if (!ok) break;
        // reference for block sidx: clamped Gamma just before token sa
        float c0 = bnd0[part], c1 = bnd1[part];
        float r0 = 0.f, r1 = 0.f;
        if (sa <= part * TP) {
            r0 = bnd0[sa / TP];
            r1 = bnd1[sa / TP];
        }
        for (int ii = 0; ii < TP; ++ii) {
            const int i = part * TP + ii;
            if (i == sa) {
                r0 = c0;
                r1 = c1;
            }
            const int t = t0 + i;
            const float2 a = raw_gate(i);
            c0 += clamp_gate(a.x);
            c1 += clamp_gate(a.y);
            const uint32_t off = sw128_offset(i, ch, kBlk);
            uint32_t hi = 0u, lo = 0u, qv = 0u;
            if (i >= sa && i < sb && t < T) {
                if (dbg)
                    *reinterpret_cast<float2 *>(p.dbg_gamma + (row0 + t) * DK + ch) =
                        make_float2(c0 - r0, c1 - r1);
                const float2 qf = unpack_bf16x2(qb[static_cast<size_t>(t) * kStride]);
                const float2 kf = unpack_bf16x2(kb[static_cast<size_t>(t) * kStride]);
                const float qs = FOLD ? p.scale : 1.f;
                qv = bf16x2_bits(qf.x * qs * __expf(c0 - r0), qf.y * qs * __expf(c1 - r1));
                split_pair(kf.x * __expf(r0 - c0), kf.y * __expf(r1 - c1), hi, lo);
            }
            *reinterpret_cast<uint32_t *>(sQ + off) = qv;
            *reinterpret_cast<uint32_t *>(sK + off) = hi;
            *reinterpret_cast<uint32_t *>(sKlo + off) = lo;
            if (i == sb - 1) {
                sG[(n & 1) * DK + ch] = __expf(c0 - r0);
                sG[(n & 1) * DK + ch + 1] = __expf(c1 - r1);
            }
        }
        if (last_part) {
            gtot0 = c0;
            gtot1 = c1;
        }
        if (pt == 0) {
            sItem[n & 1] = ItemInfo{
                t0, sa, sb,
                (sidx == n_sub - 1 ? (kItemLast | last_flags) : 0) | (store ? kItemStore : 0), lc,
                -1, bh, 0};
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarQkFull]);
        ++n;
    }
    return ok;
}

// Prep warps of one CTA of a pair.  The CTA owns key channels
// [64 rank, 64 rank + 64): 32 channel pairs x 8 token parts of 16 tokens.
// Per chunk c:
//   1. phase A on the A half tile: in-chunk prefix sums in place, part
//      offsets, and the exponent-bound verdict for these channels, which is
//      sent to the peer at once (one remote word);
//   2. phase B into registers from the raw Q and K staging tiles (Qh, Kh_hi,
//      Kh_lo for 16 tokens x 2 channels); the A and staging tiles are then
//      free and chunk c+1 is requested, so its loads overlap this chunk;
//   3. the segment decay of every channel through chunk c-1, from the state
//      factors of the previous exchange, and the window decision for chunk c;
//   4. if neither CTA's channels broke the bound: once both CTAs' MMAs have
//      released the operand tiles, the registers go to this CTA's 64-channel
//      block of the Qh, Kh_hi and Kh_lo tiles, its half of the state factors
//      e^Gamma_C to the factor table, and all four are copied into the
//      peer's shared memory at the same offsets.  The item is published at
//      once; the MMA issuer (and the TMEM warps, for the factors) wait for the
//      peer's copy themselves, so the prep warps go on to chunk c+1.
//      Otherwise both CTAs run the sub-chunk path over all channels on their
//      own (same inputs, same items).
// Threads pt < DK keep the decay since the segment start of channel pt; both
// CTAs compute it from identical bits (the exchanged factor table, or the raw
// gates), so their window decisions agree.
template <int DK, int DVT, bool PACKED, bool SCALAR, bool DBG>
__device__ __forceinline__ void prep_pair(const KParams &p, uint8_t *smem, uint32_t rank,
                                          long long g_begin, long long g_end, size_t BHn,
                                          int dv_tile) {
    using L = Smem<DK, DVT, true>;
    constexpr int DKH = DK / 2;                 // channels prepared by this CTA
    constexpr int NP = DKH / 2;                 // channel pairs
    constexpr int NQ = kPrepThreads / NP;       // token parts
    constexpr int TP = kChunk / NQ;             // tokens per part
    constexpr uint32_t kXchgBytes = 3u * kBlk + DKH * 4u;
    uint8_t *sQ = smem + L::kQ;
    uint8_t *sK = smem + L::kK;
    uint8_t *sKlo = smem + L::kKlo;
    const uint8_t *sRawQ = smem + L::kRaw;
    const uint8_t *sRawK = sRawQ + kBlk;
    float *sA = reinterpret_cast<float *>(smem + L::kA);
    float *sG = reinterpret_cast<float *>(smem + L::kG);
    ItemInfo *sItem = reinterpret_cast<ItemInfo *>(smem + L::kItem);
    ChunkReq *sReq = reinterpret_cast<ChunkReq *>(smem + L::kReq);
    uint32_t *sVerd = reinterpret_cast<uint32_t *>(smem + L::kVerd);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBar);

    const int pt = threadIdx.x;
    const int lane = pt & 31;
    const int pr = pt % NP, part = pt / NP;
    const int chl = 2 * pr;                      // channel within this CTA's half
    const int ch = static_cast<int>(rank) * DKH + chl;
    const bool last_part = part == NQ - 1;
    const float *sAc = sA + chl;
    const uint32_t peer = rank ^ 1u;

    // the pieces of this CTA's range, one after another: the current piece is
    // chunks [c, c_end) of sequence bh (the rest is recomputed at piece ends)
    int bh, c, c_end, seg_cur;
    bool closed;
    {
        const Piece pc = piece_at<PACKED>(p, g_begin, g_end);
        bh = pc.u;
        c = pc.c0;
        c_end = pc.c1;
        seg_cur = pc.seg;
        closed = p.mode == kModeFull && pc.seg == 0;
    }
    // correction semantics (every output stored, stop once the window has
    // closed): the correction pass, or a first segment's CTA going on into
    // the second segment's window
    bool corr = p.mode == kModeCorrect;
    // whether the current piece, a first segment whose start state is exact,
    // is followed by the second segment's window in this CTA
    auto continues = [&]() {
        return p.fuse != 0 && !corr && seg_cur == 0 && nseg_of<PACKED>(p, bh) == 2;
    };
    float gseg = 0.f;                            // threads pt < DK: channel pt
    int n = 0;                                   // items published
    int nx = 0;                                  // operand exchanges made
    int used = 0;                                // chunks published
    bool ok = true;
    bool pend = false;                           // last exchange's factors not yet read
    bool prepped_last = false;                   // the last chunk prepared was not used
    bool spec = false;                           // chunk lc_last + 1 requested, A not yet landed
    int lc_last = 0;
    if (pt == 0) {
        sReq[0] = ChunkReq{c * kChunk, 0, 0, bh};
        mbar_arrive(&bars[kBarReq]);
    }
    // A wait that expires clears `ok` in its thread only: every thread still
    // runs the same sequence of barriers (each wait is bounded), and the loop
    // ends at the next chunk boundary, where the threads' verdicts are combined.
    for (int lc = 0;; ++lc) {
        ok = !bar_or(4, kPrepThreads, !ok);
        const bool have = c < c_end && ok;
        const int t0 = c * kChunk;
        uint32_t rq[TP], rh[TP], rl[TP];
        float gc0 = 0.f, gc1 = 0.f;
        bool bad_here = false;
        if (have) {
            // ---- phase A: prefix sums of this thread's part (log2 units) in
            // registers; the part total goes to the A tile's last row of the part
            if (pt == 0) mbar_arrive_expect_tx(&bars[kBarVerd0 + (lc & 1)], 4u);
            ok &= mbar_wait_bounded(&bars[kBarAFull], lc & 1, p.status, wait_limit<DBG>(p));
            spec = false;
            // rows past the sequence end (the tail of a packed sequence) count
            // as gate 0 and operands 0
            const int valid = valid_rows<PACKED>(p, bh, t0);
            float c0 = 0.f, c1 = 0.f;
            float lmn = 3.0e38f, lmx = -3.0e38f;
            float2 av[TP];
            if constexpr (SCALAR) {
                // one gate per token, the same for every channel
                const Seq sq = seq_of<PACKED>(p, bh);
                const float *gr = p.g + static_cast<size_t>(sq.z) * p.T + sq.y0 + t0 + part * TP;
                const int left = sq.len - t0 - part * TP;
#pragma unroll
                for (int e = 0; e < TP; ++e) {
                    const float g = e < left ? __ldg(gr + e) : 0.f;
                    av[e] = make_float2(g, g);
                }
            } else {
#pragma unroll
                for (int e = 0; e < TP; ++e)
                    av[e] = *reinterpret_cast<const float2 *>(sAc + (part * TP + e) * DKH);
            }
            if (PACKED && valid < kChunk) {
#pragma unroll
                for (int e = 0; e < TP; ++e)
                    if (part * TP + e >= valid) av[e] = make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int e = 0; e < TP; ++e) {
                c0 = fmaf(av[e].x, kLog2e, c0);
                c1 = fmaf(av[e].y, kLog2e, c1);
                av[e] = make_float2(c0, c1);
                lmn = fminf(lmn, fminf(c0, c1));
                lmx = fmaxf(lmx, fmaxf(c0, c1));
            }
            *reinterpret_cast<float2 *>(sA + chl + (part * TP + TP - 1) * DKH) = make_float2(c0, c1);
            named_barrier(5, kPrepThreads);
            float o0 = 0.f, o1 = 0.f;
#pragma unroll
            for (int qq = 0; qq < NQ - 1; ++qq) {
                if (qq < part) {
                    const float2 tt =
                        *reinterpret_cast<const float2 *>(sAc + (qq * TP + TP - 1) * DKH);
                    o0 += tt.x;
                    o1 += tt.y;
                }
            }
            const float gmin = fminf(o0, o1) + lmn, gmax = fmaxf(o0, o1) + lmx;
            bad_here = bar_or(2, kPrepThreads,
                              fmaxf(-fminf(gmin, 0.f), fmaxf(gmax, 0.f)) > kExpBound2 ||
                                  p.force_sub != 0);
            if (pt == 0) {
                const uint32_t dst = mapa_shared(smem_u32(&sVerd[lc & 1]), peer);
                const uint32_t pbar = mapa_shared(smem_u32(&bars[kBarVerd0 + (lc & 1)]), peer);
                st_async_to_peer(dst, bad_here ? 1u : 0u, pbar);
            }
            // ---- phase B into registers (values of a chunk that broke the
            // bound are computed but never used)
            ok &= mbar_wait_bounded(&bars[kBarQkRaw], lc & 1, p.status, wait_limit<DBG>(p));
#pragma unroll
            for (int e = 0; e < TP; ++e) {
                const int i = part * TP + e;
                const uint32_t off = sw128_offset(i, chl, kBlk);
                const bool in = !PACKED || i < valid;
                const float2 qf =
                    unpack_bf16x2(in ? *reinterpret_cast<const uint32_t *>(sRawQ + off) : 0u);
                const float2 kf =
                    unpack_bf16x2(in ? *reinterpret_cast<const uint32_t *>(sRawK + off) : 0u);
                const float g0 = o0 + av[e].x, g1 = o1 + av[e].y;
                rq[e] = bf16x2_bits(qf.x * p.scale * ex2f(g0), qf.y * p.scale * ex2f(g1));
                split_pair(kf.x * ex2f(-g0), kf.y * ex2f(-g1), rh[e], rl[e]);
                if (DBG && p.dbg_gamma != nullptr) dbg_gamma_pair<PACKED>(p, bh, t0 + i, ch, g0, g1, DK);
            }
            gc0 = o0 + c0;                       // Gamma log2 e at the chunk end (last part)
            gc1 = o1 + c1;
            // the A and staging tiles are consumed: start the next chunk's loads
            named_barrier(5, kPrepThreads);
            // the next chunk of the stream: in this piece, or the next piece's first
            int nc = -1, nbh = bh;
            if (c + 1 < c_end) {
                nc = c + 1;
            } else if (continues()) {
                nc = c + 1;                      // the second segment's first chunk
            } else if (p.mode == kModeFull && !corr) {
                const long long gn = seq_of<PACKED>(p, bh).a + c_end, ge = full_range_end(p);
                if (gn < ge) {
                    const Piece next = piece_at<PACKED>(p, gn, ge);
                    nc = next.c0;
                    nbh = next.u;
                }
            }
            if (nc >= 0) {
                if (pt == 0) {
                    sReq[0] = ChunkReq{nc * kChunk, 0, 0, nbh};
                    mbar_arrive(&bars[kBarReq]);
                }
                spec = true;   // taken by the TMA thread once A(next) has landed
            }
            prepped_last = true;
            lc_last = lc;
        }
        // ---- segment decay through chunk c-1 (the previous exchange's factors)
        if (pend) {
            const int x = nx - 1;
            ok &= mbar_wait_bounded(&bars[kBarXchg0 + (x & 1)], (x >> 1) & 1, p.status, wait_limit<DBG>(p));
            if (pt < DK) gseg += __logf(sG[((n - 1) & 1) * DK + pt]);
            pend = false;
        }
        // ---- end of the segment, or (correction pass) of the decay window
        const bool win = !closed && pt < DK && gseg > -kWindowCut;
        const bool any_win = bar_or(1, kPrepThreads, win);
        if (!closed && !any_win) closed = true;
        if (!have || (corr && closed)) break;
        const bool store = corr || closed;
        // the FULL pass stores the state at the end of every piece (and keeps
        // it when the CTA goes on into the next segment's window)
        const int piece_end = (p.mode == kModeFull && !corr && c + 1 == c_end)
                                  ? (kItemPieceEnd | (continues() ? kItemKeep : 0))
                                  : 0;
        // ---- both CTAs' verdicts: one branch for all threads, even for one
        // whose wait expired
        ok &= mbar_wait_bounded(&bars[kBarVerd0 + (lc & 1)], (lc >> 1) & 1, p.status, wait_limit<DBG>(p));
        const bool bad = bar_or(2, kPrepThreads, bad_here || sVerd[lc & 1] != 0u);
        prepped_last = false;
        ++used;
        if (!bad) {
            // ---- both CTAs' MMAs are done with the previous item's tiles
            if (n > 0) ok &= mbar_wait_bounded(&bars[kBarQkEmpty], (n - 1) & 1, p.status, wait_limit<DBG>(p));
#pragma unroll
            for (int e = 0; e < TP; ++e) {
                const uint32_t off = sw128_offset(part * TP + e, ch, kBlk);
                *reinterpret_cast<uint32_t *>(sQ + off) = rq[e];
                *reinterpret_cast<uint32_t *>(sK + off) = rh[e];
                *reinterpret_cast<uint32_t *>(sKlo + off) = rl[e];
            }
            if (last_part) {
                sG[(n & 1) * DK + ch] = ex2f(gc0);
                sG[(n & 1) * DK + ch + 1] = ex2f(gc1);
            }
            fence_proxy_async_smem();
            named_barrier(5, kPrepThreads);
            if (pt == 0) {
                if (DBG && p.dbg_blk != nullptr && rank == 0) p.dbg_blk[seq_of<PACKED>(p, bh).a + c] = kChunk;
                sItem[n & 1] = ItemInfo{t0, 0, kChunk,
                                        kItemLast | (store ? kItemStore : 0) | piece_end, lc, nx,
                                        bh, 0};
                mbar_arrive_expect_tx(&bars[kBarXchg0 + (nx & 1)], kXchgBytes);
                const uint32_t pbar = mapa_shared(smem_u32(&bars[kBarXchg0 + (nx & 1)]), peer);
                const uint32_t blk = rank * kBlk;
                float *g_own = sG + (n & 1) * DK + rank * DKH;
                bulk_copy_to_peer(mapa_shared(smem_u32(sQ + blk), peer), sQ + blk, kBlk, pbar);
                bulk_copy_to_peer(mapa_shared(smem_u32(sK + blk), peer), sK + blk, kBlk, pbar);
                bulk_copy_to_peer(mapa_shared(smem_u32(sKlo + blk), peer), sKlo + blk, kBlk, pbar);
                bulk_copy_to_peer(mapa_shared(smem_u32(g_own), peer), g_own, DKH * 4u, pbar);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kBarQkFull]);
            ++n;
            ++nx;
            pend = true;
        } else {
            // ---- a chunk whose decay breaks the bound: sub-chunk items over all
            // channels, computed by each CTA of the pair on its own
            if (n > 0) ok &= mbar_wait_bounded(&bars[kBarQkEmpty], (n - 1) & 1, p.status, wait_limit<DBG>(p));
            float gt0 = 0.f, gt1 = 0.f;
            ok &= sub_chunk_items<DK, PACKED, SCALAR, true, DBG>(p, static_cast<int>(rank), bh, t0, lc, store, piece_end, pt, sQ, sK, sKlo, sG, sItem,
                                      bars, n, gt0, gt1, [] {});
            if (pt < DK) {
                // the chunk's clamped decay of channel pt, summed in token order
                const Seq sq = seq_of<PACKED>(p, bh);
                const size_t row0 = static_cast<size_t>(sq.z) * p.T + sq.y0;
                float gsum = 0.f;
                for (int i = 0; i < kChunk && t0 + i < sq.len; ++i)
                    gsum += clamp_gate(SCALAR ? p.g[row0 + t0 + i]
                                              : reinterpret_cast<const float *>(
                                                    p.a)[(row0 + t0 + i) * DK + pt]);
                gseg += gsum;
            }
        }
        ++c;
        if (piece_end) {
            // ---- end of a FULL-pass piece: its decay, then the next piece
            if (pend) {
                const int x = nx - 1;
                ok &= mbar_wait_bounded(&bars[kBarXchg0 + (x & 1)], (x >> 1) & 1, p.status, wait_limit<DBG>(p));
                if (pt < DK) gseg += __logf(sG[((n - 1) & 1) * DK + pt]);
                pend = false;
            }
            const long long a = seq_of<PACKED>(p, bh).a;
            if (nseg_of<PACKED>(p, bh) > 1 && dv_tile == 0 && pt < DK) {
                const int seg = static_cast<int>((a + c_end - 1) / p.L - a / p.L);
                p.ws_decay[(static_cast<size_t>(seg) * BHn + bh) * DK + pt] = gseg;
            }
            if (piece_end & kItemKeep) {
                // on into the second segment's window, with the exact state
                corr = true;
                seg_cur = 1;
                c_end = seq_of<PACKED>(p, bh).nch;
                gseg = 0.f;
                closed = false;
                continue;
            }
            const long long gn = a + c_end, ge = full_range_end(p);
            if (gn >= ge) break;
            const Piece next = piece_at<PACKED>(p, gn, ge);
            bh = next.u;
            c = next.c0;
            c_end = next.c1;
            seg_cur = next.seg;
            gseg = 0.f;
            closed = next.seg == 0;
        }
    }
    // ---- end of the item stream and of the load requests
    if (pend) {
        const int x = nx - 1;
        ok &= mbar_wait_bounded(&bars[kBarXchg0 + (x & 1)], (x >> 1) & 1, p.status, wait_limit<DBG>(p));
        if (pt < DK) gseg += __logf(sG[((n - 1) & 1) * DK + pt]);
    }
    // the peer's verdict for a chunk prepared here but not used has to land
    // before this CTA may exit
    if (prepped_last) ok &= mbar_wait_bounded(&bars[kBarVerd0 + (lc_last & 1)], (lc_last >> 1) & 1, p.status, wait_limit<DBG>(p));
    // the request mailbox holds one request: the end may be posted only once
    // the TMA thread has taken the last one (its A tile has landed)
    if (spec) ok &= mbar_wait_bounded(&bars[kBarAFull], (lc_last + 1) & 1, p.status, wait_limit<DBG>(p));
    named_barrier(5, kPrepThreads);
    if (pt == 0) {
        // the count of chunks used, so that no V load waits for a tile never freed
        sReq[0] = ChunkReq{used, 0, 1, 0};
        mbar_arrive(&bars[kBarReq]);
    }
    if (n > 0 && !mbar_wait_bounded(&bars[kBarQkEmpty], (n - 1) & 1, p.status, wait_limit<DBG>(p))) ok = false;
    if (pt == 0) sItem[n & 1] = ItemInfo{0, 0, 0, kItemEnd, 0, -1, 0, 0};
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[kBarQkFull]);
}

template <int DK, int DVT, bool PAIR, bool PACKED, bool SCALAR, bool DBG = false>
__global__ void __launch_bounds__(kThreads, 1) chunk_fwd_kernel(const __grid_constant__ KParams p) {
    using L = Smem<DK, DVT, PAIR>;
    using TM = Tmem<DVT>;
    constexpr int VS = L::kVSlots;   // V tile slots: chunk j uses slot j % VS
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem + L::kQ;
    uint8_t *sK = smem + L::kK;
    uint8_t *sKlo = smem + L::kKlo;
    uint8_t *sV = smem + L::kV;
    uint8_t *sS = smem + L::kS;
    float *sA = reinterpret_cast<float *>(smem + L::kA);
    float *sG = reinterpret_cast<float *>(smem + L::kG);
    ItemInfo *sItem = reinterpret_cast<ItemInfo *>(smem + L::kItem);
    ChunkReq *sReq = reinterpret_cast<ChunkReq *>(smem + L::kReq);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int dv_tile = blockIdx.x;
    const int dv0 = dv_tile * DVT;
    const int T = p.T;
    const size_t BHn = static_cast<size_t>(p.BH);
    // This CTA's chunks: FULL pass, range `unit` of the work split (one or
    // more pieces); CORRECT pass, segment 1 + unit % (seg_max - 1) of
    // sequence unit / (seg_max - 1), if that sequence has it (a CTA pair's two
    // CTAs decide alike and leave together, before any cluster barrier or TMEM
    // allocation).
    const long long unit = blockIdx.y + static_cast<long long>(blockIdx.z) * gridDim.y;
    if (unit >= p.n_units) return;
    long long g_begin, g_end;
    if (p.mode == kModeFull) {
        g_begin = unit * p.L;
        g_end = min(g_begin + p.L, p.total);
    } else {
        const int u = static_cast<int>(unit / (p.seg_max - 1));
        const int sg = 1 + static_cast<int>(unit % (p.seg_max - 1));
        const int ns = nseg_of<PACKED>(p, u);
        if (sg >= ns) return;
        const Seq q = seq_of<PACKED>(p, u);
        g_begin = q.a + seg_start<PACKED>(p, u, sg);
        g_end = q.a + (sg + 1 < ns ? seg_start<PACKED>(p, u, sg + 1) : q.nch);
    }
    if (g_begin >= g_end) return;

    // CTA pair: the two value-column tiles of one head, cluster ranks 0 and 1
    // (rank == dv_tile); each prepares the operands of one half of the key
    // channels and sends them to the other.
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i)
            mbar_init(&bars[i], (PAIR && i == kBarQkEmpty) ? 2u : kBarCounts[i]);
        fence_mbar_init();
    }
    if (warp == kTmaWarp && lane == 0) {
        prefetch_tensormap(&p.tm_q);
        prefetch_tensormap(&p.tm_k);
        if (!SCALAR) prefetch_tensormap(&p.tm_a);
        prefetch_tensormap(&p.tm_v);
        prefetch_tensormap(&p.tm_o32);
    }
    if (warp == kMmaWarp) tmem_alloc(tmem_slot, TM::kCols);
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync_all();   // the peer's barriers exist before any remote use
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < kPrepWarps && PAIR) {
        if constexpr (PAIR) {
            prep_pair<DK, DVT, PACKED, SCALAR, DBG>(p, smem, rank, g_begin, g_end, BHn, dv_tile);
        }
    } else if (warp < kPrepWarps) {
        // =========================================================== prep warps
        constexpr int NP = DK / 2;              // channel pairs
        constexpr int NQ = kPrepThreads / NP;   // token parts
        constexpr int TP = kChunk / NQ;         // tokens per part
        static_assert(TP % 8 == 0, "token parts must hold whole batches");
        const int pt = tid;
        const int pr = pt % NP, part = pt / NP;
        const int ch = 2 * pr;
        const bool last_part = part == NQ - 1;
        const float *sAc = sA + ch;         // this thread's channel pair in the A tile
        int n = 0, lc = 0;
        bool ok = true;
        for (long long g = g_begin; g < g_end && ok;) {
          // ---- one piece: chunks [pc.c0, pc.c1) of sequence pc.u
          const Piece pc = piece_at<PACKED>(p, g, g_end);
          g += pc.c1 - pc.c0;
          const int bh = pc.u;
          float gseg0 = 0.f, gseg1 = 0.f;     // decay since the segment start (last part only)
          bool closed = (p.mode == kModeFull && pc.seg == 0);  // no correction window
          for (int c = pc.c0;; ++c, ++lc) {
            // ---- decide this chunk: past the piece end, or (correction pass)
            // past the point where the segment's start state has decayed away.
            // The reduction doubles as the barrier after which the previous
            // chunk's A tile is free.
            const bool win = !closed && last_part && (gseg0 > -kWindowCut || gseg1 > -kWindowCut);
            const bool any_win = bar_or(1, kPrepThreads, win);
            if (!closed && !any_win) closed = true;
            const bool end = c >= pc.c1 || !ok || (p.mode == kModeCorrect && closed);
            if (end) break;
            if (pt == 0) {
                sReq[0] = ChunkReq{c * kChunk, n, 0, bh};
                mbar_arrive(&bars[kBarReq]);
            }
            const int t0 = c * kChunk;
            // rows past the sequence end (the tail of a packed sequence) count
            // as gate 0 and operands 0
            const int valid = valid_rows<PACKED>(p, bh, t0);
            const bool store = p.mode == kModeCorrect || closed;
            // the FULL pass stores the state at the end of every piece
            const int piece_end = (p.mode == kModeFull && c + 1 == pc.c1) ? kItemPieceEnd : 0;
            // ---- phase A (needs only the A tile, which arrives early): the
            // local prefix sum of this thread's part, written in place of A.
            constexpr int kB = 8;
            bool okw = mbar_wait_bounded(&bars[kBarAFull], lc & 1, p.status, wait_limit<DBG>(p));
            ok = !bar_or(4, kPrepThreads, !okw);   // one verdict for all prep threads
            if (!ok) break;
            float c0 = 0.f, c1 = 0.f;
            float lmn = 3.0e38f, lmx = -3.0e38f;
            {
                // the gates of token i: this thread's channel pair of the A
                // tile, or the token's one gate for every channel
                const float *gr = nullptr;
                int left = kChunk;
                if constexpr (SCALAR) {
                    const Seq sq = seq_of<PACKED>(p, bh);
                    gr = p.g + static_cast<size_t>(sq.z) * p.T + sq.y0 + t0;
                    left = sq.len - t0;
                }
                auto gate = [&](int i) -> float2 {
                    if constexpr (SCALAR) {
                        const float g = i < left ? __ldg(gr + i) : 0.f;
                        return make_float2(g, g);
                    } else {
                        return *reinterpret_cast<const float2 *>(sAc + i * DK);
                    }
                };
                float2 nx[kB];
#pragma unroll
                for (int e = 0; e < kB; ++e) nx[e] = gate(part * TP + e);
                for (int i0 = part * TP; i0 < (part + 1) * TP; i0 += kB) {
                    float2 cur[kB];
#pragma unroll
                    for (int e = 0; e < kB; ++e)
                        cur[e] = (PACKED && i0 + e >= valid) ? make_float2(0.f, 0.f) : nx[e];
                    if (i0 + kB < (part + 1) * TP) {
#pragma unroll
                        for (int e = 0; e < kB; ++e) nx[e] = gate(i0 + kB + e);
                    }
#pragma unroll
                    for (int e = 0; e < kB; ++e) {
                        c0 = fmaf(cur[e].x, kLog2e, c0);   // log2 units
                        c1 = fmaf(cur[e].y, kLog2e, c1);
                        lmn = fminf(lmn, fminf(c0, c1));
                        lmx = fmaxf(lmx, fmaxf(c0, c1));
                        *reinterpret_cast<float2 *>(const_cast<float *>(sAc) + (i0 + e) * DK) =
                            make_float2(c0, c1);
                    }
                }
            }
            named_barrier(5, kPrepThreads);
            // offset of this part: the totals of the parts before it
            float o0 = 0.f, o1 = 0.f;
            for (int qq = 0; qq < part; ++qq) {
                const float2 tt = *reinterpret_cast<const float2 *>(sAc + (qq * TP + TP - 1) * DK);
                o0 += tt.x;
                o1 += tt.y;
            }
            // Gamma_i = o + local_i; the fast path needs every |Gamma_i| <= kExpBound
            const float gmin = fminf(o0, o1) + lmn, gmax = fmaxf(o0, o1) + lmx;
            const bool bad = bar_or(2, kPrepThreads,
                                    fmaxf(-fminf(gmin, 0.f), fmaxf(gmax, 0.f)) > kExpBound2 ||
                                        p.force_sub != 0);
            okw = mbar_wait_bounded(&bars[kBarQkRaw], lc & 1, p.status, wait_limit<DBG>(p));
            ok = !bar_or(4, kPrepThreads, !okw);
            if (!ok) break;
            if (!bad) {
                // ---- phase B (needs Q, K): Qh, Kh_hi in place, Kh_lo.  Purely
                // elementwise; the next batch's loads precede this batch's stores.
                if (last_part) {
                    const float gc0 = o0 + c0, gc1 = o1 + c1;   // Gamma log2 e at the chunk end
                    sG[(n & 1) * DK + ch] = ex2f(gc0);
                    sG[(n & 1) * DK + ch + 1] = ex2f(gc1);
                    gseg0 += gc0 * kLn2;
                    gseg1 += gc1 * kLn2;
                }
                float2 ab8[kB];
                uint32_t qw8[kB], kw8[kB];
#pragma unroll
                for (int e = 0; e < kB; ++e) {
                    const int i = part * TP + e;
                    const uint32_t off = sw128_offset(i, ch, kBlk);
                    ab8[e] = *reinterpret_cast<const float2 *>(sAc + i * DK);
                    qw8[e] = *reinterpret_cast<const uint32_t *>(sQ + off);
                    kw8[e] = *reinterpret_cast<const uint32_t *>(sK + off);
                }
                for (int i0 = part * TP; i0 < (part + 1) * TP; i0 += kB) {
                    float2 ca[kB];
                    uint32_t cq[kB], ck[kB];
#pragma unroll
                    for (int e = 0; e < kB; ++e) {
                        const bool in = !PACKED || i0 + e < valid;
                        ca[e] = ab8[e];
                        cq[e] = in ? qw8[e] : 0u;
                        ck[e] = in ? kw8[e] : 0u;
                    }
                    if (i0 + kB < (part + 1) * TP) {
#pragma unroll
                        for (int e = 0; e < kB; ++e) {
                            const int i = i0 + kB + e;
                            const uint32_t off = sw128_offset(i, ch, kBlk);
                            ab8[e] = *reinterpret_cast<const float2 *>(sAc + i * DK);
                            qw8[e] = *reinterpret_cast<const uint32_t *>(sQ + off);
                            kw8[e] = *reinterpret_cast<const uint32_t *>(sK + off);
                        }
                    }
#pragma unroll
                    for (int e = 0; e < kB; ++e) {
                        const int i = i0 + e;
                        const float g0 = o0 + ca[e].x, g1 = o1 + ca[e].y;
                        if (DBG && p.dbg_gamma != nullptr && dv_tile == 0)
                            dbg_gamma_pair<PACKED>(p, bh, t0 + i, ch, g0, g1, DK);
                        const float2 qf = unpack_bf16x2(cq[e]), kf = unpack_bf16x2(ck[e]);
                        const uint32_t off = sw128_offset(i, ch, kBlk);
                        *reinterpret_cast<uint32_t *>(sQ + off) =
                            bf16x2_bits(qf.x * ex2f(g0), qf.y * ex2f(g1));
                        uint32_t hi, lo;
                        split_pair(kf.x * ex2f(-g0), kf.y * ex2f(-g1), hi, lo);
                        *reinterpret_cast<uint32_t *>(sK + off) = hi;
                        *reinterpret_cast<uint32_t *>(sKlo + off) = lo;
                    }
                }
                if (pt == 0) {
                    if (DBG && p.dbg_blk != nullptr && dv_tile == 0) p.dbg_blk[seq_of<PACKED>(p, bh).a + c] = kChunk;
                    sItem[n & 1] = ItemInfo{t0, 0, kChunk,
                                            kItemLast | (store ? kItemStore : 0) | piece_end, lc,
                                            -1, bh, 0};
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kBarQkFull]);
                ++n;
                continue;
            }
            // ---- sub-chunk rescaling (chunks whose decay exceeds the bound)
            float gtot0 = 0.f, gtot1 = 0.f;
            ok = sub_chunk_items<DK, PACKED, SCALAR, false, DBG>(p, dv_tile == 0 ? -1 : -2, bh, t0, lc, store, piece_end, pt, sQ, sK, sKlo, sG, sItem,
                                     bars, n, gtot0, gtot1, [] {});
            if (last_part) {
                gseg0 += gtot0;
                gseg1 += gtot1;
            }
            // an expired wait (!ok) ends the stream at the top of the loop
          }
          // segment summary: total decay of this segment (FULL pass, split sequence)
          if (p.mode == kModeFull && nseg_of<PACKED>(p, bh) > 1 && dv_tile == 0 && last_part) {
              float *dst = p.ws_decay + (static_cast<size_t>(pc.seg) * BHn + bh) * DK;
              dst[ch] = gseg0;
              dst[ch + 1] = gseg1;
          }
        }
        // ---- end of the requests and of the item stream
        if (pt == 0) {
            sReq[0] = ChunkReq{0, n, 1, 0};
            mbar_arrive(&bars[kBarReq]);
        }
        if (n > 0 && !mbar_wait_bounded(&bars[kBarQkEmpty], (n - 1) & 1, p.status, wait_limit<DBG>(p))) ok = false;
        if (pt == 0) sItem[n & 1] = ItemInfo{0, 0, 0, kItemEnd, 0, -1, 0, 0};
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarQkFull]);
    } else if (warp == kTmaWarp) {
        // =========================================================== TMA producer
        // Three load streams, each served as soon as its own condition holds,
        // so that none waits behind another: per requested chunk, A (and, in a
        // CTA pair, the raw Q/K staging tiles) at once; single-CTA Q and K once
        // the previous chunk's items have released the operand tiles; V once
        // its slot (also the output staging tile with two slots) is free.
        if (lane == 0) {
            int n_req = 0, n_qk = 0, n_v = 0;   // chunks requested / Q,K issued / V issued
            int withheld = -1;                  // the V tile a test withholds, if any
            int n_use = 0;                      // chunks used (known at the end request)
            bool req_end = false;
            // per requested chunk: tensor row and tensor head of its first token
            int t0s[4], firsts[4], bhs[4];      // at most 3 chunks are ever outstanding
            unsigned long long idle_since = 0;
            while (true) {
                bool progress = false;
                if (!req_end && mbar_test_wait(&bars[kBarReq], n_req & 1)) {
                    const ChunkReq rq = sReq[0];
                    progress = true;
                    if (rq.end) {
                        // a CTA pair requests one chunk ahead and says at the end
                        // how many chunks were used: no V load for the others
                        req_end = true;
                        n_use = PAIR ? rq.t0 : n_req;
                    } else {
                        const Seq sq = seq_of<PACKED>(p, rq.bh);
                        const int t0 = sq.y0 + rq.t0, bh = sq.z;
                        t0s[n_req & 3] = t0;
                        firsts[n_req & 3] = rq.first_item;
                        bhs[n_req & 3] = bh;
                        // A (and staging): the prep released them with the request
                        fence_proxy_async_smem();
                        if constexpr (SCALAR) {
                            // one gate per token: the prep threads read the
                            // chunk's 512 bytes themselves; pull them into L2
                            // (16-byte blocks inside the gate array only)
                            const uintptr_t a0 = reinterpret_cast<uintptr_t>(
                                p.g + static_cast<size_t>(bh) * p.T + t0);
                            const uintptr_t end = reinterpret_cast<uintptr_t>(
                                p.g + static_cast<size_t>(p.BH) * p.T);
                            const uintptr_t lo = (a0 + 15) & ~static_cast<uintptr_t>(15);
                            const uintptr_t hi = min(a0 + kChunk * 4, end) & ~static_cast<uintptr_t>(15);
                            if (hi > lo)
                                prefetch_l2_bulk(reinterpret_cast<const void *>(lo),
                                                 static_cast<uint32_t>(hi - lo));
                            mbar_arrive(&bars[kBarAFull]);
                        } else {
                            mbar_arrive_expect_tx(&bars[kBarAFull], L::kABytes);
                            tma_load_3d(sA, &p.tm_a, &bars[kBarAFull],
                                        static_cast<int>(rank) * L::kDKA, t0, bh);
                        }
                        if constexpr (PAIR) {
                            uint8_t *sRaw = smem + L::kRaw;
                            mbar_arrive_expect_tx(&bars[kBarQkRaw], 2u * kBlk);
                            tma_load_3d(sRaw, &p.tm_q, &bars[kBarQkRaw], static_cast<int>(rank) * 64,
                                        t0, bh);
                            tma_load_3d(sRaw + kBlk, &p.tm_k, &bars[kBarQkRaw],
                                        static_cast<int>(rank) * 64, t0, bh);
                        }
                        ++n_req;
                    }
                }
                if constexpr (!PAIR) {
                    // Q, K in place: after the last item of the previous chunk
                    if (n_qk < n_req) {
                        const int first = firsts[n_qk & 3];
                        if (first == 0 || mbar_test_wait(&bars[kBarQkEmpty], (first - 1) & 1)) {
                            const int t0 = t0s[n_qk & 3], bh = bhs[n_qk & 3];
                            mbar_arrive_expect_tx(&bars[kBarQkRaw], 2u * L::kQBytes);
#pragma unroll
                            for (int kb = 0; kb < DK / 64; ++kb) {
                                tma_load_3d(sQ + kb * kBlk, &p.tm_q, &bars[kBarQkRaw], kb * 64, t0, bh);
                                tma_load_3d(sK + kb * kBlk, &p.tm_k, &bars[kBarQkRaw], kb * 64, t0, bh);
                            }
                            ++n_qk;
                            progress = true;
                        }
                    }
                }
                // V of chunk n_v into slot n_v % VS: once the chunk that last
                // used the slot is done with it (products and output store)
                if (n_v < (req_end ? n_use : n_req) &&
                    (n_v < VS ||
                     mbar_test_wait(&bars[kBarVEmpty0 + n_v % VS], (n_v / VS - 1) & 1))) {
                    const int t0 = t0s[n_v & 3], bh = bhs[n_v & 3];
                    const int slot = n_v % VS;
                    uint8_t *dst = sV + slot * L::kVBytes;
                    if (DBG && p.mode == kModeFull && n_v + 1 == p.withhold_v) {
                        // test instrumentation: this tile is never loaded (and
                        // its barrier never armed), so its waiters time out
                        withheld = n_v;
                    } else {
                        mbar_arrive_expect_tx(&bars[kBarVFull0 + slot], L::kVBytes);
#pragma unroll
                        for (int nb = 0; nb < DVT / 64; ++nb)
                            tma_load_3d(dst + nb * kBlk, &p.tm_v, &bars[kBarVFull0 + slot],
                                        dv0 + nb * 64, t0, bh);
                    }
                    ++n_v;
                    progress = true;
                }
                if (req_end && n_v >= n_use && (PAIR || n_qk == n_req)) break;
                if (progress) {
                    idle_since = 0;
                } else {
                    const unsigned long long now = global_timer_ns();
                    if (idle_since == 0) {
                        idle_since = now;
                    } else if (now - idle_since > wait_limit<DBG>(p)) {
                        atomicOr(p.status, kStatusTimeout);
                        break;
                    }
                    __nanosleep(64);
                }
            }
            // loads issued for chunks that were never used must land before exit
            // (the last phase of each barrier; no later phase follows)
            if (n_req > 0) {
                mbar_wait_bounded(&bars[kBarAFull], (n_req - 1) & 1, p.status, wait_limit<DBG>(p));
                if (PAIR) mbar_wait_bounded(&bars[kBarQkRaw], (n_req - 1) & 1, p.status, wait_limit<DBG>(p));
            }
            for (int j = n_v - VS < 0 ? 0 : n_v - VS; j < n_v; ++j)
                if (j != withheld)
                    mbar_wait_bounded(&bars[kBarVFull0 + j % VS], (j / VS) & 1, p.status, wait_limit<DBG>(p));
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // =========================================================== MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_bf16(128, 128, false, false);   // P = Qh Kh^T
            constexpr uint32_t id_ov = idesc_bf16(128, DVT, false, true);    // O = Qh S, O += P V
            constexpr uint32_t id_kv = idesc_bf16(128, DVT, true, true);     // S += Kh^T V
            const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aKlo = smem_u32(sKlo);
            const uint32_t aV0 = smem_u32(sV), aS = smem_u32(sS);
            for (int n = 0;; ++n) {
                if (!mbar_wait_bounded(&bars[kBarQkFull], n & 1, p.status, wait_limit<DBG>(p))) break;
                const ItemInfo it = sItem[n & 1];
                mbar_arrive(&bars[kBarItem0 + (n & 1)]);
                if (it.flags & kItemEnd) break;
                const int ob = n & 1;
                const uint32_t tO = tmem + (ob ? TM::kO1 : TM::kO0);
                const uint32_t aV = aV0 + (it.lc % VS) * L::kVBytes;   // this chunk's V slot
                tc_fence_after();
                // P = Qh (Kh_hi + Kh_lo)^T, k-steps of 16 key channels.  In a CTA
                // pair the steps over this CTA's own 64-channel block go first,
                // while the peer's block may still be arriving.
                auto p_steps = [&](int kb, bool first) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t koff = kb * kBlk + kk * 32;
                        mma_bf16_ss(tmem + TM::kP, sw128_desc(aQ + koff, 16, 1024),
                                    sw128_desc(aK + koff, 16, 1024), id_qk, (first && kk == 0) ? 0 : 1);
                        mma_bf16_ss(tmem + TM::kP, sw128_desc(aQ + koff, 16, 1024),
                                    sw128_desc(aKlo + koff, 16, 1024), id_qk, 1);
                    }
                };
                // a CTA pair's item: the peer's half of the operand tiles first
                if (PAIR && it.xi >= 0) {
                    if (!mbar_wait_bounded(&bars[kBarXchg0 + (it.xi & 1)], (it.xi >> 1) & 1, p.status, wait_limit<DBG>(p)))
                        break;
                    tc_fence_after();
                }
#pragma unroll
                for (int kb = 0; kb < DK / 64; ++kb) p_steps(kb, kb == 0);
                mma_commit(&bars[kBarPFull]);
                // O = Qh S_prev: needs this O buffer drained and the previous
                // state scaled and copied
                bool okw = true;
                if (n >= 2) okw &= mbar_wait_bounded(&bars[kBarOFree0 + ob], ((n >> 1) + 1) & 1, p.status, wait_limit<DBG>(p));
                okw &= mbar_wait_bounded(&bars[kBarSReady], n & 1, p.status, wait_limit<DBG>(p));
                if (!okw) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks) {
                    const uint32_t koff = (ks >> 2) * kBlk + (ks & 3) * 32;
                    mma_bf16_ss(tO, sw128_desc(aQ + koff, 16, 1024),
                                sw128_desc(aS + ks * 2048, L::kSBlk, 1024), id_ov, ks > 0);
                }
                // S += (Kh_hi + Kh_lo)^T V
                if (!mbar_wait_bounded(&bars[kBarVFull0 + it.lc % VS], (it.lc / VS) & 1, p.status, wait_limit<DBG>(p)))
                    break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < kChunk / 16; ++ks) {
                    mma_bf16_ss(tmem + TM::kS, sw128_desc(aK + ks * 2048, kBlk, 1024),
                                sw128_desc(aV + ks * 2048, kBlk, 1024), id_kv, 1);
                    mma_bf16_ss(tmem + TM::kS, sw128_desc(aKlo + ks * 2048, kBlk, 1024),
                                sw128_desc(aV + ks * 2048, kBlk, 1024), id_kv, 1);
                }
                mma_commit(&bars[kBarSDone]);
                if constexpr (PAIR)
                    mma_commit_multicast(&bars[kBarQkEmpty], 0x3);   // both CTAs' tiles
                else
                    mma_commit(&bars[kBarQkEmpty]);
                // O += (P_hi + P_lo) V, P from TMEM
                if (!mbar_wait_bounded(&bars[kBarPSplit], n & 1, p.status, wait_limit<DBG>(p))) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < kChunk / 16; ++ks) {
                    const uint32_t pcol = TM::kP + 16 * ks;   // hi pairs, then lo pairs
                    mma_bf16_ts(tO, tmem + pcol, sw128_desc(aV + ks * 2048, kBlk, 1024), id_ov, 1);
                    mma_bf16_ts(tO, tmem + pcol + 8, sw128_desc(aV + ks * 2048, kBlk, 1024), id_ov,
                                1);
                }
                mma_commit(&bars[kBarOFull0 + ob]);
            }
            // every product issued here is complete before TMEM is freed (a
            // stream that ended on an expired wait may leave some in flight)
            mma_commit(&bars[kBarDrain]);
            mbar_wait_bounded(&bars[kBarDrain], 0, p.status, wait_limit<DBG>(p));
        }
        __syncwarp();
    } else {
        // =========================================================== TMEM warps
        const int i = tid - 32 * kTmemWarp0;      // TMEM lane = row = key channel
        const uint32_t lane_base = static_cast<uint32_t>((warp - kTmemWarp0) * 32) << 16;
        const bool has_state_row = ((warp - kTmemWarp0) * 32) < DK;  // warp-uniform
        const uint32_t tP = tmem + lane_base + TM::kP;
        const uint32_t tS = tmem + lane_base + TM::kS;

        // ---- start state of a piece into TMEM (fp32) and its bf16 copy, then
        // "state ready" for the piece's first item.  FULL pass: h0 for a
        // sequence's first segment, zero for later ones.  CORRECT pass: the
        // exact start state by the scan of the segment summaries before it; the
        // last segment's CTA also writes hT = diag(e^G) S_start + S*.
        auto load_state = [&](const Piece &pc) {
            const int bh = pc.u, seg = pc.seg;
            if (has_state_row) {
                float *hT_dst = nullptr;
                float eG = 0.f;
                const float *sstar = nullptr;
                if (p.mode == kModeCorrect && seg == nseg_of<PACKED>(p, bh) - 1 && p.hT) {
                    hT_dst = p.hT + (static_cast<size_t>(bh) * DK + i) * p.dv + dv0;
                    eG = __expf(p.ws_decay[(static_cast<size_t>(seg) * BHn + bh) * DK + i]);
                    sstar = p.ws_state + ((static_cast<size_t>(seg) * BHn + bh) * DK + i) * p.dv + dv0;
                }
#pragma unroll
                for (int c0 = 0; c0 < DVT; c0 += 32) {
                    float x[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] = 0.f;
                    if (p.mode == kModeFull) {
                        if (seg == 0 && p.h0) {
                            const float *src =
                                p.h0 + (static_cast<size_t>(bh) * DK + i) * p.dv + dv0 + c0;
#pragma unroll
                            for (int j = 0; j < 32; j += 4) {
                                const float4 v4 = *reinterpret_cast<const float4 *>(src + j);
                                x[j] = v4.x;
                                x[j + 1] = v4.y;
                                x[j + 2] = v4.z;
                                x[j + 3] = v4.w;
                            }
                        }
                    } else {
                        for (int s2 = 0; s2 < seg; ++s2) {
                            const float e =
                                __expf(p.ws_decay[(static_cast<size_t>(s2) * BHn + bh) * DK + i]);
                            const float *src = p.ws_state +
                                               ((static_cast<size_t>(s2) * BHn + bh) * DK + i) * p.dv +
                                               dv0 + c0;
#pragma unroll
                            for (int j = 0; j < 32; j += 4) {
                                const float4 v4 = *reinterpret_cast<const float4 *>(src + j);
                                x[j] = fmaf(e, x[j], v4.x);
                                x[j + 1] = fmaf(e, x[j + 1], v4.y);
                                x[j + 2] = fmaf(e, x[j + 2], v4.z);
                                x[j + 3] = fmaf(e, x[j + 3], v4.w);
                            }
                        }
                        if (hT_dst) {
#pragma unroll
                            for (int j = 0; j < 32; j += 4) {
                                const float4 v4 = *reinterpret_cast<const float4 *>(sstar + c0 + j);
                                *reinterpret_cast<float4 *>(hT_dst + c0 + j) =
                                    make_float4(fmaf(eG, x[j], v4.x), fmaf(eG, x[j + 1], v4.y),
                                                fmaf(eG, x[j + 2], v4.z), fmaf(eG, x[j + 3], v4.w));
                            }
                        }
                    }
                    uint32_t r[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(x[j]);
                    tmem_st32(tS + c0, r);
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        uint4 pk;
                        pk.x = pack_bf16x2(x[j], x[j + 1]);
                        pk.y = pack_bf16x2(x[j + 2], x[j + 3]);
                        pk.z = pack_bf16x2(x[j + 4], x[j + 5]);
                        pk.w = pack_bf16x2(x[j + 6], x[j + 7]);
                        *reinterpret_cast<uint4 *>(sS + sw128_offset(i, c0 + j, L::kSBlk)) = pk;
                    }
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kBarSReady]);
        };
        // ---- end state of a FULL-pass piece: hT for an unsplit sequence,
        // else the segment summary S* of the workspace
        auto store_state = [&](const Piece &pc) {
            if (!has_state_row) return;
            float *dst = nullptr;
            if (nseg_of<PACKED>(p, pc.u) == 1) {
                if (p.hT) dst = p.hT + (static_cast<size_t>(pc.u) * DK + i) * p.dv + dv0;
            } else {
                dst = p.ws_state + ((static_cast<size_t>(pc.seg) * BHn + pc.u) * DK + i) * p.dv + dv0;
            }
            if (!dst) return;
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < DVT; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tS + c0, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(dst + c0 + j) =
                        make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                    __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
            }
        };
        load_state(piece_at<PACKED>(p, g_begin, g_end));   // phase 0 of "state ready"

        for (int n = 0;; ++n) {
            // (one barrier per item parity, so that the MMA issuer may run up
            // to two items ahead of these warps)
            if (!__all_sync(0xffffffffu,
                            mbar_wait_bounded(&bars[kBarItem0 + (n & 1)], (n >> 1) & 1, p.status, wait_limit<DBG>(p))))
                break;
            const ItemInfo it = sItem[n & 1];
            if (it.flags & kItemEnd) break;
            const int ob = n & 1;
            // ---- causal mask of P (row i), split into the TMEM A operand of P V
            {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bars[kBarPFull], n & 1, p.status, wait_limit<DBG>(p))))
                    break;
                tc_fence_after();
                // This warp's rows are 32 wq .. 32 wq + 31: column blocks past
                // block wq are zero (nothing to read), block wq is the diagonal,
                // the blocks before it are unmasked.
                const int wq = warp - kTmemWarp0;
#pragma unroll
                for (int qd = 0; qd < kChunk / 32; qd += 2) {
                    if (qd > wq) {
                        zero_p_block(tP + 32 * qd);
                        zero_p_block(tP + 32 * (qd + 1));
                    } else if (qd + 1 > wq) {
                        uint32_t r0[32];
                        tmem_ld32(tP + 32 * qd, r0);
                        tmem_wait_ld();
                        split_p_block(tP + 32 * qd, r0, 32 * qd, i, true);
                        zero_p_block(tP + 32 * (qd + 1));
                    } else {
                        uint32_t r0[32], r1[32];
                        tmem_ld32(tP + 32 * qd, r0);
                        tmem_ld32(tP + 32 * (qd + 1), r1);
                        tmem_wait_ld();
                        split_p_block(tP + 32 * qd, r0, 32 * qd, i, false);
                        split_p_block(tP + 32 * (qd + 1), r1, 32 * (qd + 1), i, qd + 1 == wq);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kBarPSplit]);
            }
            // The state step (S <- diag(e^decay) S and its bf16 copy for the next
            // item's Qh S) and the output step (this item's rows).  With two V
            // slots the output is staged in the chunk's V slot once P V is done,
            // after the state step, which therefore waits for nothing but the
            // chunk's S products.  With one slot (dk = 128 only) the bf16 state
            // copy, which has the output tile's size and layout, is the staging
            // tile: this item's Qh S product has finished reading it once the
            // output is ready, so the output step runs first, V is free as soon
            // as P V is done, and the state step follows the staging store.
            static_assert(VS == 2 || DK == 128, "one V slot only where the state copy can stage");
            constexpr bool kStageInS = VS == 1;
            uint8_t *sStage = kStageInS ? sS : sV + (it.lc % VS) * L::kVBytes;
            const bool store_item = (it.flags & kItemStore) != 0;
            const Seq sq = seq_of<PACKED>(p, it.bh);
            // A whole chunk leaves through the staging tile, unless it is the
            // tail of a packed sequence: its tile rows past the end belong to
            // the next sequence, so its rows are stored one by one.
            const bool staged = store_item && it.r0 == 0 && it.r1 == kChunk &&
                                (!PACKED || it.t0 + kChunk <= sq.len);
            const bool piece_end = (it.flags & kItemPieceEnd) != 0;
            const bool keep = (it.flags & kItemKeep) != 0;
            auto state_step = [&]() -> bool {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bars[kBarSDone], n & 1, p.status, wait_limit<DBG>(p))))
                    return false;
                // a CTA pair's item: the peer's half of the state factors
                if (it.xi >= 0 &&
                    !__all_sync(0xffffffffu, mbar_wait_bounded(&bars[kBarXchg0 + (it.xi & 1)],
                                                               (it.xi >> 1) & 1, p.status, wait_limit<DBG>(p))))
                    return false;
                tc_fence_after();
                if (has_state_row) {
                    const float f = sG[(n & 1) * DK + i];
#pragma unroll
                    for (int c0 = 0; c0 < DVT; c0 += 32) {
                        uint32_t r[32];
                        tmem_ld32(tS + c0, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * f);
                        tmem_st32(tS + c0, r);
                        if (piece_end && !keep) continue;   // the next piece starts afresh
#pragma unroll
                        for (int j = 0; j < 32; j += 8) {
                            uint4 pk;
                            pk.x = pack_bf16x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
                            pk.y = pack_bf16x2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                            pk.z = pack_bf16x2(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5]));
                            pk.w = pack_bf16x2(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7]));
                            *reinterpret_cast<uint4 *>(sS + sw128_offset(i, c0 + j, L::kSBlk)) = pk;
                        }
                    }
                    tmem_wait_st();
                }
                if (piece_end) {
                    // this piece's end state, then the next piece's start state
                    // (both found from the item: the piece ends with its chunk)
                    const long long a = sq.a;
                    const int cl = it.t0 / kChunk;
                    Piece done;
                    done.u = it.bh;
                    done.seg = static_cast<int>((a + cl) / p.L - a / p.L);
                    store_state(done);
                    if (!keep) {
                        const long long gn = a + cl + 1, ge = full_range_end(p);
                        if (gn < ge) load_state(piece_at<PACKED>(p, gn, ge));
                        return true;
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kBarSReady]);
                return true;
            };
            auto output_step = [&]() -> bool {
                if (!__all_sync(0xffffffffu,
                                mbar_wait_bounded(&bars[kBarOFull0 + ob], (n >> 1) & 1, p.status, wait_limit<DBG>(p))))
                    return false;
                tc_fence_after();
                // staged in the state copy: the V tile is free now
                if (kStageInS && (it.flags & kItemLast) && lane == 0)
                    mbar_arrive(&bars[kBarVEmpty0 + it.lc % VS]);
                {
                    // a CTA pair folds the read-out scale into Qh
                    const float osc = PAIR ? 1.f : p.scale;
                    const uint32_t tO = tmem + lane_base + (ob ? TM::kO1 : TM::kO0);
                    const int t = it.t0 + i;
                    const bool st = store_item && !staged && i >= it.r0 && i < it.r1 && t < sq.len;
                    __nv_bfloat16 *orow =
                        p.o + (static_cast<size_t>(sq.z) * T + sq.y0 + t) * p.dv + dv0;
#pragma unroll
                    for (int c0 = 0; c0 < DVT; c0 += 64) {
                        uint32_t ra[32], rb[32];
                        tmem_ld32(tO + c0, ra);
                        tmem_ld32(tO + c0 + 32, rb);
                        tmem_wait_ld();
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const uint32_t(&r)[32] = half ? rb : ra;
                            const int cc = c0 + 32 * half;
#pragma unroll
                            for (int j = 0; j < 32; j += 8) {
                                uint4 pk;
                                pk.x = pack_bf16x2(osc * __uint_as_float(r[j]), osc * __uint_as_float(r[j + 1]));
                                pk.y = pack_bf16x2(osc * __uint_as_float(r[j + 2]), osc * __uint_as_float(r[j + 3]));
                                pk.z = pack_bf16x2(osc * __uint_as_float(r[j + 4]), osc * __uint_as_float(r[j + 5]));
                                pk.w = pack_bf16x2(osc * __uint_as_float(r[j + 6]), osc * __uint_as_float(r[j + 7]));
                                if (staged)
                                    *reinterpret_cast<uint4 *>(sStage + sw128_offset(i, cc + j, kBlk)) = pk;
                                else if (st)
                                    *reinterpret_cast<uint4 *>(orow + cc + j) = pk;
                            }
                        }
                    }
                }
                tc_fence_before();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars[kBarOFree0 + ob]);
                    // This warp's 32 rows of a staged tile leave with one TMA store
                    // per 64-column block, and the staging rows are reused only
                    // once the store has read them.
                    const int r0w = it.t0 + 32 * (warp - kTmemWarp0);
                    if (staged && r0w < sq.len) {
#pragma unroll
                        for (int nb = 0; nb < DVT / 64; ++nb)
                            tma_store_3d(&p.tm_o32, sStage + nb * kBlk + (warp - kTmemWarp0) * 32 * 128,
                                         dv0 + nb * 64, sq.y0 + r0w, sq.z);
                        tma_store_commit();
                        tma_store_wait_read_all();
                    }
                    // staged in the V tile: four arrivals free it after the stores
                    if (!kStageInS && (it.flags & kItemLast))
                        mbar_arrive(&bars[kBarVEmpty0 + it.lc % VS]);
                }
                __syncwarp();
                return true;
            };
            if constexpr (kStageInS) {
                if (!output_step() || !state_step()) break;
            } else {
                if (!state_step() || !output_step()) break;
            }
        }
        if (lane == 0) tma_store_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, TM::kCols);
    }
    // the peer may still copy into, or arrive on, this CTA's shared memory
    if constexpr (PAIR) cluster_sync_all();
}

// Final states of a two-segment plan whose correction ran inside the FULL pass:
// hT = diag(e^G_1) S*_0 + S*_1 per (sequence, key row), where S*_0 is the
// exact state at the end of the first segment, and S*_1 and G_1 are the second
// segment's end state from a zero start and its total log-decay.  One thread
// per four value columns.
__global__ void __launch_bounds__(256) two_segment_states_kernel(const float *__restrict__ ws_state,
                                                                 const float *__restrict__ ws_decay,
                                                                 float *__restrict__ hT, long long BH,
                                                                 int dk, int dv) {
    const long long quads = BH * dk * (dv / 4);
    for (long long q = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; q < quads;
         q += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = q / (dv / 4);           // (sequence, key row)
        const float e = __expf(ws_decay[BH * dk + row]);
        const float4 s0 = reinterpret_cast<const float4 *>(ws_state)[q];
        const float4 s1 = reinterpret_cast<const float4 *>(ws_state + BH * dk * dv)[q];
        reinterpret_cast<float4 *>(hT)[q] =
            make_float4(fmaf(e, s0.x, s1.x), fmaf(e, s0.y, s1.y), fmaf(e, s0.z, s1.z),
                        fmaf(e, s0.w, s1.w));
    }
}

template <int DK, int DVT, bool PAIR, bool PACKED, bool SCALAR, bool DBG = false>
int launch_tiles(const ChunkLaunch &c, cudaStream_t stream) {
    using L = Smem<DK, DVT, PAIR>;
    auto kern = chunk_fwd_kernel<DK, DVT, PAIR, PACKED, SCALAR, DBG>;
    static bool attr_set = false;  // per instantiation, per process
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(L::kAlloc));
        if (e != cudaSuccess) return static_cast<int>(e);
        attr_set = true;
    }
    KParams p;
    p.tm_q = c.tm_q;
    p.tm_k = c.tm_k;
    p.tm_a = c.tm_a;
    p.tm_v = c.tm_v;
    p.tm_o32 = c.tm_o32;
    p.q = static_cast<const uint32_t *>(c.q);
    p.k = static_cast<const uint32_t *>(c.k);
    p.a = SCALAR ? nullptr : reinterpret_cast<const float2 *>(c.log_alpha);
    p.g = SCALAR ? c.log_alpha : nullptr;
    p.h0 = c.h0;
    p.hT = c.hT;
    p.o = static_cast<__nv_bfloat16 *>(c.o);
    p.ws_state = c.ws_state;
    p.ws_decay = c.ws_decay;
    p.scale = c.scale;
    p.BH = c.B * c.H;
    p.T = c.T;
    p.dv = c.dv;
    p.NC = c.NC;
    p.L = c.L;
    p.total = c.total;
    p.seqs = c.seqs;
    p.NS = c.NS;
    p.H = c.H;
    p.seg_max = c.seg_max;
    p.force_sub = c.force_exact;
    p.status = c.status;
    p.fuse = c.fuse;
    p.wait_ns = c.wait_ns ? c.wait_ns : kWaitLimitNs;
    p.dbg_gamma = c.dbg_gamma;
    p.dbg_blk = c.dbg_blk;
    p.withhold_v = c.withhold_v;
    const int n_dvt = c.dv / DVT;
    // `count` CTAs (clusters) per tile column; the index is blockIdx.y +
    // blockIdx.z * gridDim.y, so that any count fits the grid's limits
    auto launch = [&](int mode, long long count) -> cudaError_t {
        p.mode = mode;
        p.n_units = count;
        const unsigned gy = static_cast<unsigned>(count < 32768 ? count : 32768);
        const unsigned gz = static_cast<unsigned>((count + gy - 1) / gy);
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3(n_dvt, gy, gz);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = L::kAlloc;
        cfg.stream = stream;
        if (PAIR) {
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;   // the two value-column tiles of one head
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
        }
        return cudaLaunchKernelEx(&cfg, kern, p);
    };
    // FULL pass: one CTA (cluster) per range; CORRECT pass: one per (sequence,
    // segment >= 1), those past a sequence's segment count leave at once
    cudaError_t e = launch(kModeFull, c.W);
    if (e != cudaSuccess || c.seg_max == 1) return static_cast<int>(e);
    if (c.fuse) {
        // the windows were corrected in the FULL pass; only hT remains
        if (!c.hT) return 0;
        const long long quads = static_cast<long long>(c.B) * c.H * DK * (c.dv / 4);
        const int blocks = static_cast<int>(std::min<long long>((quads + 255) / 256, 4096));
        two_segment_states_kernel<<<blocks, 256, 0, stream>>>(c.ws_state, c.ws_decay, c.hT,
                                                               static_cast<long long>(c.B) * c.H,
                                                               DK, c.dv);
        return static_cast<int>(cudaGetLastError());
    }
    return static_cast<int>(
        launch(kModeCorrect, static_cast<long long>(c.B) * c.H * (c.seg_max - 1)));
}

template <int DK, int DVT, bool PAIR>
int max_resident() {
    using L = Smem<DK, DVT, PAIR>;
    auto kern = chunk_fwd_kernel<DK, DVT, PAIR, false, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(L::kAlloc)) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (!PAIR) return sms;   // one CTA per SM (the CTA takes all of TMEM)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::kAlloc;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return clusters;
}

}  // namespace
}  // namespace gla
