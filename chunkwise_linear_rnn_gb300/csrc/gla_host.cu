// gla_host.cu — gla_chunk_fwd_host: the chunked forward on host buffers, with
// the host<->device copies pipelined against the computation.
//
// The (batch, head) rows are independent sequences ([B, H, ...] layouts are
// row-major, so a run of consecutive rows is one contiguous slice of every
// tensor).  They are processed in up to kMaxGroups groups; each group goes
// host->device on one internal stream, through gla_chunk_fwd's launch path on
// the caller's stream, and device->host on a second internal stream.  Two
// device slots for inputs and two for outputs let group g's copy in, group
// g-1's computation and group g-2's copy out run at the same time.  Events
// order everything against the caller's stream: the call is stream-ordered on
// `stream`, like the device entry points.
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "gla.h"
#include "gla_internal.h"

namespace gla {
namespace {

constexpr int kMaxGroups = 8;
constexpr int kSlots = 2;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Scratch the chunked forward needs for `rows` rows (same plan as gla_chunk_fwd).
int scratch_for(int rows, int T, int dk, int dv, size_t *bytes) {
    int nseg = 0, tile = 0, launches = 0;
    unsigned long sb = 0;
    const int st = gla_chunk_fwd_plan(1, rows, T, dk, dv, nullptr, &nseg, &tile, &launches, &sb);
    *bytes = sb;
    return st;
}

struct Slot {
    char *q, *k, *v, *a, *h0, *o, *hT, *scratch;
};

}  // namespace
}  // namespace gla

extern "C" int gla_chunk_fwd_host(const void *q, const void *k, const void *v,
                                  const float *log_alpha, float scale, const float *h0, void *o,
                                  float *hT, int B, int H, int T, int dk, int dv,
                                  cudaStream_t stream) {
    using namespace gla;
    if (!q || !k || !v || !log_alpha || !o) return GLA_ERR_ARG;
    if (B <= 0 || H <= 0 || T <= 0) return GLA_ERR_ARG;
    if (static_cast<long long>(B) * H > 0x7fffffffLL) return GLA_ERR_ARG;
    if (!(dk == 64 || dk == 128) || !(dv == 64 || dv == 128 || dv == 256)) return GLA_ERR_SHAPE;

    const int BH = B * H;
    const int rows = (BH + kMaxGroups - 1) / kMaxGroups;   // rows per group
    const int n_groups = (BH + rows - 1) / rows;           // the last group may be short
    const int last_rows = BH - (n_groups - 1) * rows;
    const size_t tok = static_cast<size_t>(T);
    const size_t b_qk = tok * dk * 2, b_a = tok * dk * 4, b_v = tok * dv * 2;   // per row
    const size_t b_st = static_cast<size_t>(dk) * dv * 4;
    // segment scratch: a short group may split its sequences further
    size_t b_scr = 0, b_scr_last = 0;
    int st = scratch_for(rows, T, dk, dv, &b_scr);
    if (st == GLA_OK) st = scratch_for(last_rows, T, dk, dv, &b_scr_last);
    if (st != GLA_OK) return st;   // no device, or sizes the plan rejects
    b_scr = std::max(b_scr, b_scr_last);

    // slot layout: inputs and outputs of one group, plus its segment scratch
    const size_t r = static_cast<size_t>(rows);
    const size_t o_q = 0, o_k = o_q + align256(r * b_qk), o_v = o_k + align256(r * b_qk);
    const size_t o_a = o_v + align256(r * b_v), o_h0 = o_a + align256(r * b_a);
    const size_t o_o = o_h0 + (h0 ? align256(r * b_st) : 0), o_hT = o_o + align256(r * b_v);
    const size_t o_scr = o_hT + (hT ? align256(r * b_st) : 0);
    const size_t slot_bytes = o_scr + align256(b_scr);

    void *mem = nullptr;
    if (cudaMallocAsync(&mem, kSlots * slot_bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return GLA_ERR_ALLOC;
    }
    Slot slot[kSlots];
    for (int s = 0; s < kSlots; ++s) {
        char *base = static_cast<char *>(mem) + s * slot_bytes;
        slot[s] = Slot{base + o_q, base + o_k, base + o_v, base + o_a,
                       h0 ? base + o_h0 : nullptr, base + o_o, hT ? base + o_hT : nullptr,
                       base + o_scr};
    }

    cudaStream_t s_in = nullptr, s_out = nullptr;
    std::vector<cudaEvent_t> ev;   // start, then in/comp/out per group
    int result = GLA_OK;
    auto fail = [&](int code) {
        cudaGetLastError();
        if (result == GLA_OK) result = code;
    };
    if (cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking) != cudaSuccess) {
        fail(GLA_ERR_LAUNCH);
    }
    ev.resize(1 + 3 * n_groups, nullptr);
    for (auto &e : ev)
        if (result == GLA_OK && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
            fail(GLA_ERR_LAUNCH);
    cudaEvent_t ev_start = ev[0];
    auto ev_in = [&](int g) { return ev[1 + 3 * g]; };
    auto ev_comp = [&](int g) { return ev[2 + 3 * g]; };
    auto ev_out = [&](int g) { return ev[3 + 3 * g]; };

    const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k);
    const char *hv = static_cast<const char *>(v);
    const char *ha = reinterpret_cast<const char *>(log_alpha);
    const char *hh0 = reinterpret_cast<const char *>(h0);
    char *ho = static_cast<char *>(o), *hhT = reinterpret_cast<char *>(hT);
    auto cp = [&](void *dst, const void *src, size_t n, cudaMemcpyKind kind, cudaStream_t s) {
        if (result == GLA_OK && cudaMemcpyAsync(dst, src, n, kind, s) != cudaSuccess)
            fail(GLA_ERR_LAUNCH);
    };
    auto wait = [&](cudaStream_t s, cudaEvent_t e) {
        if (result == GLA_OK && cudaStreamWaitEvent(s, e, 0) != cudaSuccess) fail(GLA_ERR_LAUNCH);
    };
    auto rec = [&](cudaEvent_t e, cudaStream_t s) {
        if (result == GLA_OK && cudaEventRecord(e, s) != cudaSuccess) fail(GLA_ERR_LAUNCH);
    };

    // the slots exist for the internal streams once `stream` reaches this point
    rec(ev_start, stream);
    wait(s_in, ev_start);
    wait(s_out, ev_start);
    for (int g = 0; g < n_groups && result == GLA_OK; ++g) {
        const int r0 = g * rows, nr = std::min(rows, BH - r0);
        const size_t R0 = static_cast<size_t>(r0), NR = static_cast<size_t>(nr);
        const Slot &sl = slot[g % kSlots];
        // inputs of group g, once group g-2 has finished computing from this slot
        if (g >= kSlots) wait(s_in, ev_comp(g - kSlots));
        cp(sl.q, hq + R0 * b_qk, NR * b_qk, cudaMemcpyHostToDevice, s_in);
        cp(sl.k, hk + R0 * b_qk, NR * b_qk, cudaMemcpyHostToDevice, s_in);
        cp(sl.v, hv + R0 * b_v, NR * b_v, cudaMemcpyHostToDevice, s_in);
        cp(sl.a, ha + R0 * b_a, NR * b_a, cudaMemcpyHostToDevice, s_in);
        if (h0) cp(sl.h0, hh0 + R0 * b_st, NR * b_st, cudaMemcpyHostToDevice, s_in);
        rec(ev_in(g), s_in);
        // the computation, once the inputs are in and group g-2's outputs are out
        wait(stream, ev_in(g));
        if (g >= kSlots) wait(stream, ev_out(g - kSlots));
        if (result == GLA_OK) {
            const int rc = chunk_fwd_with_scratch(sl.q, sl.k, sl.v, reinterpret_cast<const float *>(sl.a),
                                                  scale, reinterpret_cast<const float *>(sl.h0), sl.o,
                                                  reinterpret_cast<float *>(sl.hT), 1, nr, T, dk, dv,
                                                  nullptr, stream, sl.scratch, b_scr);
            if (rc != GLA_OK) fail(rc);
        }
        rec(ev_comp(g), stream);
        // outputs of group g
        wait(s_out, ev_comp(g));
        cp(ho + R0 * b_v, sl.o, NR * b_v, cudaMemcpyDeviceToHost, s_out);
        if (hT) cp(hhT + R0 * b_st, sl.hT, NR * b_st, cudaMemcpyDeviceToHost, s_out);
        rec(ev_out(g), s_out);
    }
    // `stream` resumes once every output is on the host; then the slots go
    if (result == GLA_OK) {
        wait(stream, ev_out(n_groups - 1));
        wait(stream, ev_in(n_groups - 1));
    } else {
        // on failure nothing more is enqueued; wait for what was, so that the
        // slots are not freed under a copy still in flight
        if (s_in) cudaStreamSynchronize(s_in);
        if (s_out) cudaStreamSynchronize(s_out);
        cudaGetLastError();
    }
    cudaFreeAsync(mem, stream);
    for (auto &e : ev)
        if (e) cudaEventDestroy(e);
    if (s_in) cudaStreamDestroy(s_in);
    if (s_out) cudaStreamDestroy(s_out);
    return result;
}
