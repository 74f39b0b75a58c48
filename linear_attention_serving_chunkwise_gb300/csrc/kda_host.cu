// Host-buffer prefill: the inputs and outputs of kda_prefill live in host memory and the
// call pipelines host->device copies, the prefill kernel and device->host copies over
// chunk-aligned token rounds.  Declarations and contracts: include/kda.h.
//
// Round r covers tokens [r L, (r + 1) L) of every sequence (L = segment_tokens, a multiple
// of the 64-token chunk), so each round is an ordinary kda_prefill over a packed batch of
// sequence pieces that continues the device-resident state in place; the chunk partition,
// and with it every result bit, is that of a single kda_prefill call over the whole batch.
// Two device staging sets alternate: while round r runs on the caller's stream, round r+1's
// inputs arrive on the upload stream(s) and round r-1's outputs leave on a download stream,
// ordered by events.  (Splitting each upload over two streams measured no faster on GB300:
// one host-to-device copy already moves ~210 GB/s, the link's share for this direction.)
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "../../include/kda.h"

namespace kda {
// kda_prefill on the kernels that need no workspace (defined with the C ABI)
kda_status prefill_no_workspace(const kda_prefill_desc* desc, const void* q, const void* k, const void* v,
                                const float* g, const float* beta, const int32_t* cu_seqlens, const float* init_state,
                                float* out, float* final_state, void* stream);
}  // namespace kda

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;
constexpr int kUp = 1;   // upload streams (each piece is split evenly across them)

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Streams and events of one device, created on first use and kept for the process.
struct HostPipe {
    cudaStream_t up[kUp] = {}, down = nullptr;
    cudaEvent_t start = nullptr, end = nullptr, staged[2][kUp] = {}, computed[2] = {nullptr, nullptr},
                drained[2] = {nullptr, nullptr};
    std::mutex mu;   // one pipelined call at a time per device (the events are reused)
    bool ready = false;
};

HostPipe* pipe_for_current_device()
{
    static std::mutex mu;
    static HostPipe pipes[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    HostPipe& p = pipes[dev];
    if (!p.ready) {
        const unsigned ef = cudaEventDisableTiming;
        bool ok = cudaStreamCreateWithFlags(&p.down, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p.start, ef) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p.end, ef) == cudaSuccess;
        for (int u = 0; ok && u < kUp; ++u) ok = cudaStreamCreateWithFlags(&p.up[u], cudaStreamNonBlocking) == cudaSuccess;
        for (int b = 0; ok && b < 2; ++b) {
            ok = cudaEventCreateWithFlags(&p.computed[b], ef) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p.drained[b], ef) == cudaSuccess;
            for (int u = 0; ok && u < kUp; ++u) ok = cudaEventCreateWithFlags(&p.staged[b][u], ef) == cudaSuccess;
        }
        if (!ok) return nullptr;
        p.ready = true;
    }
    return &p;
}

struct Sizes {
    size_t esz, in_row_q, in_row_v, row_g, row_beta, row_out;   // bytes per token of each tensor
    size_t round_tokens;                                         // tokens of the largest round
    size_t state_bytes, cu_bytes;
};

bool sizes_of(const kda_prefill_desc& d, int32_t L, Sizes* s)
{
    if (L <= 0 || L % 64 != 0) return false;
    const size_t H = (size_t)d.num_heads;
    s->esz = d.qkv_dtype == KDA_BF16 ? 2 : 4;
    s->in_row_q = H * d.dk * s->esz;
    s->in_row_v = H * d.dv * s->esz;
    s->row_g = H * d.dk * sizeof(float);
    s->row_beta = H * sizeof(float);
    s->row_out = H * d.dv * sizeof(float);
    const size_t cap = (size_t)d.num_seqs * (size_t)L;
    s->round_tokens = cap < (size_t)d.total_tokens ? cap : (size_t)d.total_tokens;
    s->state_bytes = (size_t)d.num_seqs * H * d.dk * d.dv * sizeof(float);
    s->cu_bytes = ((size_t)d.num_seqs + 1) * sizeof(int32_t);
    return true;
}

// Device layout of one staging set: q, k, v, g, beta, out, cu (each 256-byte aligned).
struct Stage {
    char *q, *k, *v, *g, *beta, *out;
    int32_t* cu;
};

size_t stage_bytes(const Sizes& s)
{
    const size_t T = s.round_tokens;
    return align_up(T * s.in_row_q) * 2 + align_up(T * s.in_row_v) + align_up(T * s.row_g) +
           align_up(T * s.row_beta) + align_up(T * s.row_out) + align_up(s.cu_bytes);
}

Stage carve(char* base, const Sizes& s)
{
    const size_t T = s.round_tokens;
    Stage st;
    st.q = base; base += align_up(T * s.in_row_q);
    st.k = base; base += align_up(T * s.in_row_q);
    st.v = base; base += align_up(T * s.in_row_v);
    st.g = base; base += align_up(T * s.row_g);
    st.beta = base; base += align_up(T * s.row_beta);
    st.out = base; base += align_up(T * s.row_out);
    st.cu = reinterpret_cast<int32_t*>(base);
    return st;
}

bool host_overlap(const void* a, size_t na, const void* b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const char* pa = static_cast<const char*>(a);
    const char* pb = static_cast<const char*>(b);
    return pa < pb + nb && pb < pa + na;
}

}  // namespace

extern "C" {

size_t kda_prefill_host_workspace_bytes(const kda_prefill_desc* desc, int32_t segment_tokens)
{
    if (!desc || desc->num_seqs < 0 || desc->total_tokens < 0 || desc->num_heads < 1) return 0;
    if (desc->num_seqs == 0) return 0;
    Sizes s;
    if (!sizes_of(*desc, segment_tokens, &s)) return 0;
    return align_up(s.state_bytes) + 2 * stage_bytes(s);
}

kda_status kda_prefill_host(const kda_prefill_desc* desc, const void* q, const void* k, const void* v,
                            const float* g, const float* beta, const int32_t* cu_seqlens,
                            const float* init_state, float* out, float* final_state, int32_t segment_tokens,
                            void* workspace, size_t workspace_bytes, void* stream)
{
    // ---- host-side validation (no CUDA call before it passes)
    kda_prefill_plan plan;
    kda_status st = kda_prefill_query(desc, &plan);
    if (st != KDA_OK) return st;
    const kda_prefill_desc d = *desc;
    if (d.num_seqs == 0) return KDA_OK;
    Sizes s;
    if (!sizes_of(d, segment_tokens, &s)) return KDA_ERR_INVALID_ARG;
    const size_t N = (size_t)d.num_seqs, T = (size_t)d.total_tokens;
    std::vector<int64_t> bos(N + 1);
    if (cu_seqlens) {
        if (cu_seqlens[0] != 0 || (size_t)cu_seqlens[N] != T) return KDA_ERR_INVALID_ARG;
        for (size_t n = 0; n <= N; ++n) {
            if (n > 0 && cu_seqlens[n] < cu_seqlens[n - 1]) return KDA_ERR_INVALID_ARG;
            bos[n] = cu_seqlens[n];
        }
    } else {
        if (T % N != 0) return KDA_ERR_INVALID_ARG;
        for (size_t n = 0; n <= N; ++n) bos[n] = (int64_t)(n * (T / N));
    }
    if (T > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return KDA_ERR_INVALID_ARG;
    if (workspace_bytes < kda_prefill_host_workspace_bytes(desc, segment_tokens)) return KDA_ERR_WORKSPACE;
    const void* ins[] = {q, k, v, g, beta, cu_seqlens, init_state};
    const size_t in_n[] = {T * s.in_row_q, T * s.in_row_q, T * s.in_row_v, T * s.row_g, T * s.row_beta,
                           cu_seqlens ? s.cu_bytes : 0, init_state ? s.state_bytes : 0};
    for (int i = 0; i < 7; ++i) {
        if (host_overlap(out, T * s.row_out, ins[i], in_n[i])) return KDA_ERR_INVALID_ARG;
        if (i < 6 && host_overlap(final_state, s.state_bytes, ins[i], in_n[i])) return KDA_ERR_INVALID_ARG;
    }
    if (host_overlap(final_state, s.state_bytes, out, T * s.row_out)) return KDA_ERR_INVALID_ARG;
    if (final_state && init_state && final_state != init_state &&
        host_overlap(final_state, s.state_bytes, init_state, s.state_bytes))
        return KDA_ERR_INVALID_ARG;

    // ---- round plan: tokens of sequence n in round r = clamp(len_n - r L, 0, L)
    const int64_t L = segment_tokens;
    int64_t max_len = 0;
    for (size_t n = 0; n < N; ++n) max_len = std::max<int64_t>(max_len, bos[n + 1] - bos[n]);
    const int64_t rounds = (max_len + L - 1) / L;
    std::vector<int32_t> cu_rounds((size_t)rounds * (N + 1));
    for (int64_t r = 0; r < rounds; ++r) {
        int32_t* cu = &cu_rounds[(size_t)r * (N + 1)];
        cu[0] = 0;
        for (size_t n = 0; n < N; ++n) {
            const int64_t len = bos[n + 1] - bos[n];
            const int64_t t = std::min<int64_t>(std::max<int64_t>(len - r * L, 0), L);
            cu[n + 1] = cu[n] + (int32_t)t;
        }
    }

    HostPipe* hp = pipe_for_current_device();
    if (!hp) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(hp->mu);
    cudaStream_t comp = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    float* dstate = reinterpret_cast<float*>(ws);
    Stage stage[2] = {carve(ws + align_up(s.state_bytes), s),
                      carve(ws + align_up(s.state_bytes) + stage_bytes(s), s)};

    // On an error after work has been enqueued, the caller's stream is still made to wait for
    // every copy already queued on the library's streams (best effort), so that the contract
    // holds on failure too: once `stream` has drained, no copy reads the host inputs or the
    // workspace, or writes out or final_state.
    auto join = [&]() {
        for (int u = 0; u < kUp; ++u)
            if (cudaEventRecord(hp->end, hp->up[u]) == cudaSuccess) (void)cudaStreamWaitEvent(comp, hp->end, 0);
        if (cudaEventRecord(hp->end, hp->down) == cudaSuccess) (void)cudaStreamWaitEvent(comp, hp->end, 0);
    };
#define KDA_CK(x) \
    do { \
        if ((x) != cudaSuccess) { \
            join(); \
            return KDA_ERR_CUDA; \
        } \
    } while (0)
    // everything after prior work on the caller's stream
    KDA_CK(cudaEventRecord(hp->start, comp));
    for (int u = 0; u < kUp; ++u) KDA_CK(cudaStreamWaitEvent(hp->up[u], hp->start, 0));
    KDA_CK(cudaStreamWaitEvent(hp->down, hp->start, 0));
    if (init_state)
        KDA_CK(cudaMemcpyAsync(dstate, init_state, s.state_bytes, cudaMemcpyHostToDevice, hp->up[0]));
    else
        KDA_CK(cudaMemsetAsync(dstate, 0, s.state_bytes, hp->up[0]));

    // rows [cu[n], cu[n+1]) of the round, sequence by sequence; uploads split each piece
    // into kUp parts, one per upload stream
    auto copy_rows = [&](char* dst_base, const char* src_base, size_t row, const int32_t* cu, int64_t r,
                         cudaMemcpyKind kind, bool to_device) -> bool {
        for (size_t n = 0; n < N; ++n) {
            const size_t cnt = (size_t)(cu[n + 1] - cu[n]);
            if (cnt == 0) continue;
            const size_t host_tok = (size_t)(bos[n] + r * L), dev_tok = (size_t)cu[n];
            char* dst = dst_base + (to_device ? dev_tok : host_tok) * row;
            const char* src = src_base + (to_device ? host_tok : dev_tok) * row;
            if (!to_device) {
                if (cudaMemcpyAsync(dst, src, cnt * row, kind, hp->down) != cudaSuccess) return false;
                continue;
            }
            size_t done = 0;
            for (int u = 0; u < kUp; ++u) {
                const size_t part = (cnt * (u + 1)) / kUp - done;
                if (part > 0 && cudaMemcpyAsync(dst + done * row, src + done * row, part * row, kind, hp->up[u]) !=
                                    cudaSuccess)
                    return false;
                done += part;
            }
        }
        return true;
    };

    for (int64_t r = 0; r < rounds; ++r) {
        const int b = (int)(r & 1);
        const int32_t* cu = &cu_rounds[(size_t)r * (N + 1)];
        const Stage& sg = stage[b];
        // inputs of round r, once round r-2 has left this staging set
        if (r >= 2)
            for (int u = 0; u < kUp; ++u) KDA_CK(cudaStreamWaitEvent(hp->up[u], hp->drained[b], 0));
        const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
        if (!copy_rows(sg.q, static_cast<const char*>(q), s.in_row_q, cu, r, h2d, true) ||
            !copy_rows(sg.k, static_cast<const char*>(k), s.in_row_q, cu, r, h2d, true) ||
            !copy_rows(sg.v, static_cast<const char*>(v), s.in_row_v, cu, r, h2d, true) ||
            !copy_rows(sg.g, reinterpret_cast<const char*>(g), s.row_g, cu, r, h2d, true) ||
            !copy_rows(sg.beta, reinterpret_cast<const char*>(beta), s.row_beta, cu, r, h2d, true)) {
            join();
            return KDA_ERR_CUDA;
        }
        KDA_CK(cudaMemcpyAsync(sg.cu, cu, s.cu_bytes, h2d, hp->up[0]));
        for (int u = 0; u < kUp; ++u) KDA_CK(cudaEventRecord(hp->staged[b][u], hp->up[u]));
        // round r on the caller's stream, continuing the device state in place
        for (int u = 0; u < kUp; ++u) KDA_CK(cudaStreamWaitEvent(comp, hp->staged[b][u], 0));
        kda_prefill_desc rd = d;
        rd.total_tokens = cu[N];
        st = kda::prefill_no_workspace(&rd, sg.q, sg.k, sg.v, reinterpret_cast<const float*>(sg.g),
                                       reinterpret_cast<const float*>(sg.beta), sg.cu, dstate,
                                       reinterpret_cast<float*>(sg.out), dstate, comp);
        if (st != KDA_OK) {
            join();
            return st;
        }
        KDA_CK(cudaEventRecord(hp->computed[b], comp));
        // outputs of round r
        KDA_CK(cudaStreamWaitEvent(hp->down, hp->computed[b], 0));
        if (!copy_rows(reinterpret_cast<char*>(out), sg.out, s.row_out, cu, r, cudaMemcpyDeviceToHost, false)) {
            join();
            return KDA_ERR_CUDA;
        }
        KDA_CK(cudaEventRecord(hp->drained[b], hp->down));
    }
    if (final_state) {
        if (rounds == 0) {   // no tokens at all: the state only passes through
            KDA_CK(cudaEventRecord(hp->computed[0], hp->up[0]));
            KDA_CK(cudaStreamWaitEvent(hp->down, hp->computed[0], 0));
        }
        KDA_CK(cudaMemcpyAsync(final_state, dstate, s.state_bytes, cudaMemcpyDeviceToHost, hp->down));
    }
    // the caller's stream waits for the last copies
    KDA_CK(cudaEventRecord(hp->end, hp->down));
    KDA_CK(cudaStreamWaitEvent(comp, hp->end, 0));
    if (rounds == 0) {   // the upload stream's state copy must finish before the caller reuses init_state
        KDA_CK(cudaEventRecord(hp->end, hp->up[0]));
        KDA_CK(cudaStreamWaitEvent(comp, hp->end, 0));
    }
#undef KDA_CK
    return KDA_OK;
}

}  // extern "C"
