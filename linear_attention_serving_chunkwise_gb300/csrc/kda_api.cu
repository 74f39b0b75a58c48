// C ABI of the KDA library: host-side validation, workspace sizing, dispatch
// and the per-device status word.  Declarations and contracts: include/kda.h.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kda.h"
#include "kda_common.cuh"
#include "kda_launch.h"

namespace {

constexpr int kMaxDevices = 64;

// Per-device error word written by kernels (first error wins).
__device__ int g_kda_device_status;

int* status_ptr_for_current_device()
{
    static std::mutex mu;
    static int* ptrs[kMaxDevices] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kda_device_status) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int*>(p);
    }
    return ptrs[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};
Range range_of(const void* p, size_t bytes)
{
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + bytes};
}
bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo; }

bool supported_dims(int dk, int dv) { return dk == dv && (dk == 64 || dk == 128); }

// bf16 inputs with dk = dv = 128 run on the tcgen05 kernel; everything else on the fp32 CUDA-core kernel.
bool uses_tensor_cores(const kda_prefill_desc& d)
{
    return d.qkv_dtype == KDA_BF16 && d.dk == 128 && d.dv == 128 && d.total_tokens > 0 && d.num_seqs > 0;
}

// Which tensor-core path a bf16, dk = dv = 128 call takes, from its shape alone.  One CTA per
// (sequence, head) unit walks that unit's chunks; with U units on the GB300's 152 SMs that is
// ceil(U / 152) waves of about 25.8 K cycles per chunk.  The chunk-parallel split runs the
// state-independent work of every (chunk, head) item on all SMs (about 19.5 K cycles per
// item, counted as 21.0 K: at over 120 units its separate launches overlap less) and then the
// state scan, again in ceil(U / 152) waves but of about 5 K cycles per chunk (counted as
// 6.4 K, which also keeps many short sequences, e.g. 120 of 200 tokens, on one CTA each), plus a fixed 10 K cycles (the extra launch, the pipeline's fill); its workspace holds
// 115,200 bytes per item, at most kSplitMaxItems of them.  The split is taken when its
// estimate is lower.  For 8192-token sequences that is up to about 140 units (measured: at 136
// units 1.55 ms with the split against 1.58 ms with one CTA per unit; at 144, 1.64 ms against
// 1.58 ms), and again from 153 units to the item cap, where one CTA per unit would run a
// mostly idle second wave.
constexpr long long kGpuSMs = 152;
constexpr long long kSplitMaxItems = 32768;
constexpr long long kCyclesPerChunkOneCta = 258;     // hundreds of cycles
constexpr long long kCyclesPerItemPrep = 210;
constexpr long long kCyclesPerChunkScan = 64;
constexpr long long kCyclesSplitFixed = 100;

bool uses_split(const kda_prefill_desc& d)
{
    if (!uses_tensor_cores(d)) return false;
    const long long units = (long long)d.num_seqs * d.num_heads;
    const long long items = ((long long)d.total_tokens / 64 + d.num_seqs) * d.num_heads;
    if (items > kSplitMaxItems) return false;
    const long long chunks = ((long long)d.total_tokens / d.num_seqs + 63) / 64;   // of an average sequence
    const long long waves = (units + kGpuSMs - 1) / kGpuSMs;
    const long long one_cta = waves * chunks * kCyclesPerChunkOneCta;
    const long long split =
        items * kCyclesPerItemPrep / kGpuSMs + waves * chunks * kCyclesPerChunkScan + kCyclesSplitFixed;
    return split < one_cta;
}

// Launches of one call: the chunk-parallel path is one launch of chunk offsets plus either
// the single cooperative prep-and-scan launch (while at least 32 of the 152 SMs' CTAs never
// scan) or the separate prep and scan launches; otherwise one launch.
int split_launches(const kda_prefill_desc& d)
{
    if (!uses_split(d)) return 1;
    return (long long)d.num_seqs * d.num_heads + 32 <= kGpuSMs ? 2 : 3;
}

kda_status validate_prefill(const kda_prefill_desc* d)
{
    if (!d) return KDA_ERR_INVALID_ARG;
    if (d->num_seqs < 0 || d->total_tokens < 0 || d->num_heads < 1 || d->num_heads > 65535)
        return KDA_ERR_INVALID_ARG;
    if (d->qkv_dtype != KDA_F32 && d->qkv_dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!supported_dims(d->dk, d->dv)) return KDA_ERR_UNSUPPORTED;
    if (d->num_seqs == 0 && d->total_tokens != 0) return KDA_ERR_INVALID_ARG;
    if (d->prologue & ~KDA_PROLOGUE_ALL) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

}  // namespace

extern "C" {

int32_t kda_abi_version(void) { return KDA_ABI_VERSION; }

const char* kda_status_string(kda_status s)
{
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: unsupported shape or dtype (dk == dv in {64, 128})";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE: workspace too small";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA runtime or launch failure";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: a bounded device wait gave up";
    }
    return "KDA: unknown status";
}

size_t kda_prefill_workspace_bytes(const kda_prefill_desc* desc)
{
    if (validate_prefill(desc) != KDA_OK) return 0;
    if (!uses_split(*desc)) return 0;
    return kda::prefill_split_workspace_bytes(desc->num_seqs, desc->total_tokens, desc->num_heads);
}

kda_status kda_prefill_query(const kda_prefill_desc* desc, kda_prefill_plan* plan)
{
    const kda_status st = validate_prefill(desc);
    if (st != KDA_OK) return st;
    if (!plan) return KDA_ERR_INVALID_ARG;
    plan->kernel_launches = desc->num_seqs > 0 ? split_launches(*desc) : 0;
    plan->tensor_cores = uses_tensor_cores(*desc) ? 1 : 0;
    plan->workspace_bytes = kda_prefill_workspace_bytes(desc);
    return KDA_OK;
}

}  // extern "C"

namespace {

kda_status prefill_impl(const kda_prefill_desc* desc, const void* q, const void* k, const void* v, const float* g,
                        const float* beta, const int32_t* cu_seqlens, const float* init_state, float* out,
                        float* final_state, int32_t ckpt_interval, int32_t ckpt_slots, float* checkpoints,
                        void* workspace, size_t workspace_bytes, void* stream, bool allow_split,
                        const float* gate = nullptr)
{
    kda_status st = validate_prefill(desc);
    if (st != KDA_OK) return st;
    const kda_prefill_desc d = *desc;
    if (!cu_seqlens && d.num_seqs > 0 && d.total_tokens % d.num_seqs != 0) return KDA_ERR_INVALID_ARG;
    const bool split = allow_split && uses_split(d);
    const size_t ws_need = split ? kda_prefill_workspace_bytes(desc) : 0;
    if (workspace_bytes < ws_need) return KDA_ERR_WORKSPACE;
    if (split && (!workspace || !aligned16(workspace))) return KDA_ERR_INVALID_ARG;
    if (d.num_seqs == 0) return KDA_OK;

    const size_t T = (size_t)d.total_tokens, H = (size_t)d.num_heads, N = (size_t)d.num_seqs;
    const size_t esz = d.qkv_dtype == KDA_BF16 ? 2 : 4;
    if (T > 0) {
        if (!q || !k || !v || !g || !beta || !out) return KDA_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(out))
            return KDA_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(beta) & 3u) return KDA_ERR_INVALID_ARG;
    }
    if (init_state && !aligned16(init_state)) return KDA_ERR_INVALID_ARG;
    if (final_state && !aligned16(final_state)) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return KDA_ERR_INVALID_ARG;
    if (gate && !aligned16(gate)) return KDA_ERR_INVALID_ARG;

    // outputs must not overlap inputs (init_state == final_state exactly is allowed)
    const size_t sbytes = N * H * d.dk * d.dv * sizeof(float);
    const Range r_out = range_of(out, T * H * d.dv * sizeof(float));
    const Range r_fin = range_of(final_state, final_state ? sbytes : 0);
    const Range ins[] = {range_of(q, T * H * d.dk * esz), range_of(k, T * H * d.dk * esz),
                         range_of(v, T * H * d.dv * esz), range_of(g, T * H * d.dk * sizeof(float)),
                         range_of(beta, T * H * sizeof(float)),
                         range_of(cu_seqlens, cu_seqlens ? (N + 1) * sizeof(int32_t) : 0),
                         range_of(init_state, init_state ? sbytes : 0)};
    for (const Range& r : ins) {
        if (T > 0 && overlaps(r_out, r)) return KDA_ERR_INVALID_ARG;
    }
    for (int i = 0; i < 6; ++i) {
        if (final_state && overlaps(r_fin, ins[i])) return KDA_ERR_INVALID_ARG;
    }
    if (final_state && init_state && final_state != init_state && overlaps(r_fin, ins[6]))
        return KDA_ERR_INVALID_ARG;
    if (final_state && T > 0 && overlaps(r_fin, r_out)) return KDA_ERR_INVALID_ARG;
    const Range r_gate = range_of(gate, gate ? T * H * d.dv * sizeof(float) : 0);
    if (overlaps(r_gate, r_out) || overlaps(r_gate, r_fin)) return KDA_ERR_INVALID_ARG;
    const Range r_ws = range_of(workspace, ws_need);
    if (split) {   // the workspace is written: it must not overlap anything else
        for (const Range& r : ins) {
            if (overlaps(r_ws, r)) return KDA_ERR_INVALID_ARG;
        }
        if (overlaps(r_ws, r_out) || (final_state && overlaps(r_ws, r_fin)) || overlaps(r_ws, r_gate))
            return KDA_ERR_INVALID_ARG;
    }
    if (checkpoints) {
        if (ckpt_interval <= 0 || ckpt_interval % 64 != 0 || ckpt_slots <= 0 || !aligned16(checkpoints))
            return KDA_ERR_INVALID_ARG;
        const Range r_ck = range_of(checkpoints, N * H * (size_t)ckpt_slots * d.dk * d.dv * sizeof(float));
        for (const Range& r : ins) {
            if (overlaps(r_ck, r)) return KDA_ERR_INVALID_ARG;
        }
        if ((T > 0 && overlaps(r_ck, r_out)) || (final_state && overlaps(r_ck, r_fin)) || overlaps(r_ck, r_ws))
            return KDA_ERR_INVALID_ARG;
    }

    int* status = status_ptr_for_current_device();
    if (!status) return KDA_ERR_CUDA;

    kda::PrefillArgs a;
    a.num_seqs = d.num_seqs; a.total_tokens = d.total_tokens; a.num_heads = d.num_heads;
    a.dk = d.dk; a.dv = d.dv; a.bf16 = d.qkv_dtype == KDA_BF16;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.cu_seqlens = cu_seqlens;
    a.init_state = init_state; a.out = out; a.final_state = final_state;
    a.ckpt_interval = checkpoints ? ckpt_interval : 0;
    a.ckpt_slots = checkpoints ? ckpt_slots : 0;
    a.checkpoints = checkpoints;
    a.workspace = workspace; a.workspace_bytes = workspace_bytes; a.status = status;
    a.prologue = d.prologue;
    a.gate = T > 0 ? gate : nullptr;
    const cudaStream_t sm = static_cast<cudaStream_t>(stream);
    const cudaError_t e = split                  ? kda::launch_prefill_split(a, sm)
                          : uses_tensor_cores(d) ? kda::launch_prefill_tc(a, sm)
                                                 : kda::launch_prefill_simt(a, sm);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

namespace kda {

// kda_prefill restricted to the kernels that need no workspace (the host-buffer path's rounds)
kda_status prefill_no_workspace(const kda_prefill_desc* desc, const void* q, const void* k, const void* v,
                                const float* g, const float* beta, const int32_t* cu_seqlens, const float* init_state,
                                float* out, float* final_state, void* stream)
{
    return prefill_impl(desc, q, k, v, g, beta, cu_seqlens, init_state, out, final_state, 0, 0, nullptr, nullptr, 0,
                        stream, false);
}

}  // namespace kda

extern "C" {

kda_status kda_prefill(const kda_prefill_desc* desc, const void* q, const void* k, const void* v,
                       const float* g, const float* beta, const int32_t* cu_seqlens,
                       const float* init_state, float* out, float* final_state,
                       void* workspace, size_t workspace_bytes, void* stream)
{
    return prefill_impl(desc, q, k, v, g, beta, cu_seqlens, init_state, out, final_state, 0, 0, nullptr, workspace,
                        workspace_bytes, stream, true);
}

kda_status kda_prefill_gated(const kda_prefill_desc* desc, const void* q, const void* k, const void* v,
                             const float* g, const float* beta, const float* gate, const int32_t* cu_seqlens,
                             const float* init_state, float* out, float* final_state, void* workspace,
                             size_t workspace_bytes, void* stream)
{
    return prefill_impl(desc, q, k, v, g, beta, cu_seqlens, init_state, out, final_state, 0, 0, nullptr, workspace,
                        workspace_bytes, stream, true, gate);
}

kda_status kda_prefill_checkpointed(const kda_prefill_desc* desc, const void* q, const void* k, const void* v,
                                    const float* g, const float* beta, const int32_t* cu_seqlens,
                                    const float* init_state, float* out, float* final_state,
                                    int32_t checkpoint_interval, int32_t checkpoint_slots, float* checkpoints,
                                    void* workspace, size_t workspace_bytes, void* stream)
{
    if (!checkpoints) return KDA_ERR_INVALID_ARG;
    return prefill_impl(desc, q, k, v, g, beta, cu_seqlens, init_state, out, final_state, checkpoint_interval,
                        checkpoint_slots, checkpoints, workspace, workspace_bytes, stream, true);
}

kda_status kda_decode_gated(int32_t batch, int32_t num_heads, int32_t dk, int32_t dv, int32_t qkv_dtype,
                            int32_t prologue, const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* gate, float* state, float* out, void* stream)
{
    if (batch < 0 || num_heads < 1 || (prologue & ~KDA_PROLOGUE_ALL)) return KDA_ERR_INVALID_ARG;
    if (qkv_dtype != KDA_F32 && qkv_dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!supported_dims(dk, dv)) return KDA_ERR_UNSUPPORTED;
    const size_t BH = (size_t)batch * num_heads;
    if (BH > 0x7fffffffull) return KDA_ERR_INVALID_ARG;
    if (BH == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !state || !out) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(state) || !aligned16(out))
        return KDA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(beta) & 3u) return KDA_ERR_INVALID_ARG;
    const size_t esz = qkv_dtype == KDA_BF16 ? 2 : 4;
    const Range r_state = range_of(state, BH * dk * dv * sizeof(float));
    const Range r_out = range_of(out, BH * dv * sizeof(float));
    const Range ins[] = {range_of(q, BH * dk * esz), range_of(k, BH * dk * esz), range_of(v, BH * dv * esz),
                         range_of(g, BH * dk * sizeof(float)), range_of(beta, BH * sizeof(float))};
    for (const Range& r : ins) {
        if (overlaps(r_out, r) || overlaps(r_state, r)) return KDA_ERR_INVALID_ARG;
    }
    if (overlaps(r_out, r_state)) return KDA_ERR_INVALID_ARG;
    if (gate) {
        if (!aligned16(gate)) return KDA_ERR_INVALID_ARG;
        const Range r_gate = range_of(gate, BH * dv * sizeof(float));
        if (overlaps(r_gate, r_out) || overlaps(r_gate, r_state)) return KDA_ERR_INVALID_ARG;
    }

    kda::DecodeArgs a;
    a.batch = batch; a.num_heads = num_heads; a.dk = dk; a.dv = dv; a.bf16 = qkv_dtype == KDA_BF16;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.state = state; a.out = out;
    a.prologue = prologue;
    a.gate = gate;
    const cudaError_t e = kda::launch_decode(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_decode(int32_t batch, int32_t num_heads, int32_t dk, int32_t dv, int32_t qkv_dtype,
                      int32_t prologue, const void* q, const void* k, const void* v, const float* g,
                      const float* beta, float* state, float* out, void* stream)
{
    return kda_decode_gated(batch, num_heads, dk, dv, qkv_dtype, prologue, q, k, v, g, beta, nullptr, state, out,
                            stream);
}

kda_status kda_decode_multi_gated(int32_t batch, int32_t tokens, int32_t num_heads, int32_t dk, int32_t dv,
                                  int32_t qkv_dtype, int32_t prologue, const void* q, const void* k, const void* v,
                                  const float* g, const float* beta, const float* gate, const int32_t* n_apply,
                                  float* state, float* out, void* stream)
{
    if (batch < 0 || num_heads < 1 || tokens < 1 || tokens > KDA_DECODE_MULTI_MAX_TOKENS) return KDA_ERR_INVALID_ARG;
    if (prologue & ~KDA_PROLOGUE_ALL) return KDA_ERR_INVALID_ARG;
    if (qkv_dtype != KDA_F32 && qkv_dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!supported_dims(dk, dv)) return KDA_ERR_UNSUPPORTED;
    const size_t BH = (size_t)batch * num_heads;
    if (BH > 0x7fffffffull || (size_t)batch * tokens * num_heads > 0x7fffffffull) return KDA_ERR_INVALID_ARG;
    if (BH == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !state) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(state) ||
        (out && !aligned16(out)))
        return KDA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(beta) & 3u) || (reinterpret_cast<uintptr_t>(n_apply) & 3u))
        return KDA_ERR_INVALID_ARG;
    const size_t BKH = BH * (size_t)tokens;
    const size_t esz = qkv_dtype == KDA_BF16 ? 2 : 4;
    const Range r_state = range_of(state, BH * dk * dv * sizeof(float));
    const Range r_out = range_of(out, out ? BKH * dv * sizeof(float) : 0);
    const Range ins[] = {range_of(q, BKH * dk * esz), range_of(k, BKH * dk * esz), range_of(v, BKH * dv * esz),
                         range_of(g, BKH * dk * sizeof(float)), range_of(beta, BKH * sizeof(float)),
                         range_of(n_apply, n_apply ? (size_t)batch * sizeof(int32_t) : 0)};
    for (const Range& r : ins) {
        if (overlaps(r_out, r) || overlaps(r_state, r)) return KDA_ERR_INVALID_ARG;
    }
    if (overlaps(r_out, r_state)) return KDA_ERR_INVALID_ARG;
    if (!out) gate = nullptr;
    if (gate) {
        if (!aligned16(gate)) return KDA_ERR_INVALID_ARG;
        const Range r_gate = range_of(gate, BKH * dv * sizeof(float));
        if (overlaps(r_gate, r_out) || overlaps(r_gate, r_state)) return KDA_ERR_INVALID_ARG;
    }
    int* status = status_ptr_for_current_device();
    if (!status) return KDA_ERR_CUDA;

    kda::DecodeMultiArgs a;
    a.batch = batch; a.tokens = tokens; a.num_heads = num_heads; a.dk = dk; a.dv = dv;
    a.bf16 = qkv_dtype == KDA_BF16;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.n_apply = n_apply;
    a.state = state; a.out = out; a.status = status; a.prologue = prologue;
    a.gate = gate;
    const cudaError_t e = kda::launch_decode_multi(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_decode_multi(int32_t batch, int32_t tokens, int32_t num_heads, int32_t dk, int32_t dv,
                            int32_t qkv_dtype, int32_t prologue, const void* q, const void* k, const void* v,
                            const float* g, const float* beta, const int32_t* n_apply, float* state, float* out,
                            void* stream)
{
    return kda_decode_multi_gated(batch, tokens, num_heads, dk, dv, qkv_dtype, prologue, q, k, v, g, beta, nullptr,
                                  n_apply, state, out, stream);
}

kda_status kda_last_device_status(void* stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KDA_ERR_CUDA;
    int* p = status_ptr_for_current_device();
    if (!p) return KDA_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return KDA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return KDA_ERR_CUDA;
    switch (h) {
        case kda::kDevOk: return KDA_OK;
        case kda::kDevBadSeqlens: return KDA_ERR_INVALID_ARG;
        case kda::kDevTimeout: return KDA_ERR_TIMEOUT;
        default: return KDA_ERR_CUDA;
    }
}

}  // extern "C"
