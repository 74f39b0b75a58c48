// kda_prefill_host_static: the host-buffer prefill with its device staging in a fixed
// scratch array of this library, so that a call allocates nothing and needs no device
// buffer from the caller.  It serves callers that cannot call cudaMalloc when a request
// arrives: a process whose device memory already belongs to its own pool, or a loop that
// cannot take the synchronisation a cudaMalloc may cause.  Declarations and contracts:
// include/kda.h.
//
// The scratch is one file-scope __device__ array, KDA_STATIC_SCRATCH_BYTES (64 MiB) on every
// device that loads the library, held until exit.  In host code its name is only a host-side
// stand-in, so the device address is taken once per device, on the first call with that
// device current, with cudaGetSymbolAddress (the first call also creates one event; it should
// come before any stream capture).  Calls share the array, so each call's work on the device
// is ordered after the previous call's: the caller's stream waits for an event that the
// previous call recorded on its own stream behind all of its copies and kernels, and the
// call records that event anew behind its own.  Each call writes all of the scratch it reads
// (the state is copied in or zeroed first), so nothing left by the previous call is used.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kda.h"

static __device__ __align__(256) unsigned char g_kda_static_scratch[KDA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

struct StaticScratch {
    void* base = nullptr;
    cudaEvent_t done = nullptr;   // recorded after the previous call's work
    bool used = false;
    std::mutex mu;
};

StaticScratch* scratch_for_current_device()
{
    static std::mutex mu;
    static StaticScratch slots[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    StaticScratch& s = slots[dev];
    if (!s.base) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kda_static_scratch) != cudaSuccess) return nullptr;
        if (cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming) != cudaSuccess) return nullptr;
        s.base = p;
    }
    return &s;
}

}  // namespace

extern "C" kda_status kda_prefill_host_static(const kda_prefill_desc* desc, const void* q, const void* k,
                                              const void* v, const float* g, const float* beta,
                                              const int32_t* cu_seqlens, const float* init_state, float* out,
                                              float* final_state, int32_t segment_tokens, void* stream)
{
    // host-only checks first: the arguments (through the planning query) and the size
    kda_prefill_plan plan;
    const kda_status st = kda_prefill_query(desc, &plan);
    if (st != KDA_OK) return st;
    if (desc->num_seqs == 0) return KDA_OK;
    if (segment_tokens <= 0 || segment_tokens % 64 != 0) return KDA_ERR_INVALID_ARG;
    const size_t need = kda_prefill_host_workspace_bytes(desc, segment_tokens);
    if (need > (size_t)KDA_STATIC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;

    StaticScratch* s = scratch_for_current_device();
    if (!s) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(s->mu);
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    if (s->used && cudaStreamWaitEvent(strm, s->done, 0) != cudaSuccess) return KDA_ERR_CUDA;
    const kda_status r = kda_prefill_host(desc, q, k, v, g, beta, cu_seqlens, init_state, out, final_state,
                                          segment_tokens, s->base, (size_t)KDA_STATIC_SCRATCH_BYTES, stream);
    // Whatever the outcome, the event is recorded behind this call's work: kda_prefill_host
    // leaves `strm` waiting for every copy and kernel it enqueued, on failure too, so the next
    // call cannot reuse the scratch while a failed call's partial work still runs.  (After an
    // argument error nothing was enqueued; the event then marks the previous call's end.)
    const bool recorded = cudaEventRecord(s->done, strm) == cudaSuccess;
    if (recorded) s->used = true;
    if (r != KDA_OK) return r;
    return recorded ? KDA_OK : KDA_ERR_CUDA;
}
