// Shared device helpers of the KDA library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// Device status codes (mirror kda_status in include/kda.h).
constexpr int kDevOk = 0;
constexpr int kDevBadSeqlens = -1;
constexpr int kDevTimeout = -5;

__device__ __forceinline__ void report_status(int* status, int code)
{
    // first error wins; later ones are dropped
    atomicCAS(status, kDevOk, code);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Input prologue (bits of KDA_PROLOGUE_* in include/kda.h): the workloads' recipe for q, k,
// g and beta, applied as the kernels load them.  g_min = -5 is the pages' bound on the
// log-decay (llm-atlas Q06).
constexpr int kProQK = 1, kProG = 2, kProBeta = 4;
constexpr float kGMin = -5.f;
constexpr float kL2Eps = 1e-12f;
// sigmoid(y) = 1 / (1 + e^-y) with the fast exponential and division (a few ulp of fp32 from
// the exact value; 0 and 1 at the ends), for the prologue's parametrisations, which run on
// every g element on the prefill's critical path, and the output gate.  Parity against the
// oracle's fp64 sigmoid is tested.
__device__ __forceinline__ float sigmoid_fast(float y) { return __fdividef(1.f, 1.f + __expf(-y)); }
__device__ __forceinline__ float g_of(float g, int prologue) { return (prologue & kProG) ? kGMin * sigmoid_fast(g) : g; }
__device__ __forceinline__ float beta_of(float b, int prologue) { return (prologue & kProBeta) ? sigmoid_fast(b) : b; }
// x / max(||x||, eps) as x times the row's reciprocal norm, rounded to the storage type of q and k
__device__ __forceinline__ float l2_scale(float x, float inv, float) { return x * inv; }
__device__ __forceinline__ float l2_scale(float x, float inv, __nv_bfloat16)
{
    return __bfloat162float(__float2bfloat16_rn(x * inv));
}
// 1 / max(||x||, eps) = rsqrt(max(||x||^2, eps^2)) (eps^2 = 1e-24 is a normal float), by the
// fast reciprocal square root: a few ulp of fp32, far below the bf16 rounding that follows
__device__ __forceinline__ float l2_inv(float sumsq) { return rsqrtf(fmaxf(sumsq, kL2Eps * kL2Eps)); }

// Output gate (llm-atlas Q08, read as an elementwise sigmoid over the read-out channels):
// o <- o * sigmoid(z), with the fast sigmoid (it runs on every output element, in the O
// warps of the tensor-core kernels alongside the state update).
__device__ __forceinline__ float gate1(float o, float z) { return o * sigmoid_fast(z); }
// for 4 consecutive outputs and their logits in global memory (16-byte aligned)
__device__ __forceinline__ float4 gate4(float4 o, const float* z)
{
    const float4 zz = __ldg(reinterpret_cast<const float4*>(z));
    return make_float4(gate1(o.x, zz.x), gate1(o.y, zz.y), gate1(o.z, zz.z), gate1(o.w, zz.w));
}

// Read 4 consecutive elements starting at a 4-element-aligned index.
__device__ __forceinline__ float4 load4(const float* p)
{
    return __ldg(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p)
{
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
    float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}

// Sequence bounds [bos, eos) for sequence n, validated against total_tokens.
// Returns false (and records a device error) for a malformed cu_seqlens entry.
__device__ __forceinline__ bool seq_bounds(const int32_t* cu_seqlens, int n, int num_seqs, int total_tokens,
                                           int* status, int& bos, int& eos)
{
    if (cu_seqlens == nullptr) {
        const int len = total_tokens / num_seqs;
        bos = n * len;
        eos = bos + len;
        return true;
    }
    bos = cu_seqlens[n];
    eos = cu_seqlens[n + 1];
    const bool ok = (bos >= 0) && (eos >= bos) && (eos <= total_tokens) &&
                    (n != 0 || bos == 0) && (n != num_seqs - 1 || eos == total_tokens);
    if (!ok) report_status(status, kDevBadSeqlens);
    return ok;
}

}  // namespace kda
