// kda_state_combine: one step of the exclusive scan that context-parallel prefill runs over
// the ranks holding consecutive token ranges of one sequence (llm-atlas "K3_RESEARCH.md",
// section 8 system-state table: KCP in the pretraining row; Q07: the state is passed from
// chunk to chunk).  A range r maps the state entering it affinely,
//     S_after = M_r S_before + S_r,
// with M_r (dk x dk) the product of its chunks' transitions Diag(e^{Gamma_C}) - K~^T Wk and
// S_r its state from a zero start, so the state entering range r is a fold over the ranges
// before it: S_in <- M_j S_in + S_j.  This kernel is that fold step for a batch of heads:
//     out[i] = M[i] in[i] + add[i]      (fp32, i < count)
// Declarations and contracts: include/kda.h.
#include <cuda_runtime.h>

#include "../../include/kda.h"

namespace {

constexpr int kTile = 64;      // output tile (rows x cols) per CTA
constexpr int kKStep = 32;     // K elements staged per step
constexpr int kThreads = 256;  // 16 x 16 threads, 4 x 4 outputs each

// CTA (tile, head): out[head] rows [64 ty, +64), cols [64 tx, +64).  M row-major [D][D],
// in/add/out row-major [D][D] (row = key channel, column = value channel).
template <int D>
__global__ void __launch_bounds__(kThreads) kda_state_combine_kernel(const float* __restrict__ M,
                                                                   const float* __restrict__ in,
                                                                   const float* add, float* out)
{
    constexpr int T = D / kTile;
    const int head = blockIdx.x / (T * T), tile = blockIdx.x % (T * T);
    const int r0 = (tile / T) * kTile, c0 = (tile % T) * kTile;
    const int t = threadIdx.x, tr = t / 16, tc = t % 16;
    const size_t base = (size_t)head * D * D;
    __shared__ float sM[kTile][kKStep + 1];
    __shared__ __align__(16) float sS[kKStep][kTile];

    float acc[4][4] = {};
    if (in) {
        for (int k0 = 0; k0 < D; k0 += kKStep) {
            // M tile [64 rows][32 k] and S tile [32 k][64 cols]: 2048 values each, 8 per thread
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = t + kThreads * i;
                sM[e / kKStep][e % kKStep] = __ldg(M + base + (size_t)(r0 + e / kKStep) * D + k0 + e % kKStep);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int e = t + kThreads * i;   // float4 index, 16 per row
                const float4 v = __ldg(reinterpret_cast<const float4*>(in + base + (size_t)(k0 + e / 16) * D + c0) +
                                       e % 16);
                *reinterpret_cast<float4*>(&sS[e / 16][4 * (e % 16)]) = v;
            }
            __syncthreads();
#pragma unroll 8
            for (int k = 0; k < kKStep; ++k) {
                const float4 b = *reinterpret_cast<const float4*>(&sS[k][4 * tc]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float a = sM[4 * tr + i][k];
                    acc[i][0] = fmaf(a, b.x, acc[i][0]);
                    acc[i][1] = fmaf(a, b.y, acc[i][1]);
                    acc[i][2] = fmaf(a, b.z, acc[i][2]);
                    acc[i][3] = fmaf(a, b.w, acc[i][3]);
                }
            }
            __syncthreads();
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const size_t o = base + (size_t)(r0 + 4 * tr + i) * D + c0 + 4 * tc;
        float4 r = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        if (add) {   // read before the write below: out may be add itself
            const float4 a = *reinterpret_cast<const float4*>(add + o);
            r.x += a.x; r.y += a.y; r.z += a.z; r.w += a.w;
        }
        *reinterpret_cast<float4*>(out + o) = r;
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, const void* b, size_t bytes)
{
    if (!a || !b) return false;
    const char* pa = static_cast<const char*>(a);
    const char* pb = static_cast<const char*>(b);
    return pa < pb + bytes && pb < pa + bytes;
}

}  // namespace

extern "C" kda_status kda_state_combine(int32_t count, int32_t dk, int32_t dv, const float* transition,
                                        const float* state_in, const float* state_add, float* state_out,
                                        void* stream)
{
    if (count < 0) return KDA_ERR_INVALID_ARG;
    if (dk != dv || (dk != 64 && dk != 128)) return KDA_ERR_UNSUPPORTED;
    if ((size_t)count * (dk / kTile) * (dk / kTile) > 0x7fffffffull) return KDA_ERR_INVALID_ARG;
    if (count == 0) return KDA_OK;
    if (!state_out || (state_in && !transition)) return KDA_ERR_INVALID_ARG;
    if (!aligned16(transition) || !aligned16(state_in) || !aligned16(state_add) || !aligned16(state_out))
        return KDA_ERR_INVALID_ARG;
    const size_t bytes = (size_t)count * dk * dv * sizeof(float);
    // out is written while in and the transition are still read by other CTAs: no overlap;
    // out == add exactly is allowed (each element is read by the thread that writes it)
    if (overlap(state_out, state_in, bytes) || overlap(state_out, transition, bytes)) return KDA_ERR_INVALID_ARG;
    if (state_add && state_add != state_out && overlap(state_out, state_add, bytes)) return KDA_ERR_INVALID_ARG;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int tiles = (dk / kTile) * (dk / kTile);
    if (dk == 128)
        kda_state_combine_kernel<128><<<(unsigned)(count * tiles), kThreads, 0, s>>>(transition, state_in, state_add,
                                                                                   state_out);
    else
        kda_state_combine_kernel<64><<<(unsigned)(count * tiles), kThreads, 0, s>>>(transition, state_in, state_add,
                                                                                  state_out);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
