// Chunkwise KDA prefill on CUDA cores in fp32 (the fp32-input path).
//
// Chunkwise form (llm-atlas "K3_RESEARCH.md", Q07: state passed between
// chunks, parallel matrix work inside a chunk).  For a chunk of n <= 64 tokens
// entered with state S, Gamma_r = inclusive prefix sum of g over the chunk:
//   A[r][i] = beta_r sum_c k_r[c] k_i[c] exp(Gamma_r[c] - Gamma_i[c])   (i < r)
//   P[r][i] =        sum_c q_r[c] k_i[c] exp(Gamma_r[c] - Gamma_i[c])   (i <= r)
//   (I + A) [U | Wk] = diag(beta) [V | K*exp(Gamma)]     (forward substitution)
//   W = U - Wk S;  O = (Q*exp(Gamma)) S + P W
//   S <- Diag(exp Gamma_n) S + (K*exp(Gamma_n - Gamma))^T W
// Every decay between two tokens is one exponential of a difference of prefix
// sums, each of which is <= 0 because g <= 0, so nothing overflows.
//
// One CTA per (sequence, head, 32-column slice of dv): the columns of S evolve
// independently, so the slices need no communication.  fp32 throughout.
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

constexpr int kChunk = 64;
constexpr int kSlice = 32;   // value columns per CTA
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kAld = kChunk + 1;  // padded row stride of A and P

template <int D>
constexpr size_t simt_smem_bytes()
{
    return sizeof(float) * (4 * kChunk * D + 2 * kChunk * kAld + kChunk * kSlice + D * kSlice + kChunk);
}

template <typename Tin, int D>
__global__ void __launch_bounds__(kThreads, 1) kda_prefill_simt_kernel(PrefillArgs a)
{
    extern __shared__ float smem[];
    float* sQ = smem;                  // [C][D]  q, then q * exp(Gamma)
    float* sK = sQ + kChunk * D;       // [C][D]  k, then k * exp(Gamma_n - Gamma)
    float* sG = sK + kChunk * D;       // [C][D]  g, then Gamma
    float* sKg = sG + kChunk * D;      // [C][D]  beta k exp(Gamma), then Wk
    float* sA = sKg + kChunk * D;      // [C][C+1]
    float* sP = sA + kChunk * kAld;    // [C][C+1]
    float* sV = sP + kChunk * kAld;    // [C][kSlice]  beta v, then U, then W
    float* sS = sV + kChunk * kSlice;  // [D][kSlice]  state slice
    float* sB = sS + D * kSlice;       // [C] beta

    const int n = blockIdx.x, h = blockIdx.y, js = blockIdx.z * kSlice;
    const int H = a.num_heads;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    int bos, eos;
    if (!seq_bounds(a.cu_seqlens, n, a.num_seqs, a.total_tokens, a.status, bos, eos)) return;

    const Tin* q = static_cast<const Tin*>(a.q);
    const Tin* k = static_cast<const Tin*>(a.k);
    const Tin* v = static_cast<const Tin*>(a.v);
    const size_t state_base = ((size_t)n * H + h) * D * D;

    for (int idx = t; idx < D * kSlice; idx += kThreads) {
        const int c = idx / kSlice, j = idx % kSlice;
        sS[idx] = a.init_state ? a.init_state[state_base + (size_t)c * D + js + j] : 0.f;
    }

    for (int c0 = bos; c0 < eos; c0 += kChunk) {
        const int BT = min(kChunk, eos - c0);
        __syncthreads();
        for (int idx = t; idx < BT * D; idx += kThreads) {
            const int r = idx / D, c = idx % D;
            const size_t gi = ((size_t)(c0 + r) * H + h) * D + c;
            sQ[idx] = to_f32(q[gi]);
            sK[idx] = to_f32(k[gi]);
            sG[idx] = g_of(a.g[gi], a.prologue);
        }
        for (int idx = t; idx < BT * kSlice; idx += kThreads) {
            const int r = idx / kSlice, j = idx % kSlice;
            sV[idx] = to_f32(v[((size_t)(c0 + r) * H + h) * D + js + j]);
        }
        if (t < BT) sB[t] = beta_of(a.beta[(size_t)(c0 + t) * H + h], a.prologue);
        __syncthreads();
        if (a.prologue & kProQK) {   // one warp per token row of q or k
            for (int vi = warp; vi < 2 * BT; vi += kWarps) {
                float* x = (vi & 1 ? sQ : sK) + (vi >> 1) * D;
                float ss = 0.f;
                for (int c = lane; c < D; c += 32) ss += x[c] * x[c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float inv = l2_inv(ss);
                for (int c = lane; c < D; c += 32) x[c] = l2_scale(x[c], inv, Tin{});
            }
            __syncthreads();
        }

        // Gamma: inclusive prefix sum of g down the chunk, per key channel
        if (t < D) {
            float acc = 0.f;
            for (int r = 0; r < BT; ++r) {
                acc += sG[r * D + t];
                sG[r * D + t] = acc;
            }
        }
        __syncthreads();

        // A and P, one warp per (r, i) pair, lanes over key channels
        const int npairs = BT * (BT + 1) / 2;
        for (int pidx = warp; pidx < npairs; pidx += kWarps) {
            int r = (int)((sqrtf(8.f * pidx + 1.f) - 1.f) * 0.5f);
            while (r * (r + 1) / 2 > pidx) --r;
            while ((r + 1) * (r + 2) / 2 <= pidx) ++r;
            const int i = pidx - r * (r + 1) / 2;
            float kk = 0.f, qk = 0.f;
#pragma unroll
            for (int u = 0; u < D / 32; ++u) {
                const int c = lane + 32 * u;
                const float e = expf(sG[r * D + c] - sG[i * D + c]);
                const float ki = sK[i * D + c] * e;
                kk += sK[r * D + c] * ki;
                qk += sQ[r * D + c] * ki;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                kk += __shfl_xor_sync(0xffffffffu, kk, o);
                qk += __shfl_xor_sync(0xffffffffu, qk, o);
            }
            if (lane == 0) {
                sA[r * kAld + i] = (i < r) ? sB[r] * kk : 0.f;
                sP[r * kAld + i] = qk;
            }
        }
        // right-hand sides diag(beta) [V | K exp(Gamma)]
        for (int idx = t; idx < BT * D; idx += kThreads) {
            const int r = idx / D;
            sKg[idx] = sB[r] * sK[idx] * expf(sG[idx]);
        }
        for (int idx = t; idx < BT * kSlice; idx += kThreads) sV[idx] *= sB[idx / kSlice];
        __syncthreads();

        // (I + A) X = RHS by forward substitution, one column per thread
        for (int col = t; col < kSlice + D; col += kThreads) {
            float* X = (col < kSlice) ? (sV + col) : (sKg + (col - kSlice));
            const int ld = (col < kSlice) ? kSlice : D;
            for (int r = 1; r < BT; ++r) {
                float acc = X[r * ld];
                for (int i = 0; i < r; ++i) acc -= sA[r * kAld + i] * X[i * ld];
                X[r * ld] = acc;
            }
        }
        __syncthreads();

        // decayed operands in place; W = U - Wk S (in place in sV, row r by warp)
        const float* gl = sG + (BT - 1) * D;
        for (int idx = t; idx < BT * D; idx += kThreads) {
            const int c = idx % D;
            const float e = sG[idx];
            sQ[idx] *= expf(e);
            sK[idx] *= expf(gl[c] - e);
        }
        for (int r = warp; r < BT; r += kWarps) {
            float acc = sV[r * kSlice + lane];
            for (int c = 0; c < D; ++c) acc -= sKg[r * D + c] * sS[c * kSlice + lane];
            sV[r * kSlice + lane] = acc;
        }
        __syncthreads();

        // O = Q_Gamma S + P W, written in fp32
        for (int r = warp; r < BT; r += kWarps) {
            float acc = 0.f;
            for (int c = 0; c < D; ++c) acc += sQ[r * D + c] * sS[c * kSlice + lane];
            for (int i = 0; i <= r; ++i) acc += sP[r * kAld + i] * sV[i * kSlice + lane];
            const size_t oi = ((size_t)(c0 + r) * H + h) * D + js + lane;
            a.out[oi] = a.gate ? gate1(acc, __ldg(a.gate + oi)) : acc;
        }
        // S <- Diag(exp Gamma_n) S + K~^T W
        float snew[D / kWarps];
#pragma unroll
        for (int m = 0; m < D / kWarps; ++m) {
            const int c = warp + kWarps * m;
            float acc = expf(gl[c]) * sS[c * kSlice + lane];
            for (int r = 0; r < BT; ++r) acc += sK[r * D + c] * sV[r * kSlice + lane];
            snew[m] = acc;
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < D / kWarps; ++m) sS[(warp + kWarps * m) * kSlice + lane] = snew[m];
        // state snapshot after a full chunk that ends on a checkpoint boundary
        const int done = c0 + BT - bos;
        if (a.checkpoints && BT == kChunk && done % a.ckpt_interval == 0 && done / a.ckpt_interval <= a.ckpt_slots) {
            const int slot = done / a.ckpt_interval - 1;
            float* dst = a.checkpoints + (((size_t)n * H + h) * a.ckpt_slots + slot) * D * D;
#pragma unroll
            for (int m = 0; m < D / kWarps; ++m) dst[(size_t)(warp + kWarps * m) * D + js + lane] = snew[m];
        }
    }
    __syncthreads();
    if (a.final_state) {
        for (int idx = t; idx < D * kSlice; idx += kThreads) {
            const int c = idx / kSlice, j = idx % kSlice;
            a.final_state[state_base + (size_t)c * D + js + j] = sS[idx];
        }
    }
}

template <typename Tin, int D>
cudaError_t launch_simt_t(const PrefillArgs& a, cudaStream_t stream)
{
    constexpr size_t smem = simt_smem_bytes<D>();
    cudaError_t e = cudaFuncSetAttribute(kda_prefill_simt_kernel<Tin, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)a.num_seqs, (unsigned)a.num_heads, D / kSlice);
    kda_prefill_simt_kernel<Tin, D><<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t stream)
{
    if (a.num_seqs == 0) return cudaSuccess;
    if (a.dk == 128)
        return a.bf16 ? launch_simt_t<__nv_bfloat16, 128>(a, stream) : launch_simt_t<float, 128>(a, stream);
    return a.bf16 ? launch_simt_t<__nv_bfloat16, 64>(a, stream) : launch_simt_t<float, 64>(a, stream);
}

}  // namespace kda
