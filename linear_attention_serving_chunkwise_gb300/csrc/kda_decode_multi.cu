// Multi-token KDA decode: K consecutive tokens of each sequence in one pass over the
// head's fp32 state, for speculative verification of K draft tokens (llm-atlas
// "K3_RESEARCH.md", Q28: the MTP layer tuned into an EAGLE-3 draft model; Q07: decode
// keeps the O(1) state update).
//
// One CTA per (sequence, head).  Warp w owns the state columns [16 w, 16 w + 16) over all
// dk rows; lane (rs = lane / 4, cq = lane % 4) holds rows [rs D/8, (rs + 1) D/8) of the
// float4 column 4 cq in registers for the whole call.  Per token the fused step of
// single-token decode (S' = Diag(exp g) S; r = S'^T k, p = S'^T q; w = beta (v - r);
// S <- S' + k w^T; o = p + (k . q) w): every sum runs over dk, i.e. over the 8 lanes of
// one column, so a step is three shuffle rounds and no CTA barrier.  The K tokens'
// vectors are staged in shared memory once, behind the only barrier of the kernel.
// Outputs are written for every token; the state written back is the one after the
// first n_apply[b] tokens (0 leaves it untouched).
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

// shared staging of one token: k, q, e^g in padded 16-row blocks (stride 20 floats, so the
// 8 row blocks read by one warp fall in different banks), then v, then beta
template <int D>
struct MultiLayout {
    static constexpr int kBlk = 20;                    // floats per 16-row block
    static constexpr int kVec = D / 16 * kBlk;         // floats of one padded dk vector
    static constexpr int kTok = 3 * kVec + D + 4;      // floats per token (16-byte multiple)
    __device__ static int row(int r) { return (r >> 4) * kBlk + (r & 15); }
};

template <typename Tin, int D>
__global__ void __launch_bounds__(2 * D, 2) kda_decode_multi_kernel(DecodeMultiArgs a)
{
    using Lay = MultiLayout<D>;
    constexpr int R = D / 8;                  // state rows per lane
    constexpr int kThreads = 2 * D;           // D / 16 warps of 16 columns
    extern __shared__ __align__(16) float smv[];

    const int bh = blockIdx.x;                // b * H + h
    const int b = bh / a.num_heads, h = bh % a.num_heads;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int rs = lane >> 2, cq = lane & 3;
    const int K = a.tokens;
    const int col = 16 * w + 4 * cq;          // first of this lane's 4 state columns
    const int r0 = rs * R;                    // first of this lane's R rows

    int n_apply = K;
    if (a.n_apply) {
        n_apply = a.n_apply[b];
        if (n_apply < 0 || n_apply > K) {
            if (t == 0 && h == 0) report_status(a.status, kDevBadSeqlens);
            n_apply = 0;   // an invalid count leaves the state untouched
        }
    }

    float* S = a.state + (size_t)bh * D * D + col;
    float4 s[R];
#pragma unroll
    for (int i = 0; i < R; ++i) s[i] = __ldcs(reinterpret_cast<const float4*>(S + (size_t)(r0 + i) * D));

    // stage every token's vectors (plain loads, all issued before the one barrier)
    for (int idx = t; idx < K * D; idx += kThreads) {
        const int j = idx / D, c = idx - j * D;
        const size_t tok = ((size_t)b * K + j) * a.num_heads + h;   // [B, K, H, .]
        float* base = smv + j * Lay::kTok;
        base[Lay::row(c)] = to_f32(static_cast<const Tin*>(a.k)[tok * D + c]);
        base[Lay::kVec + Lay::row(c)] = to_f32(static_cast<const Tin*>(a.q)[tok * D + c]);
        base[2 * Lay::kVec + Lay::row(c)] = expf(a.g[tok * D + c]);
        base[3 * Lay::kVec + c] = to_f32(static_cast<const Tin*>(a.v)[tok * D + c]);
        if (c == 0) base[3 * Lay::kVec + D] = a.beta[tok];
    }
    __syncthreads();

    for (int j = 0; j < K; ++j) {
        const float* base = smv + j * Lay::kTok;
        const float* kv = base + Lay::row(r0);
        const float* qv = base + Lay::kVec + Lay::row(r0);
        const float* dv = base + 2 * Lay::kVec + Lay::row(r0);
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f), p = r;
        float kq = 0.f;
#pragma unroll
        for (int i4 = 0; i4 < R / 4; ++i4) {
            const float4 k4 = *reinterpret_cast<const float4*>(kv + 4 * i4);
            const float4 q4 = *reinterpret_cast<const float4*>(qv + 4 * i4);
            const float4 d4 = *reinterpret_cast<const float4*>(dv + 4 * i4);
            const float kk[4] = {k4.x, k4.y, k4.z, k4.w}, qq[4] = {q4.x, q4.y, q4.z, q4.w},
                        dd[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float4& x = s[4 * i4 + e];
                x.x *= dd[e]; x.y *= dd[e]; x.z *= dd[e]; x.w *= dd[e];
                r.x += x.x * kk[e]; r.y += x.y * kk[e]; r.z += x.z * kk[e]; r.w += x.w * kk[e];
                p.x += x.x * qq[e]; p.y += x.y * qq[e]; p.z += x.z * qq[e]; p.w += x.w * qq[e];
                kq += kk[e] * qq[e];
            }
        }
        // sums over the 8 lanes of each column (lane bits 2-4)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            r.x += __shfl_xor_sync(0xffffffffu, r.x, o); r.y += __shfl_xor_sync(0xffffffffu, r.y, o);
            r.z += __shfl_xor_sync(0xffffffffu, r.z, o); r.w += __shfl_xor_sync(0xffffffffu, r.w, o);
            p.x += __shfl_xor_sync(0xffffffffu, p.x, o); p.y += __shfl_xor_sync(0xffffffffu, p.y, o);
            p.z += __shfl_xor_sync(0xffffffffu, p.z, o); p.w += __shfl_xor_sync(0xffffffffu, p.w, o);
            kq += __shfl_xor_sync(0xffffffffu, kq, o);
        }
        const float4 v4 = *reinterpret_cast<const float4*>(base + 3 * Lay::kVec + col);
        const float beta = base[3 * Lay::kVec + D];
        const float4 w4 = make_float4(beta * (v4.x - r.x), beta * (v4.y - r.y), beta * (v4.z - r.z),
                                      beta * (v4.w - r.w));
        if (a.out && rs == 0) {
            const size_t tok = ((size_t)b * K + j) * a.num_heads + h;
            *reinterpret_cast<float4*>(a.out + tok * D + col) =
                make_float4(p.x + kq * w4.x, p.y + kq * w4.y, p.z + kq * w4.z, p.w + kq * w4.w);
        }
#pragma unroll
        for (int i4 = 0; i4 < R / 4; ++i4) {
            const float4 k4 = *reinterpret_cast<const float4*>(kv + 4 * i4);
            const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float4& x = s[4 * i4 + e];
                x.x += kk[e] * w4.x; x.y += kk[e] * w4.y; x.z += kk[e] * w4.z; x.w += kk[e] * w4.w;
            }
        }
        if (j + 1 == n_apply) {   // the state after the applied prefix
#pragma unroll
            for (int i = 0; i < R; ++i) __stcs(reinterpret_cast<float4*>(S + (size_t)(r0 + i) * D), s[i]);
        }
    }
}

template <typename Tin, int D>
cudaError_t launch_t(const DecodeMultiArgs& a, cudaStream_t stream)
{
    const long long blocks = (long long)a.batch * a.num_heads;
    if (blocks == 0) return cudaSuccess;
    const size_t smem = (size_t)a.tokens * MultiLayout<D>::kTok * sizeof(float);
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kda_decode_multi_kernel<Tin, D>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kda_decode_multi_kernel<Tin, D><<<(unsigned)blocks, 2 * D, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_multi(const DecodeMultiArgs& a, cudaStream_t stream)
{
    if (a.dk == 128) return a.bf16 ? launch_t<__nv_bfloat16, 128>(a, stream) : launch_t<float, 128>(a, stream);
    return a.bf16 ? launch_t<__nv_bfloat16, 64>(a, stream) : launch_t<float, 64>(a, stream);
}

}  // namespace kda
