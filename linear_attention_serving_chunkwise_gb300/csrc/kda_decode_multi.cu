// Multi-token KDA decode: K consecutive tokens of each sequence in one pass over the
// head's fp32 state, for speculative verification of K draft tokens (llm-atlas
// "K3_RESEARCH.md", Q28: the MTP layer tuned into an EAGLE-3 draft model; Q07: decode
// keeps the O(1) state update).
//
// The CTAs of one (sequence, head) hold its state in registers for all K tokens: per token
// the same fused step as single-token decode (S' = Diag(exp g) S; r = S'^T k, p = S'^T q
// from one pass; w = beta (v - r); S <- S' + k w^T; o = p + (k . q) w).  Outputs are
// written for every token; the state written back is the one after the first
// n_apply[b] tokens (0 leaves it untouched), so a verify pass followed by an apply pass
// for the accepted prefix reads the state twice and writes it once.
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

constexpr int kMultiThreads = 256;

// SPLIT CTAs share one (sequence, head): CTA `half` owns the dv columns
// [half D / SPLIT, (half + 1) D / SPLIT) of the state.  Every reduction of the step runs
// over dk (rows), so the column blocks never exchange data; k . q is formed in each.
template <typename Tin, int D, int SPLIT>
__global__ void __launch_bounds__(kMultiThreads, SPLIT == 1 ? 2 : 3) kda_decode_multi_kernel(DecodeMultiArgs a)
{
    constexpr int DV = D / SPLIT;             // state columns of this CTA
    constexpr int C4 = DV / 4;                // float4 columns per state row
    constexpr int RG = kMultiThreads / C4;    // row groups
    constexpr int RP = D / RG;                // rows per thread
    static_assert(RG * C4 == kMultiThreads && RP * RG == D, "decode tiling");

    const int bh = blockIdx.x / SPLIT, half = blockIdx.x % SPLIT;   // bh = b * H + h
    const int b = bh / a.num_heads, h = bh % a.num_heads;
    const int t = threadIdx.x;
    const int cg = t % C4, rg = t / C4;
    const int K = a.tokens;
    const int c0 = half * DV;                 // first state column of this CTA

    // token vectors double-buffered by step parity: step j + 1 fills one buffer while no
    // thread can still read it (three barriers separate it from step j - 1)
    __shared__ float sk[2][D], sq[2][D], sdec[2][D], sv[2][DV], sw[DV];
    __shared__ float4 red_r[RG][C4], red_p[RG][C4];
    __shared__ float s_kq[2], s_beta[2];

    int n_apply = K;
    if (a.n_apply) {
        n_apply = a.n_apply[b];
        if (n_apply < 0 || n_apply > K) {
            if (t == 0 && h == 0 && half == 0) report_status(a.status, kDevBadSeqlens);
            n_apply = 0;   // an invalid count leaves the state untouched
        }
    }

    float* S = a.state + (size_t)bh * D * D + c0;
    float4 s[RP];
#pragma unroll
    for (int i = 0; i < RP; ++i) s[i] = __ldcs(reinterpret_cast<const float4*>(S + (size_t)(rg * RP + i) * D) + cg);

    // token j's vectors are loaded into registers during step j - 1
    auto tok_index = [&](int j) { return ((size_t)b * K + j) * a.num_heads + h; };   // [B, K, H, .]
    float nk = 0.f, nq = 0.f, nv = 0.f, ng = 0.f, nb = 0.f;
    auto fetch = [&](int j) {
        const size_t tok = tok_index(j);
        if (t < D) {
            nk = to_f32(static_cast<const Tin*>(a.k)[tok * D + t]);
            nq = to_f32(static_cast<const Tin*>(a.q)[tok * D + t]);
            ng = a.g[tok * D + t];
        }
        if (t < DV) nv = to_f32(static_cast<const Tin*>(a.v)[tok * D + c0 + t]);
        if (t == 0) nb = a.beta[tok];
    };
    fetch(0);

    for (int j = 0; j < K; ++j) {
        const int buf = j & 1;
        const size_t tok = tok_index(j);
        if (t < D) {
            sk[buf][t] = nk;
            sq[buf][t] = nq;
            sdec[buf][t] = expf(ng);
        }
        if (t < DV) sv[buf][t] = nv;
        if (t == 0) s_beta[buf] = nb;
        if (j + 1 < K) fetch(j + 1);
        __syncthreads();
        if (t < 32) {
            float kq = 0.f;
            for (int c = t; c < D; c += 32) kq += sk[buf][c] * sq[buf][c];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
            if (t == 0) s_kq[buf] = kq;
        }
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f), p = r;
#pragma unroll
        for (int i = 0; i < RP; ++i) {
            const int row = rg * RP + i;
            const float d = sdec[buf][row], kc = sk[buf][row], qc = sq[buf][row];
            s[i].x *= d; s[i].y *= d; s[i].z *= d; s[i].w *= d;
            r.x += s[i].x * kc; r.y += s[i].y * kc; r.z += s[i].z * kc; r.w += s[i].w * kc;
            p.x += s[i].x * qc; p.y += s[i].y * qc; p.z += s[i].z * qc; p.w += s[i].w * qc;
        }
        red_r[rg][cg] = r;
        red_p[rg][cg] = p;
        __syncthreads();
        if (t < DV) {
            const float* rr = reinterpret_cast<const float*>(&red_r[0][0]);
            const float* pp = reinterpret_cast<const float*>(&red_p[0][0]);
            float rs = 0.f, ps = 0.f;
#pragma unroll
            for (int gI = 0; gI < RG; ++gI) {
                rs += rr[gI * DV + t];
                ps += pp[gI * DV + t];
            }
            const float w = s_beta[buf] * (sv[buf][t] - rs);
            sw[t] = w;
            if (a.out) a.out[tok * D + c0 + t] = ps + s_kq[buf] * w;
        }
        __syncthreads();
        const float4 w4 = reinterpret_cast<const float4*>(sw)[cg];
#pragma unroll
        for (int i = 0; i < RP; ++i) {
            const float kc = sk[buf][rg * RP + i];
            s[i].x += kc * w4.x; s[i].y += kc * w4.y; s[i].z += kc * w4.z; s[i].w += kc * w4.w;
        }
        if (j + 1 == n_apply) {   // the state after the applied prefix
#pragma unroll
            for (int i = 0; i < RP; ++i) __stcs(reinterpret_cast<float4*>(S + (size_t)(rg * RP + i) * D) + cg, s[i]);
        }
    }
}

template <typename Tin, int D, int SPLIT>
cudaError_t launch_t(const DecodeMultiArgs& a, cudaStream_t stream)
{
    const long long blocks = (long long)a.batch * a.num_heads * SPLIT;
    if (blocks == 0) return cudaSuccess;
    kda_decode_multi_kernel<Tin, D, SPLIT><<<(unsigned)blocks, kMultiThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_multi(const DecodeMultiArgs& a, cudaStream_t stream)
{
    // one CTA per (sequence, head): splitting the columns over two CTAs measured slower on
    // GB300 (0.93 vs 0.83 ms for B = 256, H = 96, K = 4), the per-step barriers dominate
    if (a.dk == 128) return a.bf16 ? launch_t<__nv_bfloat16, 128, 1>(a, stream) : launch_t<float, 128, 1>(a, stream);
    return a.bf16 ? launch_t<__nv_bfloat16, 64, 1>(a, stream) : launch_t<float, 64, 1>(a, stream);
}

}  // namespace kda
