// Fused KDA decode: one token per sequence, one read and one write of each
// head's fp32 state (llm-atlas "K3_RESEARCH.md", Q07: decode keeps the O(1)
// state update; section 8, device layer: fused decode).
//
// With S' = Diag(exp g) S, one pass over S' yields both r = S'^T k and
// p = S'^T q.  Then w = beta (v - r), S_new = S' + k w^T, and the read-out
// S_new^T q = p + (k . q) w needs no second pass.  The state is held in
// registers between the read and the write, so HBM sees exactly 2 * dk * dv * 4
// bytes per (sequence, head) plus the small per-token vectors.
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

constexpr int kDecodeThreads = 256;

// kPro: the input prologue is compiled in (its own instance; the common one is unchanged).
template <typename Tin, int D, bool kPro>
__global__ void __launch_bounds__(kDecodeThreads, 2) kda_decode_kernel(DecodeArgs a)
{
    const int pro = kPro ? a.prologue : 0;
    constexpr int C4 = D / 4;                  // float4 columns per state row
    constexpr int RG = kDecodeThreads / C4;    // row groups
    constexpr int RP = D / RG;                 // rows per thread
    static_assert(RG * C4 == kDecodeThreads && RP * RG == D, "decode tiling");

    const size_t bh = blockIdx.x;              // b * H + h
    const int t = threadIdx.x;
    const int cg = t % C4, rg = t / C4;

    __shared__ float sk[D], sq[D], sdec[D], sv[D], sw[D];
    __shared__ float4 red_r[RG][C4], red_p[RG][C4];
    __shared__ float s_kq, s_beta;

    // Issue the state loads first: they are the only large stream.
    float* S = a.state + bh * D * D;
    float4 s[RP];
#pragma unroll
    for (int i = 0; i < RP; ++i) {
        const int row = rg * RP + i;
        s[i] = __ldcs(reinterpret_cast<const float4*>(S + (size_t)row * D) + cg);
    }

    const Tin* q = static_cast<const Tin*>(a.q) + bh * D;
    const Tin* k = static_cast<const Tin*>(a.k) + bh * D;
    const Tin* v = static_cast<const Tin*>(a.v) + bh * D;
    const float* g = a.g + bh * D;
    if (t < D) {
        sk[t] = to_f32(k[t]);
        sq[t] = to_f32(q[t]);
        sv[t] = to_f32(v[t]);
        sdec[t] = expf(g_of(g[t], pro));
    }
    if (t == 0) s_beta = beta_of(a.beta[bh], pro);
    __syncthreads();
    if (pro & kProQK) {   // warp 0 normalises k, warp 1 q
        if (t < 64) {
            float* x = t < 32 ? sk : sq;
            const int lane = t & 31;
            float ss = 0.f;
            for (int c = lane; c < D; c += 32) ss += x[c] * x[c];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float inv = l2_inv(ss);
            for (int c = lane; c < D; c += 32) x[c] = l2_scale(x[c], inv, Tin{});
        }
        __syncthreads();
    }
    if (t < 32) {
        float kq = 0.f;
        for (int c = t; c < D; c += 32) kq += sk[c] * sq[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
        if (t == 0) s_kq = kq;
    }

    float4 r = make_float4(0.f, 0.f, 0.f, 0.f), p = r;
#pragma unroll
    for (int i = 0; i < RP; ++i) {
        const int row = rg * RP + i;
        const float d = sdec[row], kc = sk[row], qc = sq[row];
        s[i].x *= d; s[i].y *= d; s[i].z *= d; s[i].w *= d;
        r.x += s[i].x * kc; r.y += s[i].y * kc; r.z += s[i].z * kc; r.w += s[i].w * kc;
        p.x += s[i].x * qc; p.y += s[i].y * qc; p.z += s[i].z * qc; p.w += s[i].w * qc;
    }
    red_r[rg][cg] = r;
    red_p[rg][cg] = p;
    __syncthreads();

    if (t < D) {
        const float* rr = reinterpret_cast<const float*>(&red_r[0][0]);
        const float* pp = reinterpret_cast<const float*>(&red_p[0][0]);
        float rs = 0.f, ps = 0.f;
#pragma unroll
        for (int gI = 0; gI < RG; ++gI) {
            rs += rr[gI * D + t];
            ps += pp[gI * D + t];
        }
        const float w = s_beta * (sv[t] - rs);
        sw[t] = w;
        const float o = ps + s_kq * w;
        a.out[bh * D + t] = a.gate ? gate1(o, __ldg(a.gate + bh * D + t)) : o;
    }
    __syncthreads();

    const float4 w4 = reinterpret_cast<const float4*>(sw)[cg];
#pragma unroll
    for (int i = 0; i < RP; ++i) {
        const int row = rg * RP + i;
        const float kc = sk[row];
        float4 o;
        o.x = s[i].x + kc * w4.x; o.y = s[i].y + kc * w4.y;
        o.z = s[i].z + kc * w4.z; o.w = s[i].w + kc * w4.w;
        __stcs(reinterpret_cast<float4*>(S + (size_t)row * D) + cg, o);
    }
}

template <typename Tin, int D>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t stream)
{
    const long long blocks = (long long)a.batch * a.num_heads;
    if (blocks == 0) return cudaSuccess;
    if (a.prologue)
        kda_decode_kernel<Tin, D, true><<<(unsigned)blocks, kDecodeThreads, 0, stream>>>(a);
    else
        kda_decode_kernel<Tin, D, false><<<(unsigned)blocks, kDecodeThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream)
{
    if (a.dk == 128) {
        return a.bf16 ? launch_decode_t<__nv_bfloat16, 128>(a, stream) : launch_decode_t<float, 128>(a, stream);
    }
    return a.bf16 ? launch_decode_t<__nv_bfloat16, 64>(a, stream) : launch_decode_t<float, 64>(a, stream);
}

}  // namespace kda
