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
// one column, so a step is three shuffle rounds and no CTA barrier.  The lane's columns
// are processed in pairs with the packed fp32x2 operations (one instruction, two IEEE
// results: the same roundings as two scalar ones, half the issue slots).  The K tokens'
// vectors are staged in shared memory once, behind the only barrier of the kernel.
// Outputs are written for every token; the state written back is the one after the
// first n_apply[b] tokens (0 leaves it untouched).
//
// Up to kPersistMaxTokens tokens a persistent variant runs instead: a grid of resident CTAs
// walks the (sequence, head) units, and while a CTA runs the K steps of one unit from
// registers, the next unit's state and raw token vectors stream into shared memory through
// cp.async (a hardware-tracked copy: its wait has no spin).  The state's HBM reads then
// overlap the arithmetic instead of alternating with it.  Longer drafts keep the per-unit
// kernel: their token staging would not leave room for two such CTAs per SM.
#include <algorithm>
#include <atomic>

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

__device__ __forceinline__ float2 splat(float x) { return make_float2(x, x); }
__device__ __forceinline__ float2 xor_sum(float2 x, int o)
{
    return __fadd2_rn(x, make_float2(__shfl_xor_sync(0xffffffffu, x.x, o), __shfl_xor_sync(0xffffffffu, x.y, o)));
}

// One token on the lane's R rows x 4 columns of the state, held as column pairs s[2 i]
// (columns 0, 1 of row i) and s[2 i + 1] (columns 2, 3).  kv, qv, dv point at the lane's
// first row of k, q and e^g in the staged token; v4 and beta are the token's values for
// the lane's columns.  Returns o for the lane's 4 columns (equal in all 8 lanes of a column).
template <int R>
__device__ __forceinline__ float4 token_step(float2 (&s)[2 * R], const float* kv, const float* qv, const float* dv,
                                             float4 v4, float beta)
{
    float2 r01 = make_float2(0.f, 0.f), r23 = r01, p01 = r01, p23 = r01;
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
            float2& lo = s[2 * (4 * i4 + e)];
            float2& hi = s[2 * (4 * i4 + e) + 1];
            lo = __fmul2_rn(lo, splat(dd[e]));                  // S' = Diag(e^g) S
            hi = __fmul2_rn(hi, splat(dd[e]));
            r01 = __ffma2_rn(lo, splat(kk[e]), r01);            // r = S'^T k
            r23 = __ffma2_rn(hi, splat(kk[e]), r23);
            p01 = __ffma2_rn(lo, splat(qq[e]), p01);            // p = S'^T q
            p23 = __ffma2_rn(hi, splat(qq[e]), p23);
            kq = fmaf(kk[e], qq[e], kq);
        }
    }
    // sums over the 8 lanes of each column (lane bits 2-4)
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        r01 = xor_sum(r01, o); r23 = xor_sum(r23, o);
        p01 = xor_sum(p01, o); p23 = xor_sum(p23, o);
        kq += __shfl_xor_sync(0xffffffffu, kq, o);
    }
    // w = beta (v - r)
    const float2 w01 = __fmul2_rn(splat(beta), __fadd2_rn(make_float2(v4.x, v4.y), make_float2(-r01.x, -r01.y)));
    const float2 w23 = __fmul2_rn(splat(beta), __fadd2_rn(make_float2(v4.z, v4.w), make_float2(-r23.x, -r23.y)));
#pragma unroll
    for (int i4 = 0; i4 < R / 4; ++i4) {                        // S <- S' + k w^T
        const float4 k4 = *reinterpret_cast<const float4*>(kv + 4 * i4);
        const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            s[2 * (4 * i4 + e)] = __ffma2_rn(splat(kk[e]), w01, s[2 * (4 * i4 + e)]);
            s[2 * (4 * i4 + e) + 1] = __ffma2_rn(splat(kk[e]), w23, s[2 * (4 * i4 + e) + 1]);
        }
    }
    const float2 o01 = __ffma2_rn(splat(kq), w01, p01), o23 = __ffma2_rn(splat(kq), w23, p23);   // o = p + (k.q) w
    return make_float4(o01.x, o01.y, o23.x, o23.y);
}

template <int R>
__device__ __forceinline__ void split4(float2 (&s)[2 * R], int i, float4 x)
{
    s[2 * i] = make_float2(x.x, x.y);
    s[2 * i + 1] = make_float2(x.z, x.w);
}

// The prologue's q/k L2 normalisation on the staged tokens (tokb: K tokens in
// MultiLayout<D>): warp w of the 2D / 32 takes vectors w, w + D / 16, ... of the 2K (k then
// q of each token).
template <typename Tin, int D>
__device__ __forceinline__ void normalise_tokens(float* tokb, int K, int w, int lane)
{
    using Lay = MultiLayout<D>;
    for (int vi = w; vi < 2 * K; vi += D / 16) {
        float* x = tokb + (vi >> 1) * Lay::kTok + (vi & 1) * Lay::kVec;
        float ss = 0.f;
        for (int c = lane; c < D; c += 32) ss += x[Lay::row(c)] * x[Lay::row(c)];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = l2_inv(ss);
        for (int c = lane; c < D; c += 32) x[Lay::row(c)] = l2_scale(x[Lay::row(c)], inv, Tin{});
    }
}

// kPro (both kernels): the input prologue is compiled in (own instances; the common ones
// are unchanged).
template <typename Tin, int D, bool kPro>
__global__ void __launch_bounds__(2 * D, 2) kda_decode_multi_kernel(DecodeMultiArgs a)
{
    const int pro = kPro ? a.prologue : 0;
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
    float2 s[2 * R];
#pragma unroll
    for (int i = 0; i < R; ++i) split4<R>(s, i, __ldcs(reinterpret_cast<const float4*>(S + (size_t)(r0 + i) * D)));

    // stage every token's vectors (plain loads, all issued before the one barrier)
    for (int idx = t; idx < K * D; idx += kThreads) {
        const int j = idx / D, c = idx - j * D;
        const size_t tok = ((size_t)b * K + j) * a.num_heads + h;   // [B, K, H, .]
        float* base = smv + j * Lay::kTok;
        base[Lay::row(c)] = to_f32(static_cast<const Tin*>(a.k)[tok * D + c]);
        base[Lay::kVec + Lay::row(c)] = to_f32(static_cast<const Tin*>(a.q)[tok * D + c]);
        base[2 * Lay::kVec + Lay::row(c)] = expf(g_of(a.g[tok * D + c], pro));
        base[3 * Lay::kVec + c] = to_f32(static_cast<const Tin*>(a.v)[tok * D + c]);
        if (c == 0) base[3 * Lay::kVec + D] = beta_of(a.beta[tok], pro);
    }
    __syncthreads();
    if (pro & kProQK) {
        normalise_tokens<Tin, D>(smv, K, t >> 5, lane);
        __syncthreads();
    }

    for (int j = 0; j < K; ++j) {
        const float* base = smv + j * Lay::kTok;
        const float* kv = base + Lay::row(r0);
        const float* qv = base + Lay::kVec + Lay::row(r0);
        const float* dv = base + 2 * Lay::kVec + Lay::row(r0);
        const float4 o4 = token_step<R>(s, kv, qv, dv, *reinterpret_cast<const float4*>(base + 3 * Lay::kVec + col),
                                        base[3 * Lay::kVec + D]);
        if (a.out && rs == 0) {
            const size_t tok = ((size_t)b * K + j) * a.num_heads + h;
            *reinterpret_cast<float4*>(a.out + tok * D + col) = a.gate ? gate4(o4, a.gate + tok * D + col) : o4;
        }
        if (j + 1 == n_apply) {   // the state after the applied prefix
#pragma unroll
            for (int i = 0; i < R; ++i) __stcs(reinterpret_cast<float4*>(S + (size_t)(r0 + i) * D),
                       make_float4(s[2 * i].x, s[2 * i].y, s[2 * i + 1].x, s[2 * i + 1].y));
        }
    }
}

// ---- persistent variant --------------------------------------------------------------

constexpr int kPersistMaxTokens = 8;

__device__ __forceinline__ void cp_async16(void* dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((unsigned)__cvta_generic_to_shared(dst)),
                 "l"(__cvta_generic_to_global(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((unsigned)__cvta_generic_to_shared(dst)),
                 "l"(__cvta_generic_to_global(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// shared memory of one CTA: the staged state, the converted tokens (MultiLayout), the raw
// tokens.  The state is stored in the 8 row groups the lanes own (R = D/8 rows each) with
// 16 floats of padding per group, so the two row groups one quarter-warp reads land in
// different bank halves.  A raw token is k, q, v (Tin), g (fp32), beta (fp32, padded to 16 B).
template <typename Tin, int D>
struct PersistLayout {
    static constexpr int R = D / 8;
    static constexpr int kGrp = R * D + 16;                                  // floats per row group
    static constexpr int kStateBytes = 8 * kGrp * 4;
    static constexpr int kVecChunks = D * (int)sizeof(Tin) / 16;             // 16-byte pieces of k, q or v
    static constexpr int kTokChunks = 3 * kVecChunks + D / 4;                // ... of k, q, v and g
    static constexpr int kRawTok = 16 * kTokChunks + 16;                     // bytes of one raw token
    static constexpr size_t smem(int K) { return kStateBytes + (size_t)K * MultiLayout<D>::kTok * 4 + (size_t)K * kRawTok; }
};

template <typename Tin, int D, bool kPro>
__global__ void __launch_bounds__(2 * D, 2) kda_decode_multi_persistent_kernel(DecodeMultiArgs a, int units)
{
    const int pro = kPro ? a.prologue : 0;
    using Lay = MultiLayout<D>;
    using PL = PersistLayout<Tin, D>;
    constexpr int R = D / 8;
    constexpr int kThreads = 2 * D;
    extern __shared__ __align__(16) float smv[];
    float* ss = smv;                                                         // staged state
    float* tokb = smv + PL::kStateBytes / 4;                                 // converted tokens
    unsigned char* raw = reinterpret_cast<unsigned char*>(tokb + a.tokens * Lay::kTok);

    const int H = a.num_heads, K = a.tokens;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int rs = lane >> 2, cq = lane & 3;
    const int col = 16 * w + 4 * cq;
    const int r0 = rs * R;

    // queue the copies of unit u's state and raw tokens into shared memory
    auto prefetch = [&](int u) {
        const float* src = a.state + (size_t)u * D * D;
        for (int c = t; c < D * D / 4; c += kThreads) {
            const int row = c / (D / 4), c4 = c - row * (D / 4);
            cp_async16(ss + (row / R) * PL::kGrp + (row % R) * D + 4 * c4, src + 4 * c);
        }
        const int b = u / H, h = u - b * H;
        for (int c = t; c < K * PL::kTokChunks; c += kThreads) {
            const int j = c / PL::kTokChunks, r = c - j * PL::kTokChunks;
            const size_t tok = ((size_t)b * K + j) * H + h;                  // [B, K, H, .]
            const unsigned char* s;
            if (r < PL::kVecChunks)
                s = static_cast<const unsigned char*>(a.k) + tok * D * sizeof(Tin) + 16 * r;
            else if (r < 2 * PL::kVecChunks)
                s = static_cast<const unsigned char*>(a.q) + tok * D * sizeof(Tin) + 16 * (r - PL::kVecChunks);
            else if (r < 3 * PL::kVecChunks)
                s = static_cast<const unsigned char*>(a.v) + tok * D * sizeof(Tin) + 16 * (r - 2 * PL::kVecChunks);
            else
                s = reinterpret_cast<const unsigned char*>(a.g + tok * D) + 16 * (r - 3 * PL::kVecChunks);
            cp_async16(raw + j * PL::kRawTok + 16 * r, s);
        }
        if (t < K) cp_async4(raw + t * PL::kRawTok + 16 * PL::kTokChunks, a.beta + ((size_t)b * K + t) * H + h);
        cp_async_commit();
    };

    int u = blockIdx.x;
    if (u >= units) return;
    prefetch(u);
    for (; u < units; u += gridDim.x) {
        const int b = u / H, h = u - b * H;
        int n_apply = K;
        if (a.n_apply) {
            n_apply = a.n_apply[b];
            if (n_apply < 0 || n_apply > K) {
                if (t == 0 && h == 0) report_status(a.status, kDevBadSeqlens);
                n_apply = 0;   // an invalid count leaves the state untouched
            }
        }
        cp_async_wait_all();
        __syncthreads();

        float2 s[2 * R];
#pragma unroll
        for (int i = 0; i < R; ++i) split4<R>(s, i, *reinterpret_cast<const float4*>(ss + rs * PL::kGrp + i * D + col));
        for (int idx = t; idx < K * D; idx += kThreads) {
            const int j = idx / D, c = idx - j * D;
            const unsigned char* rt = raw + j * PL::kRawTok;
            const Tin* rv = reinterpret_cast<const Tin*>(rt);
            float* base = tokb + j * Lay::kTok;
            base[Lay::row(c)] = to_f32(rv[c]);
            base[Lay::kVec + Lay::row(c)] = to_f32(rv[D + c]);
            base[2 * Lay::kVec + Lay::row(c)] =
                expf(g_of(reinterpret_cast<const float*>(rt + 3 * D * sizeof(Tin))[c], pro));
            base[3 * Lay::kVec + c] = to_f32(rv[2 * D + c]);
            if (c == 0) base[3 * Lay::kVec + D] = beta_of(*reinterpret_cast<const float*>(rt + 16 * PL::kTokChunks), pro);
        }
        __syncthreads();
        if (pro & kProQK) {
            normalise_tokens<Tin, D>(tokb, K, t >> 5, lane);
            __syncthreads();
        }
        if ((long long)u + gridDim.x < units) prefetch(u + gridDim.x);

        float* S = a.state + (size_t)u * D * D + col;
        for (int j = 0; j < K; ++j) {
            const float* base = tokb + j * Lay::kTok;
            const float* kv = base + Lay::row(r0);
            const float* qv = base + Lay::kVec + Lay::row(r0);
            const float* dv = base + 2 * Lay::kVec + Lay::row(r0);
            const float4 o4 = token_step<R>(s, kv, qv, dv, *reinterpret_cast<const float4*>(base + 3 * Lay::kVec + col),
                                            base[3 * Lay::kVec + D]);
            if (a.out && rs == 0) {
                const size_t tok = ((size_t)b * K + j) * H + h;
                *reinterpret_cast<float4*>(a.out + tok * D + col) = a.gate ? gate4(o4, a.gate + tok * D + col) : o4;
            }
            if (j + 1 == n_apply) {
#pragma unroll
                for (int i = 0; i < R; ++i) __stcs(reinterpret_cast<float4*>(S + (size_t)(r0 + i) * D),
                       make_float4(s[2 * i].x, s[2 * i].y, s[2 * i + 1].x, s[2 * i + 1].y));
            }
        }
    }
}

template <typename Tin, int D, bool kPro>
cudaError_t launch_t(const DecodeMultiArgs& a, cudaStream_t stream)
{
    const long long blocks = (long long)a.batch * a.num_heads;
    if (blocks == 0) return cudaSuccess;
    const size_t smem = (size_t)a.tokens * MultiLayout<D>::kTok * sizeof(float);
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kda_decode_multi_kernel<Tin, D, kPro>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kda_decode_multi_kernel<Tin, D, kPro><<<(unsigned)blocks, 2 * D, smem, stream>>>(a);
    return cudaGetLastError();
}

// resident CTAs per SM of one persistent variant at K tokens, and the device's SM count:
// found once per device (cached as value + 1, 0 = not yet known)
constexpr int kMaxDevices = 64;
constexpr int kVariants = 8;   // (dtype, dk, prologue)
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_resident[kMaxDevices][kVariants][kPersistMaxTokens + 1];

template <typename Tin, int D, bool kPro>
cudaError_t launch_persistent(const DecodeMultiArgs& a, int variant, cudaStream_t stream)
{
    const long long units = (long long)a.batch * a.num_heads;
    if (units == 0) return cudaSuccess;
    auto kern = kda_decode_multi_persistent_kernel<Tin, D, kPro>;
    const size_t smem = PersistLayout<Tin, D>::smem(a.tokens);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return launch_t<Tin, D, kPro>(a, stream);
    int sms = g_sm_count[dev].load(std::memory_order_relaxed) - 1;
    if (sms < 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_sm_count[dev].store(sms + 1, std::memory_order_relaxed);
    }
    std::atomic<int>& slot = g_resident[dev][variant][a.tokens];
    int per_sm = slot.load(std::memory_order_relaxed) - 1;
    if (per_sm < 0) {
        // the attribute covers the largest token count, so it is set once per device
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)PersistLayout<Tin, D>::smem(kPersistMaxTokens));
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 2 * D, smem);
        if (e != cudaSuccess) return e;
        slot.store(per_sm + 1, std::memory_order_relaxed);
    }
    if (per_sm < 1) return launch_t<Tin, D, kPro>(a, stream);
    const long long grid = std::min(units, (long long)sms * per_sm);
    kern<<<(unsigned)grid, 2 * D, smem, stream>>>(a, (int)units);
    return cudaGetLastError();
}

template <bool kPro>
cudaError_t launch_multi(const DecodeMultiArgs& a, cudaStream_t stream)
{
    constexpr int v0 = kPro ? 4 : 0;
    if (a.tokens <= kPersistMaxTokens) {
        if (a.dk == 128)
            return a.bf16 ? launch_persistent<__nv_bfloat16, 128, kPro>(a, v0, stream)
                          : launch_persistent<float, 128, kPro>(a, v0 + 1, stream);
        return a.bf16 ? launch_persistent<__nv_bfloat16, 64, kPro>(a, v0 + 2, stream)
                      : launch_persistent<float, 64, kPro>(a, v0 + 3, stream);
    }
    if (a.dk == 128)
        return a.bf16 ? launch_t<__nv_bfloat16, 128, kPro>(a, stream) : launch_t<float, 128, kPro>(a, stream);
    return a.bf16 ? launch_t<__nv_bfloat16, 64, kPro>(a, stream) : launch_t<float, 64, kPro>(a, stream);
}

}  // namespace

cudaError_t launch_decode_multi(const DecodeMultiArgs& a, cudaStream_t stream)
{
    return a.prologue ? launch_multi<true>(a, stream) : launch_multi<false>(a, stream);
}

}  // namespace kda
