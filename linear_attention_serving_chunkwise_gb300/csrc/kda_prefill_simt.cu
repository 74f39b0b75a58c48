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
// In A and P the decay between two tokens is a product of three bounded factors through
// 16-token sub-tile bases (g >= -5: each factor <= e^{80}); every other decay is one
// exponential of a difference of prefix sums, which is <= 0 because g <= 0.
//
// One CTA per (sequence, head, 32-column slice of dv): the columns of S evolve
// independently.  The slices of one (sequence, head) form a thread-block cluster and
// share the work that does not depend on the slice: each forms A and P over its own
// 32 key channels and solves for its own 32 columns of Wk, and the partial sums and the
// columns go to the other CTAs by stores into their shared memory.  fp32 throughout.
#include <cooperative_groups.h>

#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

constexpr int kChunk = 64;
constexpr int kSlice = 32;   // value columns per CTA
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kAld = kChunk + 4;  // row stride of P (16-byte aligned rows)
constexpr int kAt = kChunk + 4;   // row stride of A transposed (A^T[i][r]; 16-byte aligned rows)
constexpr int kCt = kChunk + 4;   // row stride of the transposed column operand of A and P (16-byte rows)
constexpr int kTiles = 136;       // 4 x 4 tiles on and below the diagonal of a 64 x 64 chunk

constexpr int kDq = kSlice;       // key channels (A and P) and columns of Wk per CTA of a cluster

template <int D>
constexpr size_t simt_smem_bytes()
{
    return sizeof(float) *
           (4 * kChunk * D + kChunk * kAt + kChunk * kAld + kChunk * kSlice + D * kSlice + kChunk + kDq * kCt + 7 * kDq);
}

// Four consecutive elements (16-byte aligned for fp32, 8-byte for bf16) as fp32.
__device__ __forceinline__ float4 load4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p)
{
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

template <typename Tin, int D>
__global__ void __cluster_dims__(1, 1, D / kSlice) __launch_bounds__(kThreads, 1) kda_prefill_simt_kernel(PrefillArgs a)
{
    extern __shared__ float smem[];
    float* sQ = smem;                  // [C][D]  q, then q * exp(Gamma)
    float* sK = sQ + kChunk * D;       // [C][D]  k, then k * exp(Gamma_n - Gamma)
    float* sG = sK + kChunk * D;       // [C][D]  g, then Gamma
    float* sKg = sG + kChunk * D;      // [C][D]  A/P row operand [C][kDq], then other CTAs' partial sums;
                                       //         then beta k exp(Gamma) (own columns), then Wk
    float* sA = sKg + kChunk * D;      // [C][kAt]  A transposed: sA[i * kAt + r] = A[r][i]
    float* sP = sA + kChunk * kAt;     // [C][kAld]
    float* sV = sP + kChunk * kAld;    // [C][kSlice]  beta v, then U, then W
    float* sS = sV + kChunk * kSlice;  // [D][kSlice]  state slice
    float* sB = sS + D * kSlice;       // [C] beta
    float* sCt = sB + kChunk;          // [kDq][kCt] k_i e^{rho_J' - Gamma_i} of this CTA's channels, transposed
    float* sF = sCt + kDq * kCt;       // [7][kDq]   e^{rho_J - rho_J'} per sub-tile pair J > J', then ones
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    constexpr int kNC = D / kSlice;    // CTAs in the cluster (the dv slices of this (sequence, head))
    const int cq = (int)cluster.block_rank(), cc0 = kDq * cq;   // this CTA's key channels [cc0, +kDq)

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
        // inputs four channels at a time, the loads of several rows in flight together
#pragma unroll 4
        for (int idx = 4 * t; idx < BT * D; idx += 4 * kThreads) {
            const int r = idx / D, c = idx % D;
            const size_t gi = ((size_t)(c0 + r) * H + h) * D + c;
            const float4 qv = load4(q + gi), kv = load4(k + gi), gv = load4(a.g + gi);
            *reinterpret_cast<float4*>(sQ + idx) = qv;
            *reinterpret_cast<float4*>(sK + idx) = kv;
            *reinterpret_cast<float4*>(sG + idx) =
                make_float4(g_of(gv.x, a.prologue), g_of(gv.y, a.prologue), g_of(gv.z, a.prologue), g_of(gv.w, a.prologue));
        }
        for (int idx = 4 * t; idx < BT * kSlice; idx += 4 * kThreads) {
            const int r = idx / kSlice, j = idx % kSlice;
            *reinterpret_cast<float4*>(sV + idx) = load4(v + ((size_t)(c0 + r) * H + h) * D + js + j);
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

        // A and P as register-tiled products over bounded per-token factors (g >= -5, llm-atlas
        // Q06's bounded decay).  For token r in 16-token sub-tile J, with base rho_J =
        // Gamma_{16J-1} (0 for J = 0) and J' the sub-tile of i <= r,
        //   e^{Gamma_r - Gamma_i} = e^{Gamma_r - rho_J} e^{rho_J - rho_J'} e^{rho_J' - Gamma_i},
        // factors <= 1, <= 1 and <= e^{80}.  Over this CTA's 32 key channels: the row operand
        // (k_r, then q_r, times the first factor) to sKg as [64][32] (free until the right-hand
        // sides below), the column operand k_i e^{rho_J' - Gamma_i} transposed to sCt, the
        // middle factors to sF; each of 136 threads sums one 4 x 4 tile of the lower triangle
        // over those channels, four at a time, A's partial sums into sA and then P's into sP.
        const auto rho_of = [&](int J, int c) { return J ? sG[(16 * J - 1) * D + c] : 0.f; };
        for (int idx = t; idx < kChunk * kDq; idx += kThreads) {
            const int r = idx / kDq, cl = idx % kDq, c = cc0 + cl;
            float rv = 0.f, cv = 0.f;
            if (r < BT) {
                const float rho = rho_of(r >> 4, c), gr = sG[r * D + c], kr = sK[r * D + c];
                rv = kr * expf(gr - rho);
                cv = kr * expf(rho - gr);
            }
            sKg[idx] = rv;
            sCt[cl * kCt + r] = cv;
        }
        for (int idx = t; idx < 7 * kDq; idx += kThreads) {
            const int pr = idx / kDq, c = cc0 + idx % kDq;   // pairs (1,0) (2,0) (2,1) (3,0) (3,1) (3,2), then ones
            const int J = pr < 1 ? 1 : (pr < 3 ? 2 : 3), Jp = pr - J * (J - 1) / 2;
            sF[idx] = pr == 6 ? 1.f : (16 * J - 1 < BT ? expf(rho_of(J, c) - rho_of(Jp, c)) : 0.f);
        }
        __syncthreads();
        int rb = 0;   // this thread's tile: rows [4 rb, +4), columns [4 ib, +4), ib <= rb
        while ((rb + 1) * (rb + 2) / 2 <= t) ++rb;
        const int ib = t - rb * (rb + 1) / 2;
        for (int pass = 0; pass < 2; ++pass) {
            if (pass == 1) {   // the row operand of P, over that of A
                __syncthreads();
                for (int idx = t; idx < kChunk * kDq; idx += kThreads) {
                    const int r = idx / kDq, c = cc0 + idx % kDq;
                    sKg[idx] = r < BT ? sQ[r * D + c] * expf(sG[r * D + c] - rho_of(r >> 4, c)) : 0.f;
                }
                __syncthreads();
            }
            if (t < kTiles) {
                const int Jr = rb >> 2, Ji = ib >> 2;
                const float* fr = sF + (Jr == Ji ? 6 : Jr * (Jr - 1) / 2 + Ji) * kDq;
                float acc[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
                // the channel order starts at 4 rb, so that row blocks read different banks
                for (int kx = 0; kx < kDq; kx += 4) {
                    const int c = (4 * rb + kx) & (kDq - 1);
                    const float4 f4 = *reinterpret_cast<const float4*>(fr + c);
                    float4 r4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) r4[i] = *reinterpret_cast<const float4*>(sKg + (4 * rb + i) * kDq + c);
                    const float fu[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float4 c4 = *reinterpret_cast<const float4*>(sCt + (c + u) * kCt + 4 * ib);
                        const float cv[4] = {c4.x * fu[u], c4.y * fu[u], c4.z * fu[u], c4.w * fu[u]};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float rv = u == 0 ? r4[i].x : u == 1 ? r4[i].y : u == 2 ? r4[i].z : r4[i].w;
#pragma unroll
                            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(rv, cv[j], acc[i][j]);
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 4 * rb + i;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int col = 4 * ib + j;
                        if (col <= r && r < BT) {
                            if (pass == 0) sA[col * kAt + r] = acc[i][j];
                            else sP[r * kAld + col] = acc[i][j];
                        }
                    }
                }
            }
        }
        // the partial sums of the cluster's CTAs, summed in rank order by the CTA that owns the
        // rows ([64 / kNC rank, +64 / kNC)).  Every exchange is a store into another CTA's
        // shared memory: the partial sums of the others' rows go to slots in their sKg (free
        // from the end of the tiles to the right-hand sides), the owner sums, and the sums go
        // to every CTA's sA and sP (where each CTA reads only the rows it owns meanwhile).
        {
            constexpr int kRows = kChunk / kNC, kPer = kRows * kChunk / kThreads;
            // partial sums of sender s in receiver q's sKg: slot s - (s > q), A then P, [kRows][64]
            const auto slot = [&](int s, int q, int ap) { return ((s - (s > q)) * 2 + ap) * kRows * kChunk; };
            static_assert((kNC - 1) * 2 * kRows * kChunk <= kChunk * D, "partial-sum slots fit in sKg");
            cluster.sync();   // every CTA's tiles are done: their sKg is free
            for (int qo = 1; qo < kNC; ++qo) {
                const int q = (cq + qo) % kNC;
                float* dst = cluster.map_shared_rank(sKg, q);
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    const int e = t + kThreads * k, r = kRows * q + e / kChunk, col = e % kChunk;
                    if (r < BT && col <= r) {
                        dst[slot(cq, q, 0) + e] = sA[col * kAt + r];
                        dst[slot(cq, q, 1) + e] = sP[r * kAld + col];
                    }
                }
            }
            cluster.sync();   // every partial sum is delivered
            float va[kPer], vp[kPer];
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int e = t + kThreads * k, r = kRows * cq + e / kChunk, col = e % kChunk;
                float sa = 0.f, sp = 0.f;
                if (r < BT && col <= r) {
#pragma unroll
                    for (int s = 0; s < kNC; ++s) {
                        sa += s == cq ? sA[col * kAt + r] : sKg[slot(s, cq, 0) + e];
                        sp += s == cq ? sP[r * kAld + col] : sKg[slot(s, cq, 1) + e];
                    }
                }
                va[k] = (col < r) ? sB[r] * sa : 0.f;
                vp[k] = sp;
            }
#pragma unroll
            for (int q = 0; q < kNC; ++q) {
                float* qa = cluster.map_shared_rank(sA, q);
                float* qp = cluster.map_shared_rank(sP, q);
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    const int e = t + kThreads * k, r = kRows * cq + e / kChunk, col = e % kChunk;
                    if (r < BT && col <= r) {
                        qa[col * kAt + r] = va[k];
                        qp[r * kAld + col] = vp[k];
                    }
                }
            }
            cluster.sync();   // A and P complete in every CTA; every slot read
        }
        // right-hand sides diag(beta) [V | K exp(Gamma)], K's over this CTA's columns of Wk
        for (int idx = t; idx < BT * kDq; idx += kThreads) {
            const int r = idx / kDq, c = cc0 + idx % kDq;
            sKg[r * D + c] = sB[r] * sK[r * D + c] * expf(sG[r * D + c]);
        }
        for (int idx = t; idx < BT * kSlice; idx += kThreads) sV[idx] *= sB[idx / kSlice];
        __syncthreads();

        // (I + A) X = RHS by forward substitution, one column per thread: U's 32 and this
        // CTA's 32 of Wk
        for (int col = t; col < kSlice + kDq; col += kThreads) {
            float* X = (col < kSlice) ? (sV + col) : (sKg + cc0 + (col - kSlice));
            const int ld = (col < kSlice) ? kSlice : D;
            // sixteen rows (one sub-tile) at a time: each solved value X[i] meets the block's
            // A[r][i] in four float4 of A^T, then the block's own lower triangle in registers
            // (rows past the chunk's end are formed from whatever they hold and never stored)
            for (int r0 = 0; r0 < BT; r0 += 16) {
                float x[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) x[j] = (r0 + j < BT) ? X[(r0 + j) * ld] : 0.f;
                for (int i = 0; i < r0; ++i) {
                    const float xi = X[i * ld];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const float4 a4 = *reinterpret_cast<const float4*>(sA + i * kAt + r0 + 4 * q4);
                        x[4 * q4] -= a4.x * xi;
                        x[4 * q4 + 1] -= a4.y * xi;
                        x[4 * q4 + 2] -= a4.z * xi;
                        x[4 * q4 + 3] -= a4.w * xi;
                    }
                }
#pragma unroll
                for (int j = 1; j < 16; ++j)
#pragma unroll
                    for (int jj = 0; jj < j; ++jj) x[j] -= sA[(r0 + jj) * kAt + r0 + j] * x[jj];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (r0 + j < BT) X[(r0 + j) * ld] = x[j];
            }
        }
        // this CTA's columns of Wk into the other CTAs' sKg (each solves only its own columns there)
        __syncthreads();
        for (int qo = 1; qo < kNC; ++qo) {
            float* dst = cluster.map_shared_rank(sKg, (cq + qo) % kNC);
            for (int i4 = t; i4 < BT * kDq / 4; i4 += kThreads) {
                const int o = (i4 / (kDq / 4)) * D + cc0 + 4 * (i4 % (kDq / 4));
                *reinterpret_cast<float4*>(dst + o) = *reinterpret_cast<const float4*>(sKg + o);
            }
        }
        cluster.sync();   // every CTA holds all of Wk

        // decayed operands in place; W = U - Wk S (in place in sV).  In the three products
        // below, warp w takes 8 consecutive rows (or D / 8 consecutive state rows) at once,
        // so that each value of S, W or V it loads serves all of them, and reads the other
        // operand's rows four channels at a time (each sum still runs in its own order).
        const float* gl = sG + (BT - 1) * D;
        for (int idx = t; idx < BT * D; idx += kThreads) {
            const int c = idx % D;
            const float e = sG[idx];
            sQ[idx] *= expf(e);
            sK[idx] *= expf(gl[c] - e);
        }
        const int r8 = 8 * warp;   // this warp's rows [r8, r8 + 8)
        {
            float acc[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) acc[m] = sV[(r8 + m) * kSlice + lane];
            for (int c = 0; c < D; c += 4) {
                float s4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) s4[u] = sS[(c + u) * kSlice + lane];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float4 w4 = *reinterpret_cast<const float4*>(sKg + (r8 + m) * D + c);
                    acc[m] = fmaf(-w4.x, s4[0], acc[m]);
                    acc[m] = fmaf(-w4.y, s4[1], acc[m]);
                    acc[m] = fmaf(-w4.z, s4[2], acc[m]);
                    acc[m] = fmaf(-w4.w, s4[3], acc[m]);
                }
            }
#pragma unroll
            for (int m = 0; m < 8; ++m)
                if (r8 + m < BT) sV[(r8 + m) * kSlice + lane] = acc[m];
        }
        __syncthreads();

        // O = Q_Gamma S + P W, written in fp32
        {
            float acc[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) acc[m] = 0.f;
            for (int c = 0; c < D; c += 4) {
                float s4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) s4[u] = sS[(c + u) * kSlice + lane];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float4 q4 = *reinterpret_cast<const float4*>(sQ + (r8 + m) * D + c);
                    acc[m] = fmaf(q4.x, s4[0], acc[m]);
                    acc[m] = fmaf(q4.y, s4[1], acc[m]);
                    acc[m] = fmaf(q4.z, s4[2], acc[m]);
                    acc[m] = fmaf(q4.w, s4[3], acc[m]);
                }
            }
            for (int i = 0; i < r8; i += 4) {   // tokens before the warp's rows: every row takes them
                float v4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) v4[u] = sV[(i + u) * kSlice + lane];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float4 p4 = *reinterpret_cast<const float4*>(sP + (r8 + m) * kAld + i);
                    acc[m] = fmaf(p4.x, v4[0], acc[m]);
                    acc[m] = fmaf(p4.y, v4[1], acc[m]);
                    acc[m] = fmaf(p4.z, v4[2], acc[m]);
                    acc[m] = fmaf(p4.w, v4[3], acc[m]);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {   // the warp's own tokens: row r8 + m takes i <= r8 + m
                const float v = sV[(r8 + u) * kSlice + lane];
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    if (u <= m) acc[m] = fmaf(sP[(r8 + m) * kAld + r8 + u], v, acc[m]);
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                if (r8 + m < BT) {
                    const size_t oi = ((size_t)(c0 + r8 + m) * H + h) * D + js + lane;
                    a.out[oi] = a.gate ? gate1(acc[m], __ldg(a.gate + oi)) : acc[m];
                }
            }
        }
        // S <- Diag(exp Gamma_n) S + K~^T W: warp w takes state rows [D/8 w, +D/8)
        constexpr int kRows = D / kWarps;
        const int cw = kRows * warp;
        float snew[kRows];
#pragma unroll
        for (int m = 0; m < kRows; ++m) snew[m] = expf(gl[cw + m]) * sS[(cw + m) * kSlice + lane];
        for (int r = 0; r < BT; ++r) {
            const float v = sV[r * kSlice + lane];
#pragma unroll
            for (int m4 = 0; m4 < kRows; m4 += 4) {
                const float4 k4 = *reinterpret_cast<const float4*>(sK + r * D + cw + m4);
                snew[m4] = fmaf(k4.x, v, snew[m4]);
                snew[m4 + 1] = fmaf(k4.y, v, snew[m4 + 1]);
                snew[m4 + 2] = fmaf(k4.z, v, snew[m4 + 2]);
                snew[m4 + 3] = fmaf(k4.w, v, snew[m4 + 3]);
            }
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < kRows; ++m) sS[(cw + m) * kSlice + lane] = snew[m];
        // state snapshot after a full chunk that ends on a checkpoint boundary
        const int done = c0 + BT - bos;
        if (a.checkpoints && BT == kChunk && done % a.ckpt_interval == 0 && done / a.ckpt_interval <= a.ckpt_slots) {
            const int slot = done / a.ckpt_interval - 1;
            float* dst = a.checkpoints + (((size_t)n * H + h) * a.ckpt_slots + slot) * D * D;
#pragma unroll
            for (int m = 0; m < kRows; ++m) dst[(size_t)(cw + m) * D + js + lane] = snew[m];
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
