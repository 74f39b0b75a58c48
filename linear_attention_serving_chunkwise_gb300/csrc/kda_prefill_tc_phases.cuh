// Pieces shared by the tcgen05 chunkwise prefill kernels (the fused one-CTA-per-head
// kernel and the chunk-parallel / state-scan pair): shared- and tensor-memory maps of a
// chunk's operands, the kernel parameters, and the per-chunk phase functions (cumsum and
// decay factors, decayed operands, A/P read-out, the triangular solve, Tb and the seed of
// the [Wk; -Q'] accumulator), plus the host-side TMA descriptor helpers.  The method and
// the phase schedule are described at the top of kda_prefill_tc.cu.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"
#include "kda_launch.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

// ---------------------------------------------------------------- per-phase cycle marks
// Compile-time option KDA_PHASE_CLOCKS (off in the library build; phase_clocks.py builds a
// separate instrumented library with it): thread 0 of CTA 0 adds the clock64() cycles since
// its previous mark to slot `id` of its file's phase_clock_slots array, by a reduction that
// does not wait for the memory, and counts the items or chunks it ran in the two last slots.
#ifdef KDA_PHASE_CLOCKS
constexpr int kClockSlots = 32;
struct PhaseClock {
    long long prev;
    __device__ __forceinline__ void mark(unsigned long long* slots, int id)
    {
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            const long long now = clock64();
            atomicAdd(slots + id, (unsigned long long)(now - prev));
            prev = now;
        }
    }
    __device__ __forceinline__ void count(unsigned long long* slots, int id)
    {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicAdd(slots + id, 1ull);
    }
};
__device__ unsigned long long phase_clock_slots[kClockSlots];   // one array per translation unit
#define KDA_CLK_DECL(v) PhaseClock v{clock64()}
#define KDA_CLK(v, id) v.mark(phase_clock_slots, id)
#define KDA_CLK_COUNT(v, id) v.count(phase_clock_slots, id)
#else
#define KDA_CLK_DECL(v)
#define KDA_CLK(v, id)
#define KDA_CLK_COUNT(v, id)
#endif

constexpr int kThreads = 512;
constexpr uint64_t kWaitNs = 2000000000ull;   // bound on every on-device wait
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- shared memory map (bytes)
constexpr uint32_t OFF_Q = 0;          // q tile  [64 tok][128 ch] bf16, 2 x 8 KB TMA boxes
constexpr uint32_t OFF_K = 16384;      // k tile
constexpr uint32_t OFF_G = 32768;      // g tile  [64][128] fp32, 4 x 8 KB boxes; becomes x = e^{Gamma_r - rho_J}
constexpr uint32_t OFF_V0 = 65536;     // v tile, two buffers (B operand of [Tb; M] V)
constexpr uint32_t OFF_V1 = 81920;
constexpr uint32_t OFF_X = 98304;      // 80 KB region shared by phases 1-2 / 3 / 5
constexpr uint32_t X_SA = 0;           // A fp32 [64][68]; after the solve: Tb hi/lo bf16 B operands
constexpr uint32_t X_TBH = 0;          // Tb hi, MN-major B [64 i][64 j] bf16 (8 KB)
constexpr uint32_t X_TBL = 8192;       // Tb lo
constexpr uint32_t X_ST = 17408;       // T fp32 [64][68]
constexpr uint32_t X_SY = 34816;       // solve scratch fp32 [32][LDY]
constexpr uint32_t X_SB = 40960;       // S hi bf16, MN-major B [128 dk][128 dv] (phases 3-5b)
constexpr uint32_t X_SL = 0;           // S lo bf16, same layout (phases 4-5b; the W tiles take it over in 5c)
constexpr uint32_t X_WH = 0;           // W hi bf16, MN-major B [64 tok][128 dv] (phase 5)
constexpr uint32_t X_WL = 16384;       // W lo
constexpr uint32_t OFF_KG = 180224;    // K_Gamma bf16, MN-major B [64 tok][128 ch]
constexpr uint32_t OFF_VEC = 196608;   // per-channel vectors [19][128] fp32
constexpr uint32_t OFF_BETA = OFF_VEC + 19 * 512;
constexpr uint32_t OFF_BAR = OFF_BETA + 256;
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr size_t SMEM_BYTES = SMEM_USED + 1024;   // slack for 1024-byte alignment
constexpr int LDA = 68;    // fp32 row stride of A and T: 16-byte aligned rows
constexpr int LDY = 36;    // row stride of the solve scratch: 16-byte aligned rows

// fp32 column operand of the A/P MMA: one K-major tile of 160 rows (4 blocks of 32
// channels, block stride 160 * 128 bytes); reference m owns rows [8 m (m+1), 8 (m+1)(m+2)).
constexpr uint32_t KC_ROWS = 160;
__host__ __device__ constexpr uint32_t kc_row(int m) { return 8u * m * (m + 1); }

// per-channel vectors (index * 128 floats into OFF_VEC)
constexpr int V_E = 0;     // E_J = e^{rho_J}                                (4)
constexpr int V_G = 4;     // G_J = e^{Gamma_63 - rho_{J+1}}                 (4)
constexpr int V_D = 8;     // D_J = e^{rho_{J+1} - rho_J}                    (4)
constexpr int V_GC = 12;   // gamma_C = e^{Gamma_63}                         (1)
constexpr int V_DF = 13;   // e^{rho_m - rho_J}, J < m                       (6)

__host__ __device__ constexpr int f_index(int m, int J) { return m * (m - 1) / 2 + J; }

// ---------------------------------------------------------------- tensor memory map (columns)
constexpr uint32_t TM_S = 0;      // state S [128 dk lanes][128 dv] fp32
constexpr uint32_t TM_KQ = 128;   // [K_r; Q_r] tf32 A operand, one fp32 per column (phases 1-2)
constexpr uint32_t TM_PH = 128;   // [0; P] hi, bf16 pairs (phase 3)
constexpr uint32_t TM_PL = 160;   // [0; P] lo (phase 3)
constexpr uint32_t TM_M = 192;    // M = P Tb accumulator, rows 64-127, 64 columns (phase 3)
constexpr uint32_t TM_D1 = 128;   // [W; O] accumulator: [Tb; M] V from phase 4, + [-Wk; Q'] S in phase 5
constexpr uint32_t TM_AP = 256;   // A/P accumulators, sub-tile m at 256 + 16 m (m+1) / 2 (phases 2-3)
constexpr uint32_t TM_TPH = 256;  // [Tb; M] hi, bf16 pairs (phases 3-4)
constexpr uint32_t TM_TPL = 288;  // [Tb; M] lo (phases 3-4)
constexpr uint32_t TM_D2 = 320;   // [0; -Q_Gamma] seed, then [Wk; M K_Gamma - Q_Gamma] (phases 3-4)
constexpr uint32_t TM_A1 = 320;   // [-Wk; Q'] bf16 pairs, over the read D2 (phases 4-5b)
constexpr uint32_t TM_A1L = 384;  // [0; Q' - bf16(Q')] bf16 pairs, over the read D2 (phases 4-5b)
constexpr uint32_t TM_KTL = 448;  // K~^T lo (phases 2-5)
constexpr uint32_t TM_KT = 480;   // K~^T hi, lane = key channel, bf16 pairs (phases 2-5)
constexpr uint32_t TM_COLS = 512;

__host__ __device__ constexpr uint32_t tm_ap(int m) { return TM_AP + 8u * m * (m + 1); }

struct TcParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_g, tm_o;
    CUtensorMap tm_z;   // the output gate's logits, laid out as O (set when gate != nullptr)
    const float* beta;
    const int32_t* cu_seqlens;
    const float* init_state;
    float* out;
    float* final_state;
    float* checkpoints;
    int ckpt_interval, ckpt_slots;
    int num_seqs, total_tokens, num_heads;
    int* status;
    int prologue;   // KDA_PROLOGUE_* bits
    const float* gate;   // output gate logits [T, H, 128]: out = o * sigmoid(gate); nullptr = none
};

__device__ __forceinline__ float ex2f(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcpf(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// byte offset of g[r][c] in the fp32 tile (4 boxes of 32 channels, 128-byte swizzle)
__device__ __forceinline__ uint32_t g_off(int r, int c) { return sw128_off_f32(r, c, 64); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st8u(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void st_shared_v2(uint32_t saddr, uint32_t a, uint32_t b)
{
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(saddr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void st_shared_f4(uint32_t saddr, float a, float b, float c, float d)
{
    st_shared_v4(saddr, __float_as_uint(a), __float_as_uint(b), __float_as_uint(c), __float_as_uint(d));
}

__device__ __forceinline__ float ld_shared_f32(uint32_t saddr)
{
    float a;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(a) : "r"(saddr) : "memory");
    return a;
}

__device__ __forceinline__ void st_shared_f32(uint32_t saddr, float a)
{
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(saddr), "f"(a) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t saddr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(saddr));
    return v;
}

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t saddr)
{
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(saddr));
    return v;
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t saddr)
{
    const uint4 v = ld_shared_v4(saddr);
    return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
}

__device__ __forceinline__ float2 bf2_to_f2(uint32_t u)
{
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(h);
}

__device__ __forceinline__ void unpack8(const uint4 raw, float (&v)[8])
{
    const float2 a0 = bf2_to_f2(raw.x), a1 = bf2_to_f2(raw.y), a2 = bf2_to_f2(raw.z), a3 = bf2_to_f2(raw.w);
    v[0] = a0.x; v[1] = a0.y; v[2] = a1.x; v[3] = a1.y; v[4] = a2.x; v[5] = a2.y; v[6] = a3.x; v[7] = a3.y;
}

// fp32 -> the nearest tf32 value (ties away from zero), kept in fp32 storage.  The
// tensor core drops the low 13 mantissa bits of a tf32 operand; rounding first halves
// the operand error and removes its bias.
__device__ __forceinline__ float tf32_round(float x)
{
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi): the pair carries ~16 mantissa bits.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo)
{
    const float ah = __bfloat162float(__float2bfloat16_rn(a)), bh = __bfloat162float(__float2bfloat16_rn(b));
    hi = pack_bf16x2(ah, bh);
    lo = pack_bf16x2(a - ah, b - bh);
}

// Barrier over the first `n` threads of the CTA (named barrier `id`, n a multiple of 32).
__device__ __forceinline__ void named_sync(int id, int n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
constexpr int kSolveThreads = 256;   // warps 0-7 run the solve

// Every thread waits on `bar` (bounded); returns false for all threads if any gave up.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, int* s_abort)
{
    if (!mbar_wait_bounded(bar, parity, kWaitNs)) atomicExch(s_abort, 1);
    __syncthreads();
    return *s_abort == 0;
}

// v of a chunk into one of two buffers; completes on `bar` (16 KB).
__device__ __forceinline__ void issue_v_loads(const TcParams& p, uint8_t* sm, uint64_t* bar, int vbuf, int t0, int h)
{
    mbar_arrive_expect_tx(bar, 16384u);
    uint8_t* vb = sm + (vbuf ? OFF_V1 : OFF_V0);
    tma_load_3d(vb, &p.tm_v, bar, 0, h, t0);
    tma_load_3d(vb + 8192, &p.tm_v, bar, 64, h, t0);
}

// k of a chunk; completes on `bar` (16 KB).
__device__ __forceinline__ void issue_k_loads(const TcParams& p, uint8_t* sm, uint64_t* bar, int t0, int h)
{
    mbar_arrive_expect_tx(bar, 16384u);
    tma_load_3d(sm + OFF_K, &p.tm_k, bar, 0, h, t0);
    tma_load_3d(sm + OFF_K + 8192, &p.tm_k, bar, 64, h, t0);
}

// q and g of a chunk; completes on `bar` (48 KB).
__device__ __forceinline__ void issue_qg_loads(const TcParams& p, uint8_t* sm, uint64_t* bar, int t0, int h)
{
    mbar_arrive_expect_tx(bar, 49152u);
    tma_load_3d(sm + OFF_Q, &p.tm_q, bar, 0, h, t0);
    tma_load_3d(sm + OFF_Q + 8192, &p.tm_q, bar, 64, h, t0);
#pragma unroll
    for (int b = 0; b < 4; ++b) tma_load_3d(sm + OFF_G + 8192 * b, &p.tm_g, bar, 32 * b, h, t0);
}

// The output gate on an O row staged in shared memory: the row's 32 logits were loaded by
// TMA into the same positions of the same [64 tok][32] fp32 box (128-byte swizzle), so each
// value is read, multiplied by sigmoid(z) and stored back where the O value goes.
__device__ __forceinline__ void stage_gated_row(uint32_t box, int r, const float (&a)[32])
{
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint32_t at = box + sw128_off_f32(r, 4 * q, 64);
        const float4 z = ld_shared_f4(at);
        st_shared_f4(at, gate1(a[4 * q], z.x), gate1(a[4 * q + 1], z.y), gate1(a[4 * q + 2], z.z),
                     gate1(a[4 * q + 3], z.w));
    }
}

// ---------------------------------------------------------------- unit order
// The sequence a CTA of a one-CTA-per-unit launch takes: CTA b runs rank b / H of the
// sequences ordered longest first (ties by index), so that, as the CTAs of later waves start
// where earlier ones finish, no long sequence starts last (largest-first list scheduling).
// All threads of the CTA call it, before anything else uses `scratch` (N + 1 ints of shared
// memory).  Batches of more than kUnitOrderMaxSeqs sequences keep their order: ranking them
// would cost each CTA more than it saves.  Malformed cu_seqlens still give a permutation
// (the bounds check that follows reports them).
constexpr int kUnitOrderMaxSeqs = 256;
__device__ __noinline__ int unit_sequence(const int32_t* cu_seqlens, int num_seqs, int rank, int* scratch)
{
    if (cu_seqlens == nullptr || num_seqs <= 1 || num_seqs > kUnitOrderMaxSeqs) return rank;
    const int t = threadIdx.x;
    if (t < num_seqs) scratch[t] = __ldg(cu_seqlens + t + 1) - __ldg(cu_seqlens + t);
    __syncthreads();
    if (t < num_seqs) {
        const int mine = scratch[t];
        int r = 0;
        for (int j = 0; j < num_seqs; ++j) {
            const int other = scratch[j];
            r += (other > mine || (other == mine && j < t)) ? 1 : 0;
        }
        if (r == rank) scratch[kUnitOrderMaxSeqs] = t;
    }
    __syncthreads();
    const int n = scratch[kUnitOrderMaxSeqs];
    __syncthreads();   // the scratch is free again
    return n;
}

// ---------------------------------------------------------------- phase 1a: per-channel cumsum
// sigmoid(z_i) for the prologue's four decay logits with one reciprocal: d_i = 1 + e^{-z_i}
// and 1/d_0 = d_1 d_2 d_3 / (d_0 d_1 d_2 d_3), likewise for the others.  z is clamped below at
// -20, where sigmoid(z) < 2.1e-9 (a decay e^{-5 sigmoid(z)} within 1.1e-8 of 1 either way) and
// the product of four d_i stays below 5.5e34, a normal float with a normal reciprocal.  Each
// result is a few ulp of fp32 from the exact value.
__device__ __forceinline__ void sigmoid4(float (&z)[4])
{
    float d[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = 1.f + ex2f(-fmaxf(z[i], -20.f) * kLog2e);
    const float p01 = d[0] * d[1], p23 = d[2] * d[3];
    const float r = rcpf(p01 * p23);
    const float r01 = r * p23, r23 = r * p01;   // 1 / (d_0 d_1), 1 / (d_2 d_3)
    z[0] = d[1] * r01;
    z[1] = d[0] * r01;
    z[2] = d[3] * r23;
    z[3] = d[2] * r23;
}

// Thread (c = t % 128, J = t / 128) forms the sub-tile-local cumsum
// lambda_r = sum_{s = 16J}^{r} g_s log2(e) of sub-tile J of column c (rows past the chunk's
// end count as 0), replaces g_r in the tile by x_r = 2^{lambda_r} = e^{Gamma_r - rho_J}
// (in (0, 1], a normal float since g >= -5) and stores D_J = 2^{s_J}, the last x of the
// sub-tile (s_J: the sub-tile's sum).
// With the prologue's kProG bit the tile holds logits z and g = -5 sigmoid(z) is used
// (sigmoid4 on four rows at a time; the step adds sigmoid(z) (-5 log2(e)) in one rounding).
__device__ __forceinline__ void phase1_cumsum(uint8_t* sm, float* vec, int t, int BT, int prologue = 0)
{
    const int c = t & 127, J = t >> 7;
    const bool logits = (prologue & kProG) != 0;
    const float step = logits ? kGMin * kLog2e : kLog2e;
    float acc = 0.f, x = 1.f;
    // rows [16 J + 4 m, +4) of the column: g, or sigmoid(z); 0 past the chunk's end.  All 16
    // loads go first, so that their latencies overlap.
    float w[4][4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[m][i] = *reinterpret_cast<const float*>(sm + OFF_G + g_off(16 * J + 4 * m + i, c));
        if (logits) sigmoid4(w[m]);
#pragma unroll
        for (int i = 0; i < 4; ++i) w[m][i] = (16 * J + 4 * m + i < BT) ? w[m][i] : 0.f;
    }
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc = fmaf(w[m][i], step, acc);
            x = ex2f(acc);
            *reinterpret_cast<float*>(sm + OFF_G + g_off(16 * J + 4 * m + i, c)) = x;
        }
    vec[(V_D + J) * 128 + c] = x;
}

// The prologue's L2 normalisation of the q and k tiles in place (512 threads): thread t
// takes row t / 4 of [k; q] (token r = that row mod 64) and channels [32 (t % 4), +32), the
// row's sum of squares closing over the 4 neighbouring lanes; x / max(||x||, 1e-12) in fp32
// (x times the reciprocal norm) goes back as bf16.
__device__ __forceinline__ void phase0_normalise_qk(uint8_t* sm, int t)
{
    const int row = t >> 2, qtr = t & 3, r = row & 63;
    const uint32_t tile = smem_u32(sm) + (row < 64 ? OFF_K : OFF_Q);
    float x[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float v8[8];
        unpack8(ld_shared_v4(tile + sw128_chunk(r, 4 * qtr + i, 64)), v8);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[8 * i + e] = v8[e];
    }
    float s4[4] = {0.f, 0.f, 0.f, 0.f};   // four partial sums: a chain of 8 dependent FMAs, not 32
#pragma unroll
    for (int e = 0; e < 32; ++e) s4[e & 3] = fmaf(x[e], x[e], s4[e & 3]);
    float ss = (s4[0] + s4[1]) + (s4[2] + s4[3]);
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    const float inv = l2_inv(ss);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(x[8 * i + 2 * e] * inv, x[8 * i + 2 * e + 1] * inv);
        st_shared_v4(tile + sw128_chunk(r, 4 * qtr + i, 64), w[0], w[1], w[2], w[3]);
    }
}

// Per-channel factors (thread c < 128, after phase1_cumsum), all products of the four
// D_J = e^{rho_{J+1} - rho_J}: a product of factors <= 1 underflows only where the
// exponential of the summed exponent does.
__device__ __forceinline__ void phase1_factors(float* vec, int c)
{
    const float d0 = vec[(V_D + 0) * 128 + c], d1 = vec[(V_D + 1) * 128 + c], d2 = vec[(V_D + 2) * 128 + c],
                d3 = vec[(V_D + 3) * 128 + c];
    const float d01 = d0 * d1, d12 = d1 * d2, d23 = d2 * d3, d012 = d01 * d2, d123 = d1 * d23;
    vec[(V_E + 0) * 128 + c] = 1.f;
    vec[(V_E + 1) * 128 + c] = d0;
    vec[(V_E + 2) * 128 + c] = d01;
    vec[(V_E + 3) * 128 + c] = d012;
    vec[(V_G + 0) * 128 + c] = d123;
    vec[(V_G + 1) * 128 + c] = d23;
    vec[(V_G + 2) * 128 + c] = d3;
    vec[(V_G + 3) * 128 + c] = 1.f;
    vec[V_GC * 128 + c] = d012 * d3;
    vec[(V_DF + f_index(1, 0)) * 128 + c] = d0;
    vec[(V_DF + f_index(2, 0)) * 128 + c] = d01;
    vec[(V_DF + f_index(2, 1)) * 128 + c] = d1;
    vec[(V_DF + f_index(3, 0)) * 128 + c] = d012;
    vec[(V_DF + f_index(3, 1)) * 128 + c] = d12;
    vec[(V_DF + f_index(3, 2)) * 128 + c] = d2;
}

// ---------------------------------------------------------------- phase 1c: off-diagonal column rows
// For reference m and token i of an earlier sub-tile J < m, the column operand is
// k_i e^{rho_m - Gamma_i} = (k_i e^{rho_J - Gamma_i}) e^{rho_m - rho_J}: the stored
// diagonal-tile row of token i times a per-channel factor.  Thread t covers token offset
// i16 = t % 16 and channels [4 cq, 4 cq + 4), cq = t / 16, of all six (m, J) pairs (a
// warp: 16 tokens x 2 channel quads, so its factor loads are broadcasts); the row of each
// pair is a compile-time offset from the thread's own swizzled base.
__device__ __forceinline__ void phase1_offdiag(uint8_t* sm, const float* vec, int t)
{
    const int i16 = t & 15, cq = (t >> 4) & 31, c0 = 4 * cq;
    // sw128_off_f32(row, c0, KC_ROWS) with row % 8 == i16 % 8 for every row used below
    const uint32_t base = smem_u32(sm) + OFF_X + (cq >> 3) * (KC_ROWS * 128u) + i16 * 128u +
                          ((uint32_t)((cq & 7) ^ (i16 & 7)) << 4);
    // the rows read (diagonal tiles) and written (off-diagonal ones) are disjoint: all loads
    // first, so that their latencies overlap
    uint4 d[3];
    float4 f[6];
#pragma unroll
    for (int J = 0; J < 3; ++J) d[J] = ld_shared_v4(base + (kc_row(J) + 16 * J) * 128u);
#pragma unroll
    for (int b = 0; b < 6; ++b) f[b] = *reinterpret_cast<const float4*>(vec + (V_DF + b) * 128 + c0);
#pragma unroll
    for (int b = 0; b < 6; ++b) {
        const int m = (b == 0) ? 1 : ((b < 3) ? 2 : 3);
        const int J = b - m * (m - 1) / 2;
        st_shared_f4(base + (kc_row(m) + 16 * J) * 128u, tf32_round(__uint_as_float(d[J].x) * f[b].x),
                     tf32_round(__uint_as_float(d[J].y) * f[b].y), tf32_round(__uint_as_float(d[J].z) * f[b].z),
                     tf32_round(__uint_as_float(d[J].w) * f[b].w));
    }
}

// ---------------------------------------------------------------- phase 2 side work: K~^T into TMEM
// Lane c of the K~^T operand holds K~[r][c] = k[r][c] e^{Gamma_63 - Gamma_r}, two tokens
// per column, as a bf16 hi + lo pair; this thread covers sub-tile J = part (tokens
// [16 J, 16 J + 16)), where e^{Gamma_63 - Gamma_r} = d_J g_J / x_r.  ktilde_pairs forms the
// pairs (token 16 J + 2 pr in the low half of word pr), build_ktilde stores them to TMEM.
__device__ __forceinline__ void ktilde_pairs(uint8_t* sm, const float* vec, int c, int part, int BT, uint32_t (&hi)[8],
                                             uint32_t (&lo)[8])
{
    const uint32_t kbase = smem_u32(sm + OFF_K);
    const float fJ = vec[(V_D + part) * 128 + c] * vec[(V_G + part) * 128 + c];
#pragma unroll
    for (int pr = 0; pr < 8; ++pr) {
        float f2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = 16 * part + 2 * pr + e;
            const float x = *reinterpret_cast<const float*>(sm + OFF_G + g_off(r, c));
            unsigned short kb;
            asm volatile("ld.shared.u16 %0, [%1];" : "=h"(kb) : "r"(kbase + sw128_off(r, c, 64)));
            const float kv = (r < BT) ? __uint_as_float(((uint32_t)kb) << 16) : 0.f;
            f2[e] = kv * (fJ * rcpf(x));
        }
        split_bf16x2(f2[0], f2[1], hi[pr], lo[pr]);
    }
}

__device__ __forceinline__ void build_ktilde(uint8_t* sm, const float* vec, uint32_t tm, int c, int part, int quarter,
                                             int BT)
{
    uint32_t hi[8], lo[8];
    ktilde_pairs(sm, vec, c, part, BT, hi, lo);
    tmem_st8u(tmem_addr(tm, 32 * quarter, TM_KT + 8 * part), hi);
    tmem_st8u(tmem_addr(tm, 32 * quarter, TM_KTL + 8 * part), lo);
}

// ---------------------------------------------------------------- phase 3 side work: S operand
// Lane c, columns [32 part, 32 part + 32): S -> its bf16 rounding S_hi as an MN-major B
// operand.  The state is left as it is; state_lo_and_decay (phase 4) completes the split.
__device__ __forceinline__ void build_state_operand(uint8_t* sm, uint32_t tm, int c, int part, int quarter)
{
    const uint32_t sbase = smem_u32(sm);
    float a[32];
    tmem_ld32(tmem_addr(tm, 32 * quarter, TM_S + 32 * part), a);
    tmem_wait_ld();
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(a[2 * i], a[2 * i + 1]);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        st_shared_v4(sbase + OFF_X + X_SB + sw128_chunk(c, 4 * part + q, 128), pk[4 * q], pk[4 * q + 1],
                     pk[4 * q + 2], pk[4 * q + 3]);
}

// ---------------------------------------------------------------- phase 4 side work: S lo, decay
// Lane c, columns [32 part, 32 part + 32): S_lo = bf16(S - S_hi) as a second B operand of
// the same layout (the history read-out Q' S is formed as Q'_hi S_hi + Q'_hi S_lo +
// Q'_lo S_hi, so that its operands carry ~16 mantissa bits), then S <- gamma_C[c] S (the
// chunk decay, applied before the state update accumulates).
__device__ __forceinline__ void state_lo_and_decay(uint8_t* sm, float gc, uint32_t tm, int c, int part,
                                                   int quarter)
{
    const uint32_t sbase = smem_u32(sm);
    float a[32];
    tmem_ld32(tmem_addr(tm, 32 * quarter, TM_S + 32 * part), a);
    tmem_wait_ld();
    uint32_t hi[16], lo[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) split_bf16x2(a[2 * i], a[2 * i + 1], hi[i], lo[i]);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        st_shared_v4(sbase + OFF_X + X_SL + sw128_chunk(c, 4 * part + q, 128), lo[4 * q], lo[4 * q + 1],
                     lo[4 * q + 2], lo[4 * q + 3]);
#pragma unroll
    for (int i = 0; i < 32; ++i) a[i] *= gc;
    tmem_st32(tmem_addr(tm, 32 * quarter, TM_S + 32 * part), a);
}

// ---------------------------------------------------------------- phase 1b: token operands
// Thread (lane L, part p): token r = L % 64 of the q rows (L >= 64) or k rows (L < 64),
// channels [32p, 32p + 32).  Writes the tf32 row operand [K_r; Q_r] (TMEM).  Token r's
// diagonal-tile column operand is split between the k-row and the q-row thread (channels
// c0..c0+3 and c0+4..c0+7 of each group of 8), so that the two halves, which run on
// different SMSPs, carry the same number of reciprocals; its K_Gamma B operand is split
// the same way.
__device__ __forceinline__ void phase1_tokens(uint8_t* sm, const float* vec, uint32_t tm, int L, int part,
                                              int quarter, int BT, uint32_t kg_off = OFF_KG)
{
    const int r = L & 63, J = r >> 4;
    const bool isq = L >= 64;
    const bool valid = r < BT;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t src = sbase + (isq ? OFF_Q : OFF_K);
    const uint32_t kc = sbase + OFF_X;
    float kq[32];
#pragma unroll
    for (int gi = 0; gi < 4; ++gi) {
        const int c0 = 32 * part + 8 * gi;
        const uint4 raw = ld_shared_v4(src + sw128_chunk(r, c0 >> 3, 64));
        const uint4 la = ld_shared_v4(sbase + OFF_G + g_off(r, c0));
        const uint4 lb = ld_shared_v4(sbase + OFF_G + g_off(r, c0 + 4));
        float xv[8], xs[8];
        unpack8(raw, xv);
        xs[0] = __uint_as_float(la.x); xs[1] = __uint_as_float(la.y); xs[2] = __uint_as_float(la.z);
        xs[3] = __uint_as_float(la.w); xs[4] = __uint_as_float(lb.x); xs[5] = __uint_as_float(lb.y);
        xs[6] = __uint_as_float(lb.z); xs[7] = __uint_as_float(lb.w);   // e^{Gamma_r - rho_J} in (0, 1]
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            xv[e] = valid ? xv[e] : 0.f;
            kq[8 * gi + e] = tf32_round(xv[e] * xs[e]);
        }
        // diagonal-tile column operand of reference J, k_r e^{rho_J - Gamma_r} <= e^{80} |k_r|:
        // channels [c0, c0 + 4) from the k-row thread, [c0 + 4, c0 + 8) from the q-row thread
        // K_Gamma B operand: k_r e^{Gamma_r} = k_r x_r E_J (bf16)
        const uint32_t rj = kc_row(J) + r;
        const uint32_t kg = sbase + kg_off + sw128_chunk(r, c0 >> 3, 64);
        if (!isq) {   // xv holds k_r here
            st_shared_f4(kc + sw128_off_f32(rj, c0, KC_ROWS), tf32_round(xv[0] * rcpf(xs[0])),
                         tf32_round(xv[1] * rcpf(xs[1])), tf32_round(xv[2] * rcpf(xs[2])),
                         tf32_round(xv[3] * rcpf(xs[3])));
            const float4 e4 = *reinterpret_cast<const float4*>(vec + (V_E + J) * 128 + c0);
            st_shared_v2(kg, pack_bf16x2(xv[0] * xs[0] * e4.x, xv[1] * xs[1] * e4.y),
                         pack_bf16x2(xv[2] * xs[2] * e4.z, xv[3] * xs[3] * e4.w));
        } else {
            // channels c0 + 4 .. c0 + 7 of k_r: the upper half of the 16-byte chunk
            const uint2 k2 = ld_shared_v2(sbase + OFF_K + sw128_chunk(r, c0 >> 3, 64) + 8u);
            const float2 ka = bf2_to_f2(k2.x), kb = bf2_to_f2(k2.y);
            float kv[8];
            kv[4] = valid ? ka.x : 0.f;
            kv[5] = valid ? ka.y : 0.f;
            kv[6] = valid ? kb.x : 0.f;
            kv[7] = valid ? kb.y : 0.f;
            st_shared_f4(kc + sw128_off_f32(rj, c0 + 4, KC_ROWS), tf32_round(kv[4] * rcpf(xs[4])),
                         tf32_round(kv[5] * rcpf(xs[5])), tf32_round(kv[6] * rcpf(xs[6])),
                         tf32_round(kv[7] * rcpf(xs[7])));
            const float4 e4 = *reinterpret_cast<const float4*>(vec + (V_E + J) * 128 + c0 + 4);
            st_shared_v2(kg + 8u, pack_bf16x2(kv[4] * xs[4] * e4.x, kv[5] * xs[5] * e4.y),
                         pack_bf16x2(kv[6] * xs[6] * e4.z, kv[7] * xs[7] * e4.w));
        }
    }
    tmem_st32(tmem_addr(tm, 32 * quarter, TM_KQ + 32 * part), kq);
}

// ---------------------------------------------------------------- phase 3: A/P read-out
// Lane L, part p: columns [16p, 16p + 16) of row r = L % 64 of A (L < 64: scaled by
// beta_r, strictly lower) into shared memory in fp32, or of P (L >= 64: lower with
// diagonal) into TMEM as bf16 hi + lo pairs (the A operand of M = P Tb; lanes 0-63
// get zeros).
__device__ __forceinline__ void phase3_readout(uint8_t* sm, uint32_t tm, int L, int quarter, int part,
                                               const float* sbeta)
{
    const int r = L & 63, J = r >> 4;
    const bool isP = L >= 64;
    const uint32_t lane0 = 32 * quarter;
    const int j0 = 2 * (quarter & 1);   // the two sub-tiles of this warp's rows: j0, j0 + 1
    float va[16], vb[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) va[i] = vb[i] = 0.f;
    if (part <= j0) tmem_ld16(tmem_addr(tm, lane0, tm_ap(j0) + 16 * part), va);
    if (part <= j0 + 1) tmem_ld16(tmem_addr(tm, lane0, tm_ap(j0 + 1) + 16 * part), vb);
    tmem_wait_ld();
    float row[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) row[i] = (part <= J) ? ((J == j0) ? va[i] : vb[i]) : 0.f;
    uint32_t hi[8], lo[8];
    if (!isP) {
        const uint32_t arow = smem_u32(sm) + OFF_X + X_SA + 4u * (r * LDA + 16 * part);
        const float b = sbeta[r];
#pragma unroll
        for (int i = 0; i < 16; ++i) row[i] = (16 * part + i < r) ? b * row[i] : 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) st_shared_f4(arow + 16u * q, row[4 * q], row[4 * q + 1], row[4 * q + 2], row[4 * q + 3]);
#pragma unroll
        for (int i = 0; i < 8; ++i) hi[i] = lo[i] = 0u;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = 16 * part + 2 * i;
            split_bf16x2((c <= r) ? row[2 * i] : 0.f, (c + 1 <= r) ? row[2 * i + 1] : 0.f, hi[i], lo[i]);
        }
    }
    tmem_st8u(tmem_addr(tm, lane0, TM_PH + 8 * part), hi);
    tmem_st8u(tmem_addr(tm, lane0, TM_PL + 8 * part), lo);
}

// ---------------------------------------------------------------- phase 3: T = (I + A)^-1
// Threads 0..kSolveThreads-1 (warps 0-7, named barrier 1).  A is strictly lower triangular
// (beta folded in), so T is unit lower triangular.  Writes the blocks on and below the
// block diagonal of sT and zeros in blocks (0,1) and (2,3); nothing else is read.
//   1  the four 16x16 diagonal blocks by forward substitution (block m on warp m, one lane
//      per column), while warps 4-7 zero blocks (0,1) and (2,3);
//   2  the two 32x32 diagonal halves: T_{2b+1,2b} = -T_{2b+1,2b+1} A_{2b+1,2b} T_{2b,2b};
//   3  the lower half: T[32:64, 0:32] = -H1 A[32:64, 0:32] H0, with H0, H1 the halves.
__device__ __forceinline__ void phase3_solve(uint8_t* sm, int t)
{
    const float* sA = reinterpret_cast<const float*>(sm + OFF_X + X_SA);
    float* sT = reinterpret_cast<float*>(sm + OFF_X + X_ST);
    float* sY = reinterpret_cast<float*>(sm + OFF_X + X_SY);
    if (t < 128) {
        if ((t & 31) < 16) {
            const int m = t >> 5, j = t & 15, b = 16 * m;
            float x[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) x[q] = (q == j) ? 1.f : 0.f;
#pragma unroll
            for (int rr = 1; rr < 16; ++rr) {
                const float4* arow4 = reinterpret_cast<const float4*>(sA + (b + rr) * LDA + b);
                float av[16];
#pragma unroll
                for (int i4 = 0; i4 < 4; ++i4) {
                    if (4 * i4 < rr) {
                        const float4 v4 = arow4[i4];
                        av[4 * i4] = v4.x; av[4 * i4 + 1] = v4.y; av[4 * i4 + 2] = v4.z; av[4 * i4 + 3] = v4.w;
                    }
                }
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int i = 0; i < rr; ++i) {
                    if (i & 1) a1 = fmaf(-av[i], x[i], a1);
                    else a0 = fmaf(-av[i], x[i], a0);
                }
                if (rr > j) x[rr] = a0 + a1;
            }
#pragma unroll
            for (int q = 0; q < 16; ++q) sT[(b + q) * LDA + b + j] = x[q];
        }
    } else {
        const int u = t - 128, blk = u >> 6, row = (u >> 2) & 15, c4 = 4 * (u & 3);
        *reinterpret_cast<float4*>(sT + (32 * blk + row) * LDA + 32 * blk + 16 + c4) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    named_sync(1, kSolveThreads);
    {   // 2a: Y_b = A_{2b+1,2b} T_{2b,2b} (thread: half b, row i, columns j2, j2 + 1)
        const int b = t >> 7, i = (t >> 3) & 15, j2 = 2 * (t & 7);
        const int r0 = 32 * b + 16, c0 = 32 * b;
        const float* arow = sA + (r0 + i) * LDA + c0;
        const float* tcol = sT + c0 * LDA + c0 + j2;
        float2 acc = make_float2(0.f, 0.f), acc2 = acc;
#pragma unroll
        for (int q = 0; q < 16; q += 2) {
            const float a0 = arow[q], a1 = arow[q + 1];
            const float2 t0 = *reinterpret_cast<const float2*>(tcol + q * LDA);
            const float2 t1 = *reinterpret_cast<const float2*>(tcol + (q + 1) * LDA);
            acc.x = fmaf(a0, t0.x, acc.x); acc.y = fmaf(a0, t0.y, acc.y);
            acc2.x = fmaf(a1, t1.x, acc2.x); acc2.y = fmaf(a1, t1.y, acc2.y);
        }
        *reinterpret_cast<float2*>(sY + (16 * b + i) * LDY + j2) = make_float2(acc.x + acc2.x, acc.y + acc2.y);
    }
    named_sync(1, kSolveThreads);
    {   // 2b: T_{2b+1,2b} = -T_{2b+1,2b+1} Y_b
        const int b = t >> 7, i = (t >> 3) & 15, j2 = 2 * (t & 7);
        const int r0 = 32 * b + 16, c0 = 32 * b;
        const float* trow = sT + (r0 + i) * LDA + r0;
        const float* y = sY + 16 * b * LDY + j2;
        float2 acc = make_float2(0.f, 0.f), acc2 = acc;
#pragma unroll
        for (int q = 0; q < 16; q += 2) {
            const float a0 = trow[q], a1 = trow[q + 1];
            const float2 y0 = *reinterpret_cast<const float2*>(y + q * LDY);
            const float2 y1 = *reinterpret_cast<const float2*>(y + (q + 1) * LDY);
            acc.x = fmaf(a0, y0.x, acc.x); acc.y = fmaf(a0, y0.y, acc.y);
            acc2.x = fmaf(a1, y1.x, acc2.x); acc2.y = fmaf(a1, y1.y, acc2.y);
        }
        *reinterpret_cast<float2*>(sT + (r0 + i) * LDA + c0 + j2) = make_float2(-(acc.x + acc2.x), -(acc.y + acc2.y));
    }
    named_sync(1, kSolveThreads);
    // steps 3a/3b: a thread sums over one parity qh of the inner index and the two parities of
    // an output sit 16 lanes apart, summed with one shuffle.
    const int lane = t & 31, w = t >> 5;
    float acc[8];
    {   // 3a: Y = A[32:64, 0:32] H0.  Warp w takes columns [8 jg, 8 jg + 8) of rows
        // [16 (w / 4), +16) (lane % 16 the row).  H0 is lower triangular, so only the inner
        // indices k >= 8 jg contribute (the skipped terms are exact zeros): 16 - 4 jg pair
        // steps, with jg = w for warps 0-3 and 7 - w for warps 4-7, so that the two warps that
        // share an SM sub-partition (w and w + 4) take 20 steps between them.
        const int jg = w < 4 ? w : 7 - w, i = 16 * (w >> 2) + (lane & 15), qh = lane >> 4;
        const float* arow = sA + (32 + i) * LDA + qh;
        const float* hcol = sT + qh * LDA + 8 * jg;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (k < 4 * jg) continue;
            const float a = arow[2 * k];
            const float4 h0 = *reinterpret_cast<const float4*>(hcol + 2 * k * LDA);
            const float4 h1 = *reinterpret_cast<const float4*>(hcol + 2 * k * LDA + 4);
            acc[0] = fmaf(a, h0.x, acc[0]); acc[1] = fmaf(a, h0.y, acc[1]);
            acc[2] = fmaf(a, h0.z, acc[2]); acc[3] = fmaf(a, h0.w, acc[3]);
            acc[4] = fmaf(a, h1.x, acc[4]); acc[5] = fmaf(a, h1.y, acc[5]);
            acc[6] = fmaf(a, h1.z, acc[6]); acc[7] = fmaf(a, h1.w, acc[7]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 16);
        if (qh == 0) {
            *reinterpret_cast<float4*>(sY + i * LDY + 8 * jg) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            *reinterpret_cast<float4*>(sY + i * LDY + 8 * jg + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
    }
    named_sync(1, kSolveThreads);
    {   // 3b: T[32:64, 0:32] = -H1 Y.  Warp w takes rows [4 g, 4 g + 4) (columns [8 jg, +8),
        // jg = lane % 4).  H1 is lower triangular, so only k <= 4 g + 3 contribute (the skipped
        // terms are exact zeros): 2 g + 2 pair steps, with g = w for warps 0-3 and 11 - w for
        // warps 4-7, so that warps w and w + 4 take 18 steps between them.
        const int g = w < 4 ? w : 11 - w;
        const int jg = lane & 3, i = 4 * g + ((lane >> 2) & 3), qh = lane >> 4;
        const float* hrow = sT + (32 + i) * LDA + 32 + qh;
        const float* y = sY + qh * LDY + 8 * jg;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (k > 2 * g + 1) continue;
            const float a = hrow[2 * k];
            const float4 y0 = *reinterpret_cast<const float4*>(y + 2 * k * LDY);
            const float4 y1 = *reinterpret_cast<const float4*>(y + 2 * k * LDY + 4);
            acc[0] = fmaf(a, y0.x, acc[0]); acc[1] = fmaf(a, y0.y, acc[1]);
            acc[2] = fmaf(a, y0.z, acc[2]); acc[3] = fmaf(a, y0.w, acc[3]);
            acc[4] = fmaf(a, y1.x, acc[4]); acc[5] = fmaf(a, y1.y, acc[5]);
            acc[6] = fmaf(a, y1.z, acc[6]); acc[7] = fmaf(a, y1.w, acc[7]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 16);
        if (qh == 0) {
            *reinterpret_cast<float4*>(sT + (32 + i) * LDA + 8 * jg) = make_float4(-acc[0], -acc[1], -acc[2], -acc[3]);
            *reinterpret_cast<float4*>(sT + (32 + i) * LDA + 8 * jg + 4) =
                make_float4(-acc[4], -acc[5], -acc[6], -acc[7]);
        }
    }
}

// Tb = T diag(beta) as bf16 hi + lo MN-major B operands [64 i][64 j] (512 threads,
// one 8-column chunk each).  The solve writes only the blocks on and below the block
// diagonal; the chunks above it are zeros here.
__device__ __forceinline__ void phase3_tb_operands(uint8_t* sm, int t, const float* sbeta)
{
    const uint32_t sbase = smem_u32(sm);
    const int i = t >> 3, ch = t & 7;   // row i, 8-column chunk ch
    uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
    if ((ch >> 1) <= (i >> 4)) {
        const uint32_t trow = sbase + OFF_X + X_ST + 4u * (i * LDA + 8 * ch);
        const float4 t0 = ld_shared_f4(trow), t1 = ld_shared_f4(trow + 16u);
        const float4 b0 = *reinterpret_cast<const float4*>(sbeta + 8 * ch);
        const float4 b1 = *reinterpret_cast<const float4*>(sbeta + 8 * ch + 4);
        split_bf16x2(t0.x * b0.x, t0.y * b0.y, hi[0], lo[0]);
        split_bf16x2(t0.z * b0.z, t0.w * b0.w, hi[1], lo[1]);
        split_bf16x2(t1.x * b1.x, t1.y * b1.y, hi[2], lo[2]);
        split_bf16x2(t1.z * b1.z, t1.w * b1.w, hi[3], lo[3]);
    }
    st_shared_v4(sbase + OFF_X + X_TBH + sw128_chunk(i, ch, 64), hi[0], hi[1], hi[2], hi[3]);
    st_shared_v4(sbase + OFF_X + X_TBL + sw128_chunk(i, ch, 64), lo[0], lo[1], lo[2], lo[3]);
}

// 32 values of a row (as 16 packed bf16 pairs) -> chunks [4 chunk0, 4 chunk0 + 4) of row
// `row` of a 128-byte-swizzled bf16 tile with `rows` rows per 64-column block.
__device__ __forceinline__ void store_row32_bf16(uint32_t tile, int row, int chunk0, int rows, const uint32_t (&pk)[16])
{
#pragma unroll
    for (int q = 0; q < 4; ++q)
        st_shared_v4(tile + sw128_chunk(row, chunk0 + q, rows), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                     pk[4 * q + 3]);
}

// Seed of the [Wk; M K_Gamma] accumulator, columns [32p, 32p + 32): zeros in rows 0-63
// (lanes L < 64) and -Q_Gamma in rows 64-127 (token r = L - 64; rows past the chunk's end
// stay 0).  The MMA then adds [Tb; M] K_Gamma on top, so the strongly cancelling
// Q' = Q_Gamma - M K_Gamma is formed in fp32 and rounded to bf16 once.  The seed's
// columns are free from the A/P read-out on, so it is written during the solve.
__device__ __forceinline__ void phase3_seed(uint8_t* sm, const float* vec, uint32_t tm, int L, int p, int quarter,
                                            int BT)
{
    const int r = L - 64, J = (r >> 4) & 3;
    const bool valid = L >= 64 && r < BT;
    const uint32_t sbase = smem_u32(sm);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint32_t v[16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = 32 * p + 16 * half + 8 * h;
            if (valid) {
                float qv[8];
                unpack8(ld_shared_v4(sbase + OFF_Q + sw128_chunk(r, c >> 3, 64)), qv);
                const float4 xa = ld_shared_f4(sbase + OFF_G + g_off(r, c));
                const float4 xb = ld_shared_f4(sbase + OFF_G + g_off(r, c + 4));
                const float4 ea = *reinterpret_cast<const float4*>(vec + (V_E + J) * 128 + c);
                const float4 eb = *reinterpret_cast<const float4*>(vec + (V_E + J) * 128 + c + 4);
                v[8 * h + 0] = __float_as_uint(-(qv[0] * (xa.x * ea.x)));
                v[8 * h + 1] = __float_as_uint(-(qv[1] * (xa.y * ea.y)));
                v[8 * h + 2] = __float_as_uint(-(qv[2] * (xa.z * ea.z)));
                v[8 * h + 3] = __float_as_uint(-(qv[3] * (xa.w * ea.w)));
                v[8 * h + 4] = __float_as_uint(-(qv[4] * (xb.x * eb.x)));
                v[8 * h + 5] = __float_as_uint(-(qv[5] * (xb.y * eb.y)));
                v[8 * h + 6] = __float_as_uint(-(qv[6] * (xb.z * eb.z)));
                v[8 * h + 7] = __float_as_uint(-(qv[7] * (xb.w * eb.w)));
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[8 * h + e] = 0u;
            }
        }
        tmem_st16u(tmem_addr(tm, 32 * quarter, TM_D2 + 32 * p + 16 * half), v);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 3-D map over a [T][H][128] tensor: box = {box_c channels, 1 head, 64 tokens}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esz, int H, int T, int box_c)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)128 * esz, (cuuint64_t)H * 128 * esz};
    cuuint32_t box[3] = {(cuuint32_t)box_c, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace kda
