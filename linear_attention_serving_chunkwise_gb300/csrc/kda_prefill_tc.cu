// Chunkwise KDA prefill on the Blackwell tensor cores (tcgen05), bf16 q/k/v,
// dk = dv = 128, 64-token chunks cut into four 16-token sub-tiles.
//
// Method (llm-atlas "K3_RESEARCH.md": Q04/Q05 recurrence and delta-rule write,
// Q06 + Figure 3 bounded log-decay g >= -5 so the diagonal tile can use the
// tensor cores, Q07 chunkwise form with the state passed between chunks; agihunt
// digest: FlashKDA's 16-token tiles).  For a chunk entered with state S and
// Gamma_r the inclusive prefix sum of g over the chunk (per key channel):
//   A[r][i] = beta_r <k_r e^{Gamma_r - Gamma_i}, k_i>  (i < r),   P[r][i] = <q_r e^{Gamma_r - Gamma_i}, k_i>  (i <= r)
//   Tb = (I + A)^-1 diag(beta),   M = P Tb,   Wk = Tb K_Gamma,   Q' = Q_Gamma - M K_Gamma
//   W = Tb V - Wk S,   O = Q' S + M V,   S <- Diag(e^{Gamma_63}) S + (K e^{Gamma_63 - Gamma})^T W
// (O = Q_Gamma S + P W rewritten so that the read-out needs no product with W.)
//
// Intra-chunk decays are split at sub-tile boundaries so that every operand
// factor is finite: for row r in sub-tile J with base rho_J (Gamma just before the
// sub-tile), e^{Gamma_r - Gamma_i} = e^{Gamma_r - rho_J} e^{rho_J - Gamma_i}; the
// row factor is <= 1 and the column factor is <= e^{5*16} on the diagonal tile
// and <= 1 off it.
//
// Precision: A and P use tf32 MMAs (operands rounded to nearest tf32 first, since
// the tensor core truncates); Tb, M and W enter their MMAs as bf16 hi + lo pairs, and
// so does K~ in the state update; S, Wk, Q' and K_Gamma are single bf16 (Q' rounded
// once, after its fp32 subtraction); accumulation and the carried state are fp32.
//
// One CTA owns one (sequence, head) and walks its chunks in order; the fp32 state
// lives in tensor memory for the whole sequence.  Per chunk:
//   1  g cumsum per channel; decayed operands to TMEM (A operands) and shared
//      memory (B operands); TMA prefetch of the next chunk's v.
//   2  A and P by one tf32 MMA over the four sub-tile references side by side, while
//      all warps build K~^T (TMEM).
//   3  T = (I + A)^-1 in fp32 on CUDA cores (8 warps) while the other 8 build the
//      state's bf16 B operand, apply the chunk decay to S and seed the next
//      accumulator with [0; -Q_Gamma]; M = P Tb by three bf16 MMAs (hi/lo splits);
//      TMA prefetch of the next chunk's k.
//   4  [Wk; -Q'] by MMA onto the seed, and the state-independent half of D1,
//      [Tb; M] V, queued behind it; then the [-Wk; Q'] operand over the read
//      accumulator; TMA prefetch of the next chunk's q and g.
//   5  D1 += [-Wk; Q'] S by MMA: rows 0-63 are W, rows 64-127 are O; W to shared
//      memory; S += K~^T W by MMA while O is staged in shared memory and written by
//      TMA bulk stores (direct stores for a sequence's ragged last chunk).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"
#include "kda_launch.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

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
constexpr uint32_t X_OST = 65536;      // O staging, dv columns 0-63: 2 x [64 tok][32] fp32 boxes (phase 5,
                                       // after the MMA that reads S bf16 has completed)
constexpr uint32_t X_SB = 40960;       // S bf16, MN-major B [128 dk][128 dv] (phases 3-5b)
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
constexpr uint32_t TM_KTL = 448;  // K~^T lo (phases 2-5)
constexpr uint32_t TM_KT = 480;   // K~^T hi, lane = key channel, bf16 pairs (phases 2-5)
constexpr uint32_t TM_COLS = 512;

__host__ __device__ constexpr uint32_t tm_ap(int m) { return TM_AP + 8u * m * (m + 1); }

struct TcParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_g, tm_o;
    const float* beta;
    const int32_t* cu_seqlens;
    const float* init_state;
    float* out;
    float* final_state;
    float* checkpoints;
    int ckpt_interval, ckpt_slots;
    int num_seqs, total_tokens, num_heads;
    int* status;
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

__device__ __forceinline__ void st_shared_f4(uint32_t saddr, float a, float b, float c, float d)
{
    st_shared_v4(saddr, __float_as_uint(a), __float_as_uint(b), __float_as_uint(c), __float_as_uint(d));
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t saddr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(saddr));
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

// ---------------------------------------------------------------- phase 1a: per-channel cumsum
// Thread (c = t % 128, J = t / 128) forms the sub-tile-local cumsum
// lambda_r = sum_{s = 16J}^{r} g_s log2(e) of sub-tile J of column c (rows past the chunk's
// end count as 0), replaces g_r in the tile by x_r = 2^{lambda_r} = e^{Gamma_r - rho_J}
// (in (0, 1], a normal float since g >= -5) and stores D_J = 2^{s_J}, the last x of the
// sub-tile (s_J: the sub-tile's sum).
__device__ __forceinline__ void phase1_cumsum(uint8_t* sm, float* vec, int t, int BT)
{
    const int c = t & 127, J = t >> 7;
    float acc = 0.f, x = 1.f;
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
        const int r = 16 * J + rr;
        float* gp = reinterpret_cast<float*>(sm + OFF_G + g_off(r, c));
        const float gv = (r < BT) ? *gp : 0.f;
        acc = fmaf(gv, kLog2e, acc);
        x = ex2f(acc);
        *gp = x;
    }
    vec[(V_D + J) * 128 + c] = x;
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
#pragma unroll
    for (int b = 0; b < 6; ++b) {
        const int m = (b == 0) ? 1 : ((b < 3) ? 2 : 3);
        const int J = b - m * (m - 1) / 2;
        const uint4 d = ld_shared_v4(base + (kc_row(J) + 16 * J) * 128u);
        const float4 f = *reinterpret_cast<const float4*>(vec + (V_DF + b) * 128 + c0);
        st_shared_f4(base + (kc_row(m) + 16 * J) * 128u, tf32_round(__uint_as_float(d.x) * f.x),
                     tf32_round(__uint_as_float(d.y) * f.y), tf32_round(__uint_as_float(d.z) * f.z),
                     tf32_round(__uint_as_float(d.w) * f.w));
    }
}

// ---------------------------------------------------------------- phase 2 side work: K~^T into TMEM
// Lane c of the K~^T operand holds K~[r][c] = k[r][c] e^{Gamma_63 - Gamma_r}, two tokens
// per column, as a bf16 hi + lo pair; this thread covers sub-tile J = part (tokens
// [16 J, 16 J + 16)), where e^{Gamma_63 - Gamma_r} = d_J g_J / x_r.
__device__ __forceinline__ void build_ktilde(uint8_t* sm, const float* vec, uint32_t tm, int c, int part, int quarter,
                                             int BT)
{
    uint32_t hi[8], lo[8];
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
    tmem_st8u(tmem_addr(tm, 32 * quarter, TM_KT + 8 * part), hi);
    tmem_st8u(tmem_addr(tm, 32 * quarter, TM_KTL + 8 * part), lo);
}

// ---------------------------------------------------------------- phase 3 side work: S operand
// Lane c, columns [32 part, 32 part + 32): S -> bf16 MN-major B operand, then
// S <- gamma_C[c] S (the chunk decay, applied before the state update accumulates).
__device__ __forceinline__ void build_state_operand(uint8_t* sm, const float* vec, uint32_t tm, int c, int part,
                                                    int quarter)
{
    const uint32_t sbase = smem_u32(sm);
    const float gc = vec[V_GC * 128 + c];
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
#pragma unroll
    for (int i = 0; i < 32; ++i) a[i] *= gc;
    tmem_st32(tmem_addr(tm, 32 * quarter, TM_S + 32 * part), a);
}

// ---------------------------------------------------------------- phase 1b: token operands
// Thread (lane L, part p): token r = L % 64 of the q rows (L >= 64) or k rows (L < 64),
// channels [32p, 32p + 32).  Writes the tf32 row operand [K_r; Q_r] (TMEM).  Token r's
// diagonal-tile column operand is split between the k-row and the q-row thread, and the
// q-row thread also writes its K_Gamma B operand, so that the two halves (which run on
// different SMSPs) carry the same number of reciprocals.
__device__ __forceinline__ void phase1_tokens(uint8_t* sm, const float* vec, uint32_t tm, int L, int part,
                                              int quarter, int BT)
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
        const uint32_t rj = kc_row(J) + r;
        if (!isq) {
            st_shared_f4(kc + sw128_off_f32(rj, c0, KC_ROWS), tf32_round(xv[0] * rcpf(xs[0])),
                         tf32_round(xv[1] * rcpf(xs[1])), tf32_round(xv[2] * rcpf(xs[2])),
                         tf32_round(xv[3] * rcpf(xs[3])));
        } else {      // and the K_Gamma B operand: k_r e^{Gamma_r} = k_r x_r E_J (bf16)
            float kv[8];
            unpack8(ld_shared_v4(sbase + OFF_K + sw128_chunk(r, c0 >> 3, 64)), kv);
#pragma unroll
            for (int e = 0; e < 8; ++e) kv[e] = valid ? kv[e] : 0.f;
            st_shared_f4(kc + sw128_off_f32(rj, c0 + 4, KC_ROWS), tf32_round(kv[4] * rcpf(xs[4])),
                         tf32_round(kv[5] * rcpf(xs[5])), tf32_round(kv[6] * rcpf(xs[6])),
                         tf32_round(kv[7] * rcpf(xs[7])));
            const float4 e4a = *reinterpret_cast<const float4*>(vec + (V_E + J) * 128 + c0);
            const float4 e4b = *reinterpret_cast<const float4*>(vec + (V_E + J) * 128 + c0 + 4);
            const float ev[8] = {e4a.x, e4a.y, e4a.z, e4a.w, e4b.x, e4b.y, e4b.z, e4b.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) kv[e] = kv[e] * xs[e] * ev[e];
            st_shared_v4(sbase + OFF_KG + sw128_chunk(r, c0 >> 3, 64), pack_bf16x2(kv[0], kv[1]),
                         pack_bf16x2(kv[2], kv[3]), pack_bf16x2(kv[4], kv[5]), pack_bf16x2(kv[6], kv[7]));
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
    // steps 3a/3b: thread (row i of the lower half, columns [8 jg, 8 jg + 8), q parity qh); the
    // two q parities of an output sit 16 lanes apart and are summed with one shuffle.
    const int lane = t & 31, w = t >> 5;
    const int jg = lane & 3, i = 4 * w + ((lane >> 2) & 3), qh = lane >> 4;
    float acc[8];
    {   // 3a: Y = A[32:64, 0:32] H0
        const float* arow = sA + (32 + i) * LDA + qh;
        const float* hcol = sT + qh * LDA + 8 * jg;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
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
    {   // 3b: T[32:64, 0:32] = -H1 Y; rows 0-15 of H1 are zero past column 15
        const float* hrow = sT + (32 + i) * LDA + 32 + qh;
        const float* y = sY + qh * LDY + 8 * jg;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        auto step = [&](int k) {
            const float a = hrow[2 * k];
            const float4 y0 = *reinterpret_cast<const float4*>(y + 2 * k * LDY);
            const float4 y1 = *reinterpret_cast<const float4*>(y + 2 * k * LDY + 4);
            acc[0] = fmaf(a, y0.x, acc[0]); acc[1] = fmaf(a, y0.y, acc[1]);
            acc[2] = fmaf(a, y0.z, acc[2]); acc[3] = fmaf(a, y0.w, acc[3]);
            acc[4] = fmaf(a, y1.x, acc[4]); acc[5] = fmaf(a, y1.y, acc[5]);
            acc[6] = fmaf(a, y1.z, acc[6]); acc[7] = fmaf(a, y1.w, acc[7]);
        };
        if (w < 4) {   // i < 16
#pragma unroll
            for (int k = 0; k < 8; ++k) step(k);
        } else {
#pragma unroll
            for (int k = 0; k < 16; ++k) step(k);
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

// ---------------------------------------------------------------- the kernel
// 16 warps: warp w reaches TMEM lanes [32 (w % 4), +32) and works on column part w / 4.
__global__ void __launch_bounds__(kThreads, 1) kda_prefill_tc_kernel(const __grid_constant__ TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base; offsetting the __shared__ array itself (rather than rounding an
    // integer address) keeps every access through `sm` in the shared state space
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int quarter = warp & 3, part = warp >> 2;
    const int L = 32 * quarter + lane;   // the TMEM lane this thread may access
    float* vec = reinterpret_cast<float*>(sm + OFF_VEC);
    float* sbeta = reinterpret_cast<float*>(sm + OFF_BETA);
    uint64_t* bar_v = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint64_t* bar_k = bar_v + 1;
    uint64_t* bar_qg = bar_v + 2;
    uint64_t* bar_mma = bar_v + 3;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_v + 4);
    int* s_abort = reinterpret_cast<int*>(tslot + 1);
    const uint32_t sbase = smem_u32(sm);

    const int H = p.num_heads;
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    int bos, eos;
    if (!seq_bounds(p.cu_seqlens, n, p.num_seqs, p.total_tokens, p.status, bos, eos)) return;
    const int nchunks = (eos - bos + 63) >> 6;
    const size_t sbase_g = ((size_t)n * H + h) * 128 * 128;

    if (t == 0) {
        mbar_init(bar_v, 1);
        mbar_init(bar_k, 1);
        mbar_init(bar_qg, 1);
        mbar_init(bar_mma, 1);
        mbar_fence_init();
        *s_abort = 0;
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        tma_prefetch_desc(&p.tm_g);
        tma_prefetch_desc(&p.tm_o);
    }
    if (warp == 0) {
        tmem_alloc(tslot, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = *tslot;

    bool v_pending = false, k_pending = false, qg_pending = false, o_pending = false;   // thread 0 only
    bool mma_open = false;   // thread 0: MMAs issued after the last commit
    if (t == 0 && nchunks > 0) {
        issue_v_loads(p, sm, bar_v, 0, bos, h);
        issue_k_loads(p, sm, bar_k, bos, h);
        issue_qg_loads(p, sm, bar_qg, bos, h);
        v_pending = k_pending = qg_pending = true;
    }

    // initial state -> TMEM: lane L = key channel, columns [32 part, 32 part + 32)
    {
        float v[32];
        if (p.init_state) {
            const float4* src = reinterpret_cast<const float4*>(p.init_state + sbase_g + (size_t)L * 128 + 32 * part);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 f = __ldg(src + i);
                v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        tmem_st32(tmem_addr(tm, 32 * quarter, TM_S + 32 * part), v);
        tmem_wait_st();
    }

    float beta_next = (t < 64 && bos + t < eos) ? __ldg(p.beta + (size_t)(bos + t) * H + h) : 0.f;
    uint32_t v_par = 0, k_par = 0, qg_par = 0, mma_par = 0;
    bool ok = true;

    for (int ci = 0; ci < nchunks; ++ci) {
        const int t0 = bos + 64 * ci;
        const int BT = min(64, eos - t0);
        if (t < 64) sbeta[t] = beta_next;
        // this chunk's inputs (one barrier for the three copies)
        if (!(mbar_wait_bounded(bar_v, v_par, kWaitNs) && mbar_wait_bounded(bar_k, k_par, kWaitNs) &&
              mbar_wait_bounded(bar_qg, qg_par, kWaitNs)))
            atomicExch(s_abort, 1);
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        if (*s_abort) {
            ok = false;
            break;
        }
        v_par ^= 1u;
        k_par ^= 1u;
        qg_par ^= 1u;
        if (t == 0) v_pending = k_pending = qg_pending = false;
        if (t < 64) {
            const int tn = t0 + 64 + t;
            beta_next = (ci + 1 < nchunks && tn < eos) ? __ldg(p.beta + (size_t)tn * H + h) : 0.f;
        }

        // ---- phase 1: decayed operands
        phase1_cumsum(sm, vec, t, BT);
        __syncthreads();
        if (t < 128) phase1_factors(vec, t);
        if (t == 0 && o_pending) {   // the previous chunk's O staging must be read out before reuse
            bulk_wait_read();
            o_pending = false;
        }
        __syncthreads();
        phase1_tokens(sm, vec, tm, L, part, quarter, BT);
        __syncthreads();
        phase1_offdiag(sm, vec, t);
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before_sync();
        __syncthreads();

        // ---- next chunk's v, then phase 2: A and P by one tf32 MMA
        if (t == 0) {
            tc_fence_after_sync();
            if (ci + 1 < nchunks) {
                issue_v_loads(p, sm, bar_v, (ci + 1) & 1, t0 + 64, h);
                v_pending = true;
            }
            // all four references at once: N = 160 columns, reference m in columns [8m(m+1), 8(m+1)(m+2))
            const uint32_t idesc = idesc_tf32_f32(128, KC_ROWS);
            const uint32_t kc = sbase + OFF_X;
#pragma unroll
            for (int ks = 0; ks < 16; ++ks)
                umma_tf32_tmem_a(tm + TM_AP, tm + TM_KQ + 8 * ks, desc_kmajor(kc, KC_ROWS, ks), idesc,
                                 ks > 0 ? 1u : 0u);
            umma_commit(bar_mma);
        }
        build_ktilde(sm, vec, tm, L, part, quarter, BT);   // overlaps the MMA above
        tmem_wait_st();
        if (!(ok = wait_all(bar_mma, mma_par, s_abort))) break;
        mma_par ^= 1u;
        tc_fence_after_sync();

        // ---- phase 3: A/P read-out; solve; M = P Tb by MMA; [Tb; M] hi/lo into TMEM
        phase3_readout(sm, tm, L, quarter, part, sbeta);
        tmem_wait_st();
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        if (t < kSolveThreads) {
            phase3_solve(sm, t);
        } else {   // meanwhile warps 8-15: the state's bf16 B operand, S <- gamma_C S, and the seed
            build_state_operand(sm, vec, tm, L, 2 * (part - 2), quarter);
            build_state_operand(sm, vec, tm, L, 2 * (part - 2) + 1, quarter);
            phase3_seed(sm, vec, tm, L, 2 * (part - 2), quarter, BT);
            phase3_seed(sm, vec, tm, L, 2 * (part - 2) + 1, quarter, BT);
            tmem_wait_st();
            fence_proxy_async_smem();
        }
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        // the k tile of this chunk is no longer read: fetch the next chunk's
        if (t == 0 && ci + 1 < nchunks) {
            issue_k_loads(p, sm, bar_k, t0 + 64, h);
            k_pending = true;
        }
        phase3_tb_operands(sm, t, sbeta);
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        if (t == 0) {
            tc_fence_after_sync();
            const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 1);
            const uint32_t tbh = sbase + OFF_X + X_TBH, tbl = sbase + OFF_X + X_TBL;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + TM_M, tm + TM_PH + 8 * ks, desc_mnmajor(tbh, 64, ks), idesc, ks > 0 ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + TM_M, tm + TM_PH + 8 * ks, desc_mnmajor(tbl, 64, ks), idesc, 1u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + TM_M, tm + TM_PL + 8 * ks, desc_mnmajor(tbh, 64, ks), idesc, 1u);
            umma_commit(bar_mma);
        }
        if (quarter < 2) {   // Tb rows (lanes 0-63), columns [16 part, +16), from the hi/lo B-operand tiles
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const uint4 h4 = ld_shared_v4(sbase + OFF_X + X_TBH + sw128_chunk(L, 2 * part + cc, 64));
                const uint4 l4 = ld_shared_v4(sbase + OFF_X + X_TBL + sw128_chunk(L, 2 * part + cc, 64));
                hi[4 * cc] = h4.x; hi[4 * cc + 1] = h4.y; hi[4 * cc + 2] = h4.z; hi[4 * cc + 3] = h4.w;
                lo[4 * cc] = l4.x; lo[4 * cc + 1] = l4.y; lo[4 * cc + 2] = l4.z; lo[4 * cc + 3] = l4.w;
            }
            tmem_st8u(tmem_addr(tm, 32 * quarter, TM_TPH + 8 * part), hi);
            tmem_st8u(tmem_addr(tm, 32 * quarter, TM_TPL + 8 * part), lo);
        }
        if (!(ok = wait_all(bar_mma, mma_par, s_abort))) break;
        mma_par ^= 1u;
        tc_fence_after_sync();
        if (quarter >= 2) {   // M rows (lanes 64-127), columns [16 part, +16) -> hi/lo
            float a[16];
            tmem_ld16(tmem_addr(tm, 32 * quarter, TM_M + 16 * part), a);
            tmem_wait_ld();
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) split_bf16x2(a[2 * i], a[2 * i + 1], hi[i], lo[i]);
            tmem_st8u(tmem_addr(tm, 32 * quarter, TM_TPH + 8 * part), hi);
            tmem_st8u(tmem_addr(tm, 32 * quarter, TM_TPL + 8 * part), lo);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncthreads();

        // ---- phase 4: D2 = [0; -Q_Gamma] + [Tb; M] K_Gamma (hi + lo) = [Wk; -Q'], A1 = -D2; the
        // state-independent half of D1, [Tb; M] V (hi + lo), queued right behind it
        if (t == 0) {
            tc_fence_after_sync();
            // the q and g tiles of this chunk are no longer read: fetch the next chunk's
            if (ci + 1 < nchunks) {
                issue_qg_loads(p, sm, bar_qg, t0 + 64, h);
                qg_pending = true;
            }
            const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + TM_D2, tm + TM_TPH + 8 * ks, desc_mnmajor(sbase + OFF_KG, 64, ks), idesc, 1u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + TM_D2, tm + TM_TPL + 8 * ks, desc_mnmajor(sbase + OFF_KG, 64, ks), idesc, 1u);
            umma_commit(bar_mma);
            const uint32_t vb = sbase + ((ci & 1) ? OFF_V1 : OFF_V0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + TM_D1, tm + TM_TPH + 8 * ks, desc_mnmajor(vb, 64, ks), idesc, ks > 0 ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + TM_D1, tm + TM_TPL + 8 * ks, desc_mnmajor(vb, 64, ks), idesc, 1u);
            mma_open = true;   // committed with phase 5b's MMAs
        }
        if (!(ok = wait_all(bar_mma, mma_par, s_abort))) break;
        mma_par ^= 1u;
        tc_fence_after_sync();
        {   // A1 = -D2 = [-Wk; Q'], columns [16 part, +16), written over D2 once every thread has read it
            float a[32];
            tmem_ld32(tmem_addr(tm, 32 * quarter, TM_D2 + 32 * part), a);
            tmem_wait_ld();
            tc_fence_before_sync();
            __syncthreads();
            tc_fence_after_sync();
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(-a[2 * i], -a[2 * i + 1]);
            tmem_st16u(tmem_addr(tm, 32 * quarter, TM_A1 + 16 * part), pk);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncthreads();
        // ---- phase 5b: D1 += [-Wk; Q'] S (the [Tb; M] V half was queued in phase 4)
        if (t == 0) {
            tc_fence_after_sync();
            const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                umma_bf16_tmem_a(tm + TM_D1, tm + TM_A1 + 8 * ks, desc_mnmajor(sbase + OFF_X + X_SB, 128, ks), idesc,
                                 1u);
            umma_commit(bar_mma);
            mma_open = false;
        }
        if (!(ok = wait_all(bar_mma, mma_par, s_abort))) break;
        mma_par ^= 1u;
        tc_fence_after_sync();

        // ---- phase 5c: rows 0-63 -> W (hi + lo) B operands
        if (quarter < 2) {
            float a[32];
            tmem_ld32(tmem_addr(tm, 32 * quarter, TM_D1 + 32 * part), a);
            tmem_wait_ld();
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) split_bf16x2(a[2 * i], a[2 * i + 1], hi[i], lo[i]);
            store_row32_bf16(sbase + OFF_X + X_WH, L, 4 * part, 64, hi);
            store_row32_bf16(sbase + OFF_X + X_WL, L, 4 * part, 64, lo);
            fence_proxy_async_smem();
        }
        tc_fence_before_sync();
        __syncthreads();

        // ---- phase 5d: S += K~^T W (hi hi + hi lo + lo hi), while rows 64-127 (O) go out
        if (t == 0) {
            tc_fence_after_sync();
            const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + TM_S, tm + TM_KT + 8 * ks, desc_mnmajor(sbase + OFF_X + X_WH, 64, ks), idesc,
                                 1u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + TM_S, tm + TM_KT + 8 * ks, desc_mnmajor(sbase + OFF_X + X_WL, 64, ks), idesc,
                                 1u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + TM_S, tm + TM_KTL + 8 * ks, desc_mnmajor(sbase + OFF_X + X_WH, 64, ks), idesc,
                                 1u);
            umma_commit(bar_mma);
        }
        if (quarter >= 2) {
            tc_fence_after_sync();
            const int r = L - 64;
            float a[32];
            tmem_ld32(tmem_addr(tm, 32 * quarter, TM_D1 + 32 * part), a);
            tmem_wait_ld();
            if (BT == 64) {
                // stage in 128-byte-swizzled [64 tok][32] fp32 boxes, one TMA store per box:
                // boxes 0-1 in the free top of the X region, 2-3 in this chunk's v buffer
                const uint32_t box = (part < 2) ? sbase + OFF_X + X_OST + 8192 * part
                                                : sbase + ((ci & 1) ? OFF_V1 : OFF_V0) + 8192 * (part - 2);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    st_shared_f4(box + sw128_off_f32(r, 4 * q, 64), a[4 * q], a[4 * q + 1], a[4 * q + 2], a[4 * q + 3]);
                fence_proxy_async_smem();
            } else if (r < BT) {
                float4* dst = reinterpret_cast<float4*>(p.out + ((size_t)(t0 + r) * H + h) * 128 + 32 * part);
#pragma unroll
                for (int i = 0; i < 8; ++i) dst[i] = make_float4(a[4 * i], a[4 * i + 1], a[4 * i + 2], a[4 * i + 3]);
            }
        }
        if (!(ok = wait_all(bar_mma, mma_par, s_abort))) break;
        mma_par ^= 1u;
        // state snapshot after a full chunk that ends on a checkpoint boundary
        {
            const int done = t0 + 64 - bos;
            if (p.checkpoints && BT == 64 && done % p.ckpt_interval == 0 && done / p.ckpt_interval <= p.ckpt_slots) {
                tc_fence_after_sync();
                const int slot = done / p.ckpt_interval - 1;
                float v[32];
                tmem_ld32(tmem_addr(tm, 32 * quarter, TM_S + 32 * part), v);
                tmem_wait_ld();
                float4* dst = reinterpret_cast<float4*>(
                    p.checkpoints + (((size_t)n * H + h) * p.ckpt_slots + slot) * 128 * 128 + (size_t)L * 128 + 32 * part);
#pragma unroll
                for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                tc_fence_before_sync();
            }
        }
        if (t == 0 && BT == 64) {
            const uint8_t* vb = sm + ((ci & 1) ? OFF_V1 : OFF_V0);
            tma_store_3d(&p.tm_o, sm + OFF_X + X_OST, 0, h, t0);
            tma_store_3d(&p.tm_o, sm + OFF_X + X_OST + 8192, 32, h, t0);
            tma_store_3d(&p.tm_o, vb, 64, h, t0);
            tma_store_3d(&p.tm_o, vb + 8192, 96, h, t0);
            bulk_commit();
            o_pending = true;
        }
    }
    if (t == 0) bulk_wait_all();   // staged O fully written before the CTA's shared memory goes away

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (ok && p.final_state) {
        float v[32];
        tmem_ld32(tmem_addr(tm, 32 * quarter, TM_S + 32 * part), v);
        tmem_wait_ld();
        float4* dst = reinterpret_cast<float4*>(p.final_state + sbase_g + (size_t)L * 128 + 32 * part);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
    if (!ok && t == 0) {
        // a wait gave up: record it, let in-flight copies and MMAs land (bounded), then leave
        report_status(p.status, kDevTimeout);
        if (v_pending) mbar_wait_bounded(bar_v, v_par, kWaitNs);
        if (k_pending) mbar_wait_bounded(bar_k, k_par, kWaitNs);
        if (qg_pending) mbar_wait_bounded(bar_qg, qg_par, kWaitNs);
        mbar_wait_bounded(bar_mma, mma_par, kWaitNs);
        if (mma_open) {   // MMAs queued behind that commit: commit and wait for them too
            umma_commit(bar_mma);
            mbar_wait_bounded(bar_mma, mma_par ^ 1u, kWaitNs);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, TM_COLS);
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

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream)
{
    TcParams p;
    if (!make_map(&p.tm_q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.num_heads, a.total_tokens, 64) ||
        !make_map(&p.tm_k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.num_heads, a.total_tokens, 64) ||
        !make_map(&p.tm_v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.num_heads, a.total_tokens, 64) ||
        !make_map(&p.tm_g, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.num_heads, a.total_tokens, 32) ||
        !make_map(&p.tm_o, a.out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.num_heads, a.total_tokens, 32))
        return cudaErrorInvalidValue;
    p.beta = a.beta;
    p.cu_seqlens = a.cu_seqlens;
    p.init_state = a.init_state;
    p.out = a.out;
    p.final_state = a.final_state;
    p.checkpoints = a.checkpoints;
    p.ckpt_interval = a.checkpoints ? a.ckpt_interval : 64;
    p.ckpt_slots = a.ckpt_slots;
    p.num_seqs = a.num_seqs;
    p.total_tokens = a.total_tokens;
    p.num_heads = a.num_heads;
    p.status = a.status;
    cudaError_t e = cudaFuncSetAttribute(kda_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long units = (long long)a.num_seqs * a.num_heads;
    kda_prefill_tc_kernel<<<(unsigned)units, kThreads, SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
