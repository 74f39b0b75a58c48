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
//   1  decayed operands to TMEM (A operands) and shared memory (B operands) from the
//      per-channel g cumsums and factors (the first chunk's formed here, the others'
//      under the previous chunk's MMAs).
//   2  A and P by one tf32 MMA over the four sub-tile references side by side, while
//      all warps build K~^T (TMEM); TMA prefetch of the next chunk's v once the last
//      chunk's O store has read its staging.
//   3  T = (I + A)^-1 in fp32 on CUDA cores (8 warps) while the other 8 build the
//      state's bf16 B operand, apply the chunk decay to S and seed the next
//      accumulator with [0; -Q_Gamma]; TMA prefetch of the next chunk's q, k and g;
//      M = P Tb by three bf16 MMAs (hi/lo splits).
//   4  [Wk; -Q'] by MMA onto the seed (the next chunk's cumsums alongside), and the
//      state-independent half of D1, [Tb; M] V, queued behind it; then the [-Wk; Q']
//      operand over the read accumulator.
//   5  D1 += [-Wk; Q'] S by MMA (the next chunk's factors alongside): rows 0-63 are W,
//      rows 64-127 are O; W to shared memory; S += K~^T W by MMA while O is staged in
//      shared memory (two boxes past the shared map, two in the chunk's v buffer) and
//      written by TMA bulk stores (direct stores for a sequence's ragged last chunk).
#include "kda_prefill_tc_phases.cuh"

namespace kda {
namespace {

using namespace sm100;

// O staging boxes 0-1 (dv columns 0-63: 2 x [64 tok][32] fp32, 128-byte swizzle) past the
// shared map (boxes 2-3 go to the chunk's v buffer): phase 1 then writes the X region without
// waiting for the last chunk's O store, which only has to have read its boxes before the next
// v load (phase 2).
constexpr uint32_t T_OST = ((uint32_t)SMEM_USED + 1023u) & ~1023u;
constexpr size_t TC_SMEM_BYTES = T_OST + 16384 + 1024;   // + slack for 1024-byte alignment
static_assert(TC_SMEM_BYTES <= 232448, "one-CTA-per-unit shared memory");

// ---------------------------------------------------------------- the kernel
// 16 warps: warp w reaches TMEM lanes [32 (w % 4), +32) and works on column part w / 4.
// kPro: the input prologue is compiled in (a separate instance, so that the common one
// keeps its registers).
template <bool kPro>
__global__ void __launch_bounds__(kThreads, 1) kda_prefill_tc_kernel(const __grid_constant__ TcParams p)
{
    const int pro = kPro ? p.prologue : 0;
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
    uint64_t* bar_z = bar_v + 5;   // the gate's logits (bytes 40-47 of the barrier block)
    const uint32_t sbase = smem_u32(sm);

    const int H = p.num_heads;
    const int n = unit_sequence(p.cu_seqlens, p.num_seqs, (int)blockIdx.x / H, reinterpret_cast<int*>(sm + OFF_X));
    const int h = blockIdx.x % H;
    int bos, eos;
    if (!seq_bounds(p.cu_seqlens, n, p.num_seqs, p.total_tokens, p.status, bos, eos)) return;
    const int nchunks = (eos - bos + 63) >> 6;
    const size_t sbase_g = ((size_t)n * H + h) * 128 * 128;

    if (t == 0) {
        mbar_init(bar_v, 1);
        mbar_init(bar_k, 1);
        mbar_init(bar_qg, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_z, 1);
        mbar_fence_init();
        *s_abort = 0;
        if (p.gate) tma_prefetch_desc(&p.tm_z);
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

    bool v_pending = false, k_pending = false, qg_pending = false, o_pending = false, z_pending = false;   // thread 0
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

    float beta_next = (t < 64 && bos + t < eos) ? beta_of(__ldg(p.beta + (size_t)(bos + t) * H + h), pro) : 0.f;
    uint32_t v_par = 0, k_par = 0, qg_par = 0, mma_par = 0, z_par = 0;
    bool ok = true;
    KDA_CLK_DECL(clk);

    for (int ci = 0; ci < nchunks; ++ci) {
        const int t0 = bos + 64 * ci;
        const int BT = min(64, eos - t0);
        if (t < 64) sbeta[t] = beta_next;
        // chunks after the first had their q and g tiles in, and their cumsums and factors
        // formed, under the previous chunk's [Wk; -Q'] and D1 MMAs
        const bool pre_done = ci > 0;
        // this chunk's inputs (one barrier for the copies)
        if (!(mbar_wait_bounded(bar_v, v_par, kWaitNs) && mbar_wait_bounded(bar_k, k_par, kWaitNs) &&
              (pre_done || mbar_wait_bounded(bar_qg, qg_par, kWaitNs))))
            atomicExch(s_abort, 1);
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        if (*s_abort) {
            ok = false;
            break;
        }
        KDA_CLK(clk, 0);   // this chunk's inputs in
        v_par ^= 1u;
        k_par ^= 1u;
        if (!pre_done) qg_par ^= 1u;
        if (t == 0) v_pending = k_pending = qg_pending = false;
        if (t < 64) {
            const int tn = t0 + 64 + t;
            beta_next = (ci + 1 < nchunks && tn < eos) ? beta_of(__ldg(p.beta + (size_t)tn * H + h), pro) : 0.f;
        }

        if (pro & kProQK) {
            phase0_normalise_qk(sm, t);
            __syncthreads();
        }
        // ---- phase 1: decayed operands
        if (!pre_done) {
            phase1_cumsum(sm, vec, t, BT, pro);
            __syncthreads();
            if (t < 128) phase1_factors(vec, t);
            __syncthreads();
        }
        phase1_tokens(sm, vec, tm, L, part, quarter, BT);
        __syncthreads();
        phase1_offdiag(sm, vec, t);
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before_sync();
        __syncthreads();
        KDA_CLK(clk, 1);   // phase 1

        // ---- next chunk's v, then phase 2: A and P by one tf32 MMA
        if (t == 0) {
            tc_fence_after_sync();
            // all four references at once: N = 160 columns, reference m in columns [8m(m+1), 8(m+1)(m+2))
            const uint32_t idesc = idesc_tf32_f32(128, KC_ROWS);
            const uint32_t kc = sbase + OFF_X;
#pragma unroll
            for (int ks = 0; ks < 16; ++ks)
                umma_tf32_tmem_a(tm + TM_AP, tm + TM_KQ + 8 * ks, desc_kmajor(kc, KC_ROWS, ks), idesc,
                                 ks > 0 ? 1u : 0u);
            umma_commit(bar_mma);
            if (o_pending) {   // the last chunk's O store has read its boxes (one is the v buffer loaded next)
                bulk_wait_read();
                o_pending = false;
            }
            if (ci + 1 < nchunks) {
                issue_v_loads(p, sm, bar_v, (ci + 1) & 1, t0 + 64, h);
                v_pending = true;
            }
        }
        build_ktilde(sm, vec, tm, L, part, quarter, BT);   // overlaps the MMA above
        tmem_wait_st();
        if (!(ok = wait_all(bar_mma, mma_par, s_abort))) break;
        mma_par ^= 1u;
        tc_fence_after_sync();
        KDA_CLK(clk, 2);   // A/P MMA with K~ alongside

        // ---- phase 3: A/P read-out; solve; M = P Tb by MMA; [Tb; M] hi/lo into TMEM
        phase3_readout(sm, tm, L, quarter, part, sbeta);
        tmem_wait_st();
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        KDA_CLK(clk, 3);   // A/P read-out
        if (t < kSolveThreads) {
            phase3_solve(sm, t);
        } else {   // meanwhile warps 8-15: the state's bf16 B operand, S <- gamma_C S, and the seed
            build_state_operand(sm, tm, L, 2 * (part - 2), quarter);
            build_state_operand(sm, tm, L, 2 * (part - 2) + 1, quarter);
            phase3_seed(sm, vec, tm, L, 2 * (part - 2), quarter, BT);
            phase3_seed(sm, vec, tm, L, 2 * (part - 2) + 1, quarter, BT);
            tmem_wait_st();
            fence_proxy_async_smem();
        }
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        KDA_CLK(clk, 4);   // solve, with the state operand and the seed alongside
        // the q, k and g tiles of this chunk are no longer read: fetch the next chunk's
        if (t == 0 && ci + 1 < nchunks) {
            issue_k_loads(p, sm, bar_k, t0 + 64, h);
            issue_qg_loads(p, sm, bar_qg, t0 + 64, h);
            k_pending = qg_pending = true;
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
        KDA_CLK(clk, 5);   // Tb operands, M = P Tb, [Tb; M] hi/lo

        // ---- phase 4: D2 = [0; -Q_Gamma] + [Tb; M] K_Gamma (hi + lo) = [Wk; -Q'], A1 = -D2; the
        // state-independent half of D1, [Tb; M] V (hi + lo), queued right behind it
        if (t == 0) {
            tc_fence_after_sync();
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
        // meanwhile the next chunk's cumsums (its q and g tiles were fetched after the solve;
        // this chunk no longer reads the g tile or vec[V_D]), its factors under the D1 MMAs of
        // phase 5b; gamma_C of this chunk is kept in a register, as those overwrite vec
        const float gamma_c = vec[V_GC * 128 + L];
        if (ci + 1 < nchunks) {
            if (!mbar_wait_bounded(bar_qg, qg_par, kWaitNs)) atomicExch(s_abort, 1);
            qg_par ^= 1u;
            if (t == 0) qg_pending = false;
            phase1_cumsum(sm, vec, t, min(64, eos - t0 - 64), pro);
        }
        if (!(ok = wait_all(bar_mma, mma_par, s_abort))) break;
        mma_par ^= 1u;
        tc_fence_after_sync();
        KDA_CLK(clk, 6);   // [Wk; -Q'] MMA
        {   // A1 = -D2 = [-Wk; Q'] (hi) and [0; Q' lo], columns [16 part, +16), written over D2 once
            // every thread has read it
            float a[32];
            tmem_ld32(tmem_addr(tm, 32 * quarter, TM_D2 + 32 * part), a);
            tmem_wait_ld();
            tc_fence_before_sync();
            __syncthreads();
            tc_fence_after_sync();
            uint32_t pk[16], pl[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) split_bf16x2(-a[2 * i], -a[2 * i + 1], pk[i], pl[i]);
            if (quarter < 2) {
#pragma unroll
                for (int i = 0; i < 16; ++i) pl[i] = 0u;
            }
            tmem_st16u(tmem_addr(tm, 32 * quarter, TM_A1 + 16 * part), pk);
            tmem_st16u(tmem_addr(tm, 32 * quarter, TM_A1L + 16 * part), pl);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncthreads();
        KDA_CLK(clk, 7);   // [-Wk; Q'] hi/lo operands
        // ---- phase 5b: D1 += [-Wk; Q'] S_hi + [0; Q' lo] S_hi, then + [-Wk; Q'] S_lo once the
        // state's lo operand, formed while the first two run, is in (the [Tb; M] V half was
        // queued in phase 4; the order is the chunk-parallel scan's)
        if (t == 0) {
            tc_fence_after_sync();
            const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
            const uint32_t sh = sbase + OFF_X + X_SB;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                umma_bf16_tmem_a(tm + TM_D1, tm + TM_A1 + 8 * ks, desc_mnmajor(sh, 128, ks), idesc, 1u);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                umma_bf16_tmem_a(tm + TM_D1, tm + TM_A1L + 8 * ks, desc_mnmajor(sh, 128, ks), idesc, 1u);
        }
        state_lo_and_decay(sm, gamma_c, tm, L, part, quarter);   // and S <- gamma_C S
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before_sync();
        __syncthreads();
        if (t == 0) {
            tc_fence_after_sync();
            const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
            const uint32_t sl = sbase + OFF_X + X_SL;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                umma_bf16_tmem_a(tm + TM_D1, tm + TM_A1 + 8 * ks, desc_mnmajor(sl, 128, ks), idesc, 1u);
            umma_commit(bar_mma);
            mma_open = false;
        }
        // while the D1 MMAs run: the next chunk's factors (its cumsums were formed under the
        // [Wk; -Q'] MMA, several barriers ago)
        if (t < 128 && ci + 1 < nchunks) phase1_factors(vec, t);
        if (!(ok = wait_all(bar_mma, mma_par, s_abort))) break;
        mma_par ^= 1u;
        tc_fence_after_sync();
        KDA_CLK(clk, 8);   // the S half of D1, the state's lo operand and decay alongside
        if (t == 0 && p.gate && BT == 64) {   // the gate's logits into the O staging boxes (now free)
            const uint8_t* vbz = sm + ((ci & 1) ? OFF_V1 : OFF_V0);
            mbar_arrive_expect_tx(bar_z, 32768u);
            tma_load_3d(sm + T_OST, &p.tm_z, bar_z, 0, h, t0);
            tma_load_3d(sm + T_OST + 8192, &p.tm_z, bar_z, 32, h, t0);
            tma_load_3d(const_cast<uint8_t*>(vbz), &p.tm_z, bar_z, 64, h, t0);
            tma_load_3d(const_cast<uint8_t*>(vbz) + 8192, &p.tm_z, bar_z, 96, h, t0);
            z_pending = true;
            if (ci + 1 < nchunks) {   // and the next chunk's into L2
#pragma unroll
                for (int j = 0; j < 4; ++j) tma_prefetch_3d(&p.tm_z, 32 * j, h, t0 + 64);
            }
        }

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
        KDA_CLK(clk, 9);   // W hi/lo

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
                const uint32_t box = (part < 2) ? sbase + T_OST + 8192 * part
                                                : sbase + ((ci & 1) ? OFF_V1 : OFF_V0) + 8192 * (part - 2);
                if (p.gate) {   // the output gate, o * sigmoid(z), on the logits TMA put in the boxes
                    if (!mbar_wait_bounded(bar_z, z_par, kWaitNs)) atomicExch(s_abort, 1);
                    z_par ^= 1u;
                    stage_gated_row(box, r, a);
                } else {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        st_shared_f4(box + sw128_off_f32(r, 4 * q, 64), a[4 * q], a[4 * q + 1], a[4 * q + 2],
                                     a[4 * q + 3]);
                }
                fence_proxy_async_smem();
            } else if (r < BT) {
                const size_t o0 = ((size_t)(t0 + r) * H + h) * 128 + 32 * part;
                float4* dst = reinterpret_cast<float4*>(p.out + o0);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 o = make_float4(a[4 * i], a[4 * i + 1], a[4 * i + 2], a[4 * i + 3]);
                    dst[i] = p.gate ? gate4(o, p.gate + o0 + 4 * i) : o;
                }
            }
        }
        if (!(ok = wait_all(bar_mma, mma_par, s_abort))) break;
        mma_par ^= 1u;
        if (t == 0 && z_pending) {   // the O warps have waited on it: the logits are in
            z_par ^= 1u;
            z_pending = false;
        }
        KDA_CLK(clk, 10);   // state update, O staged
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
            tma_store_3d(&p.tm_o, sm + T_OST, 0, h, t0);
            tma_store_3d(&p.tm_o, sm + T_OST + 8192, 32, h, t0);
            tma_store_3d(&p.tm_o, vb, 64, h, t0);
            tma_store_3d(&p.tm_o, vb + 8192, 96, h, t0);
            bulk_commit();
            o_pending = true;
        }
        KDA_CLK(clk, 11);   // checkpoint, O stores issued
        KDA_CLK_COUNT(clk, 31);
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
        if (z_pending) mbar_wait_bounded(bar_z, z_par, kWaitNs);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, TM_COLS);
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream)
{
    TcParams p;
    if (!make_map(&p.tm_q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.num_heads, a.total_tokens, 64) ||
        !make_map(&p.tm_k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.num_heads, a.total_tokens, 64) ||
        !make_map(&p.tm_v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.num_heads, a.total_tokens, 64) ||
        !make_map(&p.tm_g, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.num_heads, a.total_tokens, 32) ||
        !make_map(&p.tm_o, a.out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.num_heads, a.total_tokens, 32) ||
        (a.gate && !make_map(&p.tm_z, a.gate, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.num_heads, a.total_tokens, 32)))
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
    p.prologue = a.prologue;
    p.gate = a.gate;
    auto kern = a.prologue ? kda_prefill_tc_kernel<true> : kda_prefill_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long units = (long long)a.num_seqs * a.num_heads;
    kern<<<(unsigned)units, kThreads, TC_SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda

#ifdef KDA_PHASE_CLOCKS
// Instrumented build only: copy out and clear this file's cycle marks (kClockSlots values).
extern "C" int kda_phase_clocks_tc(unsigned long long* out)
{
    if (cudaMemcpyFromSymbol(out, kda::phase_clock_slots, sizeof(kda::phase_clock_slots)) != cudaSuccess) return -1;
    static const unsigned long long zero[kda::kClockSlots] = {};
    return cudaMemcpyToSymbol(kda::phase_clock_slots, zero, sizeof(zero)) == cudaSuccess ? 0 : -1;
}
#endif
