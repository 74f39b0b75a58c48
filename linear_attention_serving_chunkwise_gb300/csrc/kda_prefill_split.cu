// Chunk-parallel KDA prefill on the tcgen05 tensor cores (bf16 q/k/v, dk = dv = 128):
// the chunkwise form of llm-atlas "K3_RESEARCH.md" Q07 split at the one place where it
// is sequential.  Everything a chunk needs that does not depend on the state entering it
// (the g cumsum, A and P, T = (I + A)^-1, Tb = T diag(beta), M = P Tb, Wk = Tb K_Gamma,
// Q' = Q_Gamma - M K_Gamma and K~ = K e^{Gamma_63 - Gamma}) depends only on that chunk's
// q, k, g and beta, so it is computed for all (sequence, head, chunk) items at once; the
// state recurrence
//   W = Tb V - Wk S,   O = Q' S + M V,   S <- Diag(gamma_C) S + K~^T W
// then walks each (sequence, head)'s chunks in order.  Three launches per call, or two when
// at least 32 SMs' CTAs are left over from the scans: then steps 2 and 3 share one
// cooperative launch (kda_prep_scan_kernel) and the scans overlap the last prep items:
//   1  kda_chunk_offsets_kernel: per-sequence chunk offsets (prefix sums of ceil(len / 64)),
//      the cu_seqlens check, and a table of every chunk's (first token, sequence end), into
//      the workspace;
//   2  kda_chunk_prep_kernel: persistent CTAs over the items.  Each item runs the phases
//      of the one-CTA-per-head kernel up to [Wk; -Q'] (same functions, same arithmetic) and
//      writes the operands of its state step -- [-Wk; Q'] bf16, [Tb; M] and K~^T as bf16
//      hi + lo, gamma_C -- to the workspace as the byte images of 128-byte-swizzled K-major
//      tiles, so that they can be copied into shared memory as they are;
//   3  kda_state_scan_kernel: one CTA per (sequence, head), the state transposed (S^T, dv on
//      the lanes) in tensor memory, the CTA split into CUDA warps, an MMA-issuing thread and
//      a copy-issuing thread (see scan_unit).  Per chunk: S^T's bf16 operands (hi, lo) into
//      tensor memory and S^T <- S^T gamma_C; D1^T = V^T [Tb; M]^T + S^T [-Wk; Q']^T by MMAs
//      whose A operands are v and S^T and whose B operands are the images as they are; W^T
//      (hi + lo) into tensor memory and O out through shared memory by TMA; S^T += W^T K~.
//      The item's images arrive by bulk asynchronous copies ahead of their use, v by TMA.
// Each output element is the same sum of the same products as in the one-CTA-per-head
// kernel, so the results are the same; the work of steps 1-2 spreads over every SM
// instead of one SM per (sequence, head), at the price of 112.5 KB of operands per item
// written and read back through HBM.  The prep kernels come in two instances: with the
// input prologue (q/k normalisation, g and beta from logits) compiled in, and without.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "kda_prefill_tc_phases.cuh"

namespace kda {
namespace {

using namespace sm100;

// ---------------------------------------------------------------- one item's operand images (bytes)
constexpr uint32_t IMG_A1 = 0;          // [-Wk; Q'] bf16, K-major [128 rows][128 K] (2 x 16 KB)
constexpr uint32_t IMG_TBH = 32768;     // [Tb; M] hi bf16, K-major [128 rows][64 K]
constexpr uint32_t IMG_TBL = 49152;     // [Tb; M] lo
constexpr uint32_t IMG_GAM = 65536;     // gamma_C fp32 [128]
constexpr uint32_t IMG_FRONT = 66048;   // bytes [0, IMG_FRONT): read at the start of a chunk step
constexpr uint32_t IMG_KTH = 66048;     // K~^T hi bf16, K-major [128 dk rows][64 K tokens]
constexpr uint32_t IMG_KTL = 82432;     // K~^T lo
constexpr uint32_t IMG_BACK = 32768;    // bytes [IMG_KTH, IMG_KTH + IMG_BACK): read for the state update
constexpr uint32_t IMG_QLO = 98816;     // Q' lo = bf16(Q' - bf16(Q')), K-major [64 rows][128 K] (2 x 8 KB),
                                        // read at the start of a chunk step with the front
constexpr uint32_t IMG_BYTES = 115200;

// ---------------------------------------------------------------- state-scan shared memory (bytes)
constexpr uint32_t B_A1 = 0;            // the front image, copied whole
constexpr uint32_t B_TBH = IMG_TBH;
constexpr uint32_t B_TBL = IMG_TBL;
constexpr uint32_t B_GAM = IMG_GAM;
constexpr uint32_t B_KTH = 66560;       // the back image (1024-byte aligned)
constexpr uint32_t B_KTL = B_KTH + 16384;
constexpr uint32_t B_V0 = 99328;        // v tiles [64 tok][128 ch] bf16, two buffers
constexpr uint32_t B_V1 = 115712;
constexpr uint32_t B_QLO = 132096;      // Q' lo, K-major [64 rows][128 K] (2 x 8 KB), as the image holds it
constexpr uint32_t B_OST = 148480;      // O staging, two buffers of 4 x [64 tok][32 dv] fp32 boxes, 128-byte
                                        // swizzle (32 KB each), for the TMA store
constexpr uint32_t B_BAR = 230400;      // past the chunk prep's shared memory (the single launch runs both)
constexpr size_t B_SMEM_BYTES = B_BAR + 256 + 1024;
// the 256-byte block at B_BAR: the separate scan kernel's TMEM slot (word 40), the scan's abort
// word (44), the single launch's TMEM slot (48); from byte 64 the scan's mbarriers, by index:
constexpr uint32_t B_WORD_TSLOT = 40, B_WORD_ABORT = 44, B_WORD_TSLOT1 = 48, B_BARS = 64;
constexpr int B_BAR_FRONT = 0;     // [-Wk; Q'] and Q' lo of a chunk are in
constexpr int B_BAR_TB = 1;        // [Tb; M] hi + lo of a chunk are in
constexpr int B_BAR_BACK = 2;      // the back image (K~^T) is in
constexpr int B_BAR_V = 3;         // v of a chunk is in, one per buffer (2)
constexpr int B_BAR_GAMMA = 5;     // gamma_C of a chunk is in
constexpr int B_BAR_MMA = 6;       // D1's MMAs are done, then the state update's
constexpr int B_BAR_VDONE = 7;     // the V^T [Tb; M]^T MMAs are done
constexpr int B_BAR_SHI = 8;       // S^T_hi is written (the 14 CUDA warps arrive)
constexpr int B_BAR_SLO = 9;       // S^T_lo is written and S^T decayed (14 warps)
constexpr int B_BAR_WREADY = 10;   // W^T is written (14 warps)
constexpr int B_BAR_DREAD = 11;    // D1 is read out (14 warps)
constexpr int B_BAR_END = 12;      // the MMA issuer's last commit
constexpr int B_BAR_OSTAGED = 13;  // O of a chunk is staged (14 warps)
constexpr int B_BAR_SFREE = 14;    // a chunk's staged O taken (its store issued, the one before read)
constexpr int B_BAR_Z = 15;        // the gate logits of a chunk are in its O staging buffer, one per buffer (2)
constexpr int B_BAR_UPD = 17;      // a chunk's state update is done (for the producer: the back image is free)
constexpr int B_BAR_D1P = 18;      // a chunk's D1 is done (for the producer: the front image is free)
constexpr int B_BAR_COUNT = 19;
static_assert(B_WORD_TSLOT1 + 4 <= B_BARS && B_BARS + 8 * B_BAR_COUNT <= 256, "scan word block");
// tensor memory (columns), everything transposed: lane = dv
constexpr uint32_t B_TM_S = 0;          // S^T [128 dv][128 dk] fp32
constexpr uint32_t B_TM_D1 = 128;       // D1^T [128 dv][W^T: tokens 0-63 | O^T: tokens 0-63] fp32
constexpr uint32_t B_TM_SH = 256;       // S^T_hi, bf16 pairs along dk (64 columns)
constexpr uint32_t B_TM_SL = 320;       // S^T_lo
constexpr uint32_t B_TM_WH = 384;       // W^T_hi, bf16 pairs along the tokens (32 columns)
constexpr uint32_t B_TM_WL = 416;       // W^T_lo
constexpr uint32_t B_TM_COLS = 512;

// single-launch form: at least this many CTAs never scan (they finish the prep items), and
// the switch point uses these costs (cycles on GB300: a scan's 7.2 K per chunk as measured,
// the prep's 19.8 K per item (23.1 K with the input prologue) less an allowance for the
// scans' start and flag waits; swept on the B=1, H=96, T=8192 shape)
constexpr long long kSingleMinProducers = 32;
constexpr long long kScanCyclesPerChunk = 6000;
constexpr long long kPrepCyclesPerItem = 19600;
constexpr long long kPrepCyclesPerItemPrologue = 22900;   // the prologue instances' prep

static_assert(B_KTH % 1024 == 0 && B_V0 % 1024 == 0 && B_QLO % 1024 == 0, "tile alignment");
static_assert(B_KTH >= IMG_FRONT && B_V0 >= B_KTH + IMG_BACK && B_V1 == B_V0 + 16384 && B_QLO >= B_V1 + 16384 &&
                  B_OST >= B_QLO + 16384 && B_OST % 1024 == 0 && B_BAR >= B_OST + 65536 && B_SMEM_BYTES <= 232448 && B_TM_WL + 32 <= B_TM_COLS,
              "state-scan map overlaps");
static_assert(IMG_KTL == IMG_KTH + 16384 && IMG_QLO == IMG_KTH + IMG_BACK && IMG_BYTES == IMG_QLO + 16384 &&
                  IMG_BYTES % 16 == 0,
              "image map");

struct SplitParams {
    TcParams p;                 // inputs, outputs, tensor maps, status (as the one-CTA-per-head kernel)
    uint8_t* ops;               // operand images, item (global chunk gc, head h) at ((gc * H) + h) * IMG_BYTES
    int32_t* chunk_off;         // [num_seqs + 1]: first global chunk of each sequence
    int2* chunk_info;           // [chunks]: (first token, end of its sequence) of each global chunk
    int* counter;               // next unclaimed item (the single-launch form claims items from it)
    int* flags;                 // [items]: 1 once the item's images are in memory (single-launch form)
    int num_flags;              // entries of flags (an upper bound on the items)
};

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem_dst)),
                 "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// contiguous shared -> global copy (bulk-group completion); both 16-byte aligned, size % 16 == 0
__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(smem_src)),
                 "r"(bytes)
                 : "memory");
}

// Items are claimed from the global counter with one fetch-and-add each (handed out in
// increasing order).  A claim's raw index is resolved here: -1 once all `items` are taken;
// an index at or past `limit` is still this CTA's to do (so no item is ever dropped), but
// stops its further claims.
__device__ __forceinline__ int resolve_claim(int v, int items, int limit, bool& stop)
{
    if (v < 0 || v >= items) {
        stop = true;
        return -1;
    }
    if (v >= limit) stop = true;
    return v;
}

// The next claim: the counter's old value when `want`, else -1.  The fetch-and-add is
// predicated instead of selected on, so that nothing reads its result (and waits for the
// round trip to L2) before that result is resolved, an item later.
__device__ __forceinline__ int claim_async(int* counter, bool want)
{
    int v = -1;
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p atom.global.add.u32 %0, [%1], 1;\n\t}"
                 : "+r"(v)
                 : "l"(counter), "r"((unsigned)want)
                 : "memory");
    return v;
}

// acquire fence at GPU scope (after relaxed reads of flags that were set by release stores)
__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ int ld_relaxed_gpu(const int* p)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// wait until at most N committed bulk stores are incomplete (their writes not yet performed)
template <int N>
__device__ __forceinline__ void bulk_wait_group()
{
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// wait until at most N committed bulk stores are still reading their shared-memory source
template <int N>
__device__ __forceinline__ void bulk_wait_read_group()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// A wait of one role of the state scan: bounded like every wait, and it also gives up at once
// when another role has recorded an abort, so that one failure does not cost each role a
// full time-out.  The waiting thread sleeps between tests (up to 20 us each, woken when the
// phase completes), so that waiting warps take no issue slots from working ones.
__device__ __forceinline__ bool role_wait(uint64_t* bar, uint32_t parity, const int* s_abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*reinterpret_cast<const volatile int*>(s_abort) != 0 || globaltimer_ns() - t0 > kWaitNs) return false;
    }
}

// order this thread's generic-proxy and async-proxy accesses to global memory
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__device__ __forceinline__ void st_release_gpu(int* p, int v)
{
    asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// wait (bounded by kWaitNs of wall time) until *flag != 0; false if it gave up
__device__ __forceinline__ bool wait_flag(const int* flag)
{
    if (ld_acquire_gpu(flag)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!ld_acquire_gpu(flag)) {
        if (globaltimer_ns() - t0 > kWaitNs) return false;
        __nanosleep(64);
    }
    return true;
}

__device__ __forceinline__ void mbar_inval(uint64_t* bar)
{
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// start moving [gsrc, gsrc + bytes) into L2 (no completion to wait for)
__device__ __forceinline__ void prefetch_l2(const void* gsrc, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}

// the prep kernel stages each 32 KB piece of an item's image in shared memory and writes it
// with one bulk store, all three in turn in the v buffers of the shared map (which it does
// not use).  K_Gamma, the B operand of the item's last MMA, has two buffers (the shared
// map's and A_KG2), so that the next item's token phase can write its own while that MMA
// runs.  beta comes by cp.async into two buffers, one item ahead.
constexpr uint32_t A_STAGE = OFF_V0;
constexpr uint32_t A_KG2 = ((uint32_t)SMEM_USED + 1023u) & ~1023u;
constexpr uint32_t A_BETA2 = A_KG2 + 16384;
constexpr uint32_t A_INFO = A_BETA2 + 256;   // two chunk-table entries (int2), see prep_items
constexpr uint32_t A_USED = A_INFO + 16;
constexpr size_t A_SMEM_BYTES = A_USED + 1024;   // slack for 1024-byte alignment
static_assert(A_USED <= B_BAR, "the prep layout ends below the scan's word block, which the single launch's "
                                "TMEM slot occupies from the start");
static_assert(A_SMEM_BYTES <= 232448, "prep shared memory");
static_assert(B_BAR >= A_USED, "the scan's barrier block lies past the chunk prep's shared memory");
static_assert(OFF_V1 + 16384 == A_STAGE + 32768, "staging buffer");
static_assert(A_KG2 % 1024 == 0 && A_BETA2 % 16 == 0 && A_INFO % 8 == 0, "second K_Gamma, beta, info buffers");

__device__ __forceinline__ void cp_async4_zfill(void* smem_dst, const void* gsrc, bool valid)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(smem_dst)), "l"(gsrc),
                 "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem_dst, const void* gsrc)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// K~^T hi + lo into the prep's staging buffer (the back image's layout: K-major [128 dk rows]
// [64 tokens], 128-byte swizzle), each value as ktilde_pairs forms it.  Thread t takes key
// channels c, c + 1 (c = 2 (t % 64)) and tokens [8 g, 8 g + 8) (g = t / 64): one 4-byte load of
// k and one 8-byte load of x per token serve both channels.  A warp's stores land on rows of
// every residue mod 8 (lanes 4-7 of each group of 8 store row c + 1 first), so that each store
// instruction meets no more bank conflicts than its 512 bytes need.
__device__ __forceinline__ void ktilde_stage(uint8_t* sm, const float* vec, int t, int BT, uint32_t stage)
{
    const int cp = t & 63, g = t >> 6, c = 2 * cp, J = g >> 1;
    const uint32_t sbase = smem_u32(sm);
    const float2 dj = *reinterpret_cast<const float2*>(vec + (V_D + J) * 128 + c);
    const float2 gj = *reinterpret_cast<const float2*>(vec + (V_G + J) * 128 + c);
    const float f0 = dj.x * gj.x, f1 = dj.y * gj.y;
    float v0[8], v1[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int r = 8 * g + e;
        uint32_t kk;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(kk) : "r"(sbase + OFF_K + sw128_off(r, c, 64)));
        const float2 x = *reinterpret_cast<const float2*>(sm + OFF_G + sw128_off_f32(r, c, 64));
        const float k0 = (r < BT) ? __uint_as_float(kk << 16) : 0.f;
        const float k1 = (r < BT) ? __uint_as_float(kk & 0xffff0000u) : 0.f;
        v0[e] = k0 * (f0 * rcpf(x.x));
        v1[e] = k1 * (f1 * rcpf(x.y));
    }
    uint32_t h0[4], l0[4], h1[4], l1[4];
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
        split_bf16x2(v0[2 * pr], v0[2 * pr + 1], h0[pr], l0[pr]);
        split_bf16x2(v1[2 * pr], v1[2 * pr + 1], h1[pr], l1[pr]);
    }
    const bool odd_first = (t >> 2) & 1;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const bool one = (s == 0) == odd_first;   // this store writes channel c + 1
        const uint32_t row = c + (one ? 1 : 0);
        const uint32_t* h = one ? h1 : h0;
        const uint32_t* l = one ? l1 : l0;
        st_shared_v4(stage + sw128_chunk(row, g, 128), h[0], h[1], h[2], h[3]);
        st_shared_v4(stage + 16384 + sw128_chunk(row, g, 128), l[0], l[1], l[2], l[3]);
    }
}

// ---------------------------------------------------------------- step 1: chunk offsets
// One CTA of 1024 threads: chunk_off[n] = sum over m < n of ceil(len_m / 64), lengths of
// sequences that fail the cu_seqlens check counted as 0 (and the failure reported); then
// chunk_info[gc] = (first token, end of the sequence) of every global chunk, so that a
// chunk's item needs one load and no search.  Also zeroes the item counter and flags that
// the single-launch form claims and publishes items with.
__global__ void __launch_bounds__(1024) kda_chunk_offsets_kernel(const int32_t* cu_seqlens, int num_seqs,
                                                                 int total_tokens, int32_t* chunk_off,
                                                                 int2* chunk_info, int* counter, int* flags,
                                                                 int num_flags, int* status)
{
    __shared__ int warp_sums[32];
    __shared__ int carry;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    // the single-launch form's claim counter and item flags start from zero on every call
    for (int i = t; i < num_flags; i += 1024) flags[i] = 0;
    if (t == 0) {
        *counter = 0;
        carry = 0;
    }
    __syncthreads();
    for (int base = 0; base < num_seqs; base += 1024) {
        const int n = base + t;
        int cnt = 0;
        if (n < num_seqs) {
            int bos, eos;
            if (seq_bounds(cu_seqlens, n, num_seqs, total_tokens, status, bos, eos)) cnt = (eos - bos + 63) >> 6;
        }
        int x = cnt;   // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[w] = x;
        __syncthreads();
        if (w == 0) {
            int s = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += y;
            }
            warp_sums[lane] = s;   // inclusive over warps
        }
        __syncthreads();
        const int before = carry + (w > 0 ? warp_sums[w - 1] : 0) + x - cnt;
        if (n < num_seqs) chunk_off[n] = before;
        __syncthreads();
        if (t == 1023) carry = before + cnt;
        __syncthreads();
    }
    if (t == 0) chunk_off[num_seqs] = carry;
    __syncthreads();
    // chunk gc belongs to the last n with chunk_off[n] <= gc (chunk_off written above by this
    // CTA: plain loads)
    const int total = carry;
    for (int gc = t; gc < total; gc += 1024) {
        int lo = 0, hi = num_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (chunk_off[mid] <= gc) lo = mid;
            else hi = mid - 1;
        }
        int bos, eos;
        seq_bounds(cu_seqlens, lo, num_seqs, total_tokens, status, bos, eos);   // valid: it has chunks
        chunk_info[gc] = make_int2(bos + 64 * (gc - chunk_off[lo]), eos);
    }
}

// ---------------------------------------------------------------- step 2: per-item operands
struct Item {
    int h, t0, eos, gc;
};

// item = gc * H + h, with its (t0, eos) entry of the chunk table (read now: the prologue only)
__device__ __forceinline__ Item item_at(const SplitParams& sp, int item)
{
    const int H = sp.p.num_heads;
    Item it;
    it.gc = item / H;
    it.h = item - it.gc * H;
    const int2 info = __ldg(sp.chunk_info + it.gc);
    it.t0 = info.x;
    it.eos = info.y;
    return it;
}

// The chunk-prep work of one CTA.  Items come either in a fixed order (kDyn = false: CTA b
// takes b, b + gridDim.x, ...) or claimed one at a time from the global counter below
// `limit` (kDyn = true), in which case each item's flag is set once its three image pieces
// are in memory (two items later, or at the end).  The next item's q, k and g tiles are
// fetched by TMA while the current one is worked on (k once the A/P MMA is done, q and g
// once the seed of phase 3 is), its beta by cp.async into the other of two buffers.  Its
// phase 1 up to the off-diagonal rows runs while the current item's last MMA does.  16 warps; warp w reaches TMEM lanes [32 (w % 4), +32) and works on column part w / 4, as in
// the one-CTA-per-head kernel.  `tm`: 512 allocated TMEM columns.  On return the CTA's
// barriers are invalidated and its copies complete, so shared memory can be reused.
// kPro: the input prologue is compiled in (instances of their own, so that the common ones
// keep their registers and schedule).
template <bool kDyn, bool kPro>
__device__ __forceinline__ void prep_items(const SplitParams& sp, uint8_t* sm, uint32_t tm, int limit)
{
    const TcParams& p = sp.p;
    const int pro = kPro ? p.prologue : 0;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int quarter = warp & 3, part = warp >> 2;
    const int L = 32 * quarter + lane;
    float* vec = reinterpret_cast<float*>(sm + OFF_VEC);
    auto sbeta_buf = [&](int b) { return reinterpret_cast<float*>(sm + (b ? A_BETA2 : OFF_BETA)); };
    auto kg_buf = [](int b) { return b ? A_KG2 : OFF_KG; };
    uint64_t* bar_k = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint64_t* bar_qg = bar_k + 1;
    uint64_t* bar_mma = bar_k + 2;
    int* s_abort = reinterpret_cast<int*>(sm + OFF_BAR + 36);
    int* s_seq = reinterpret_cast<int*>(sm + OFF_BAR + 40);   // claimed item indices (kDyn)
    int2* s_info = reinterpret_cast<int2*>(sm + A_INFO);
    const uint32_t sbase = smem_u32(sm);
    const int H = p.num_heads;
    const int items = __ldg(sp.chunk_off + p.num_seqs) * H;
    const int G = gridDim.x;
    // kDyn: thread 0 claims the first two items; from then on the claims are kStorer's, one per
    // item, issued during the solve and resolved at the next item's top
    bool stop = false;                   // kStorer: no more claims
    int claim_raw = -1;                  // kStorer: a claim issued during the last solve, unresolved

    if (t == 0) {
        mbar_init(bar_k, 1);
        mbar_init(bar_qg, 1);
        mbar_init(bar_mma, 1);
        mbar_fence_init();
        *s_abort = 0;
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_g);
        if constexpr (kDyn) {
            s_seq[0] = resolve_claim(atomicAdd(sp.counter, 1), items, limit, stop);
            s_seq[1] = stop ? -1 : resolve_claim(atomicAdd(sp.counter, 1), items, limit, stop);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    // The tile loads are issued, the image pieces stored, waited for and published, and the
    // items claimed by kStorer, a thread of the warps that only write the seed during the
    // solve, so that this work fits in their idle time instead of delaying thread 0 (which
    // issues the MMAs).
    constexpr int kStorer = kSolveThreads;
    // the current and next items (index -1: none); the one after is looked up an item ahead
    // of its use, so that its chunk-table load is never waited for
    int item, nidx;
    if constexpr (kDyn) {
        item = s_seq[0];
        nidx = s_seq[1];
        if (t == kStorer) {   // thread 0's stop, and the claim resolved at the first item
            stop = nidx < 0 || nidx >= limit;
            claim_raw = claim_async(sp.counter, !stop);
        }
    } else {
        item = (int)blockIdx.x < items ? (int)blockIdx.x : -1;
        nidx = (item >= 0 && item + G < items) ? item + G : -1;
    }
    bool k_pending = false, qg_pending = false;   // kStorer: a load issued, not yet waited for
    int pub2 = -1, pub1 = -1;                     // kStorer (kDyn): done, not yet published
    Item cur{}, nxt{};
    if (nidx >= 0) nxt = item_at(sp, nidx);
    if (item >= 0) {
        cur = item_at(sp, item);
        if (t == kStorer) {
            issue_k_loads(p, sm, bar_k, cur.t0, cur.h);
            issue_qg_loads(p, sm, bar_qg, cur.t0, cur.h);
            k_pending = qg_pending = true;
        }
    }
    // beta of an item (tokens t0 .. t0 + 63, zero past the sequence's end) into buffer b
    auto fetch_beta = [&](const Item& it, int b) {
        if (t < 64) {
            const bool valid = it.t0 + t < it.eos;
            cp_async4_zfill(sbeta_buf(b) + t, valid ? p.beta + (size_t)(it.t0 + t) * H + it.h : p.beta, valid);
            cp_async_commit();
        }
    };
    if (item >= 0) fetch_beta(cur, 0);
    uint32_t k_par = 0, qg_par = 0, mma_par = 0;
    // phase 1 of an item up to the off-diagonal rows, once its tiles are in: per-channel
    // cumsums (g becomes x in place) and factors into vec, then the token rows into TMEM,
    // the [K; Q] operand in the X region and K_Gamma into buffer b.  The item's first
    // barrier orders these writes before they are read.
    auto phase1ab = [&](const Item& it, int b) -> bool {
        const int BTn = min(64, it.eos - it.t0);
        if (!mbar_wait_bounded(bar_qg, qg_par, kWaitNs)) atomicExch(s_abort, 1);
        __syncthreads();
        if (*s_abort) return false;
        qg_par ^= 1u;
        if (t == kStorer) qg_pending = false;
        phase1_cumsum(sm, vec, t, BTn, pro);
        __syncthreads();
        if (t < 128) phase1_factors(vec, t);
        if (!mbar_wait_bounded(bar_k, k_par, kWaitNs)) atomicExch(s_abort, 1);
        __syncthreads();
        if (*s_abort) return false;
        k_par ^= 1u;
        if (t == kStorer) k_pending = false;
        if (pro & kProQK) {
            phase0_normalise_qk(sm, t);
            __syncthreads();
        }
        phase1_tokens(sm, vec, tm, L, part, quarter, BTn, kg_buf(b));
        return true;
    };
    bool ok = item < 0 || phase1ab(cur, 0);
    KDA_CLK_DECL(clk);

    for (int li = 0; ok && item >= 0; ++li) {
        const float* sbeta = sbeta_buf(li & 1);
        const int h = cur.h, t0 = cur.t0;
        const int BT = min(64, cur.eos - t0);
        uint8_t* img = sp.ops + ((size_t)cur.gc * H + h) * IMG_BYTES;
        const bool has_next = nidx >= 0;
        const uint32_t kg = kg_buf(li & 1);
        if (t < 64) {
            cp_async_wait_all();   // this item's beta; thread 0: the next item's entry
            if ((pro & kProBeta) && t < BT) sbeta_buf(li & 1)[t] = sigmoid_fast(sbeta_buf(li & 1)[t]);
        }
        if constexpr (kDyn) {
            // the item after next: the claim issued during the last item's solve
            if (t == kStorer) s_seq[2] = has_next ? resolve_claim(claim_raw, items, limit, stop) : -1;
        }
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        KDA_CLK(clk, 0);   // loop top: claims, beta
        int n2;   // the item after next
        if constexpr (kDyn) n2 = s_seq[2];
        else n2 = (has_next && nidx + G < items) ? nidx + G : -1;
        if (li > 0 && has_next) {   // the next item's chunk-table entry, copied an item ago
            const int2 inf = s_info[(li + 1) & 1];
            nxt.t0 = inf.x;
            nxt.eos = inf.y;
        }
        if (has_next) fetch_beta(nxt, (li + 1) & 1);   // the buffer the previous item used
        // the chunk-table entry of the item after next, copied by thread 0 and read from shared
        // memory at the next item's top, so that no thread waits for the load
        if (t == 0 && n2 >= 0) {
            cp_async8(s_info + (li & 1), sp.chunk_info + n2 / H);
            cp_async_commit();
        }
        // ---- phase 1: decayed operands (all but the off-diagonal rows are done)
        phase1_offdiag(sm, vec, t);
        fence_proxy_async_smem();
        tmem_wait_st();
        if (t == kStorer) bulk_wait_read();   // the previous item's pieces have left the staging buffer
        tc_fence_before_sync();
        __syncthreads();
        KDA_CLK(clk, 1);   // off-diagonal rows

        // ---- phase 2: A and P by one tf32 MMA, while K~^T goes to the image
        if (t == 0) {
            tc_fence_after_sync();
            const uint32_t idesc = idesc_tf32_f32(128, KC_ROWS);
            const uint32_t kc = sbase + OFF_X;
#pragma unroll
            for (int ks = 0; ks < 16; ++ks)
                umma_tf32_tmem_a(tm + TM_AP, tm + TM_KQ + 8 * ks, desc_kmajor(kc, KC_ROWS, ks), idesc,
                                 ks > 0 ? 1u : 0u);
            umma_commit(bar_mma);
        }
        if constexpr (kPro) {   // the prologue instance keeps one key channel per thread (measured faster there)
            uint32_t hi[8], lo[8];
            ktilde_pairs(sm, vec, L, part, BT, hi, lo);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                st_shared_v4(sbase + A_STAGE + sw128_chunk(L, 2 * part + cc, 128), hi[4 * cc], hi[4 * cc + 1],
                             hi[4 * cc + 2], hi[4 * cc + 3]);
                st_shared_v4(sbase + A_STAGE + 16384 + sw128_chunk(L, 2 * part + cc, 128), lo[4 * cc],
                             lo[4 * cc + 1], lo[4 * cc + 2], lo[4 * cc + 3]);
            }
        } else {
            ktilde_stage(sm, vec, t, BT, sbase + A_STAGE);
        }
        fence_proxy_async_smem();
        if (t < 128) reinterpret_cast<float*>(img + IMG_GAM)[t] = vec[V_GC * 128 + t];
        if (!(ok = wait_all(bar_mma, mma_par, s_abort))) break;
        mma_par ^= 1u;
        tc_fence_after_sync();
        KDA_CLK(clk, 2);   // A/P MMA with K~ staged alongside
        if (t == kStorer) {
            if (has_next) {   // the k tile is no longer read
                issue_k_loads(p, sm, bar_k, nxt.t0, nxt.h);
                k_pending = true;
            }
            bulk_store(img + IMG_KTH, sm + A_STAGE, IMG_BACK);
            bulk_commit();
        }

        // ---- phase 3: A/P read-out; solve while warps 8-15 seed D2; M = P Tb; [Tb; M] hi/lo
        phase3_readout(sm, tm, L, quarter, part, sbeta);
        tmem_wait_st();
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        KDA_CLK(clk, 3);   // A/P read-out
        if (t < kSolveThreads) {
            phase3_solve(sm, t);
        } else {
            phase3_seed(sm, vec, tm, L, 2 * (part - 2), quarter, BT);
            phase3_seed(sm, vec, tm, L, 2 * (part - 2) + 1, quarter, BT);
            tmem_wait_st();
            if (t == kStorer) {
                if constexpr (kDyn) claim_raw = claim_async(sp.counter, !stop && n2 >= 0);   // resolved at the next top
                bulk_wait_read();   // the K~ piece has left the staging buffer ([Tb; M] goes there next)
                if constexpr (kDyn) {
                    if (pub2 >= 0) {   // the item two back: its pieces are older than the last three
                        bulk_wait_group<3>();
                        fence_proxy_async_global();
                        st_release_gpu(sp.flags + pub2, 1);
                    }
                    pub2 = pub1;
                    pub1 = item;
                }
            }
            if (has_next) {
                named_sync(2, kThreads - kSolveThreads);   // every seed has read this item's q and x
                if (t == kStorer) {
                    issue_qg_loads(p, sm, bar_qg, nxt.t0, nxt.h);
                    qg_pending = true;
                }
            }
        }
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        KDA_CLK(clk, 4);   // solve, with the seed, stores and publication alongside
        phase3_tb_operands(sm, t, sbeta);
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        KDA_CLK(clk, 5);   // Tb operands
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
        // [Tb; M] hi/lo: row L, K = tokens [16 part, +16), to TMEM (the D2 MMA) and the staging buffer
        uint32_t hi[8], lo[8];
        if (quarter < 2) {   // Tb rows (lanes 0-63) from the hi/lo B-operand tiles
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
        KDA_CLK(clk, 6);   // M = P Tb, Tb rows to TMEM
        if (quarter >= 2) {   // M rows (lanes 64-127), split into hi/lo
            float a[16];
            tmem_ld16(tmem_addr(tm, 32 * quarter, TM_M + 16 * part), a);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i) split_bf16x2(a[2 * i], a[2 * i + 1], hi[i], lo[i]);
            tmem_st8u(tmem_addr(tm, 32 * quarter, TM_TPH + 8 * part), hi);
            tmem_st8u(tmem_addr(tm, 32 * quarter, TM_TPL + 8 * part), lo);
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            st_shared_v4(sbase + A_STAGE + sw128_chunk(L, 2 * part + cc, 128), hi[4 * cc], hi[4 * cc + 1],
                         hi[4 * cc + 2], hi[4 * cc + 3]);
            st_shared_v4(sbase + A_STAGE + 16384 + sw128_chunk(L, 2 * part + cc, 128), lo[4 * cc], lo[4 * cc + 1],
                         lo[4 * cc + 2], lo[4 * cc + 3]);
        }
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before_sync();
        __syncthreads();
        KDA_CLK(clk, 7);   // M rows, [Tb; M] staged

        // ---- phase 4: D2 = [0; -Q_Gamma] + [Tb; M] K_Gamma (hi + lo) = [Wk; -Q']; A1 = -D2 to the image
        if (t == kStorer) {
            bulk_store(img + IMG_TBH, sm + A_STAGE, 32768);
            bulk_commit();
        }
        if (t == 0) {
            tc_fence_after_sync();
            const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + TM_D2, tm + TM_TPH + 8 * ks, desc_mnmajor(sbase + kg, 64, ks), idesc, 1u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + TM_D2, tm + TM_TPL + 8 * ks, desc_mnmajor(sbase + kg, 64, ks), idesc, 1u);
            umma_commit(bar_mma);
        }
        // the next item's phase 1 meanwhile.  It writes the g tile, vec, the X region, TMEM
        // columns [128, 256) and the other K_Gamma buffer, none of which this item still reads.
        if (has_next && !(ok = phase1ab(nxt, (li + 1) & 1))) break;
        KDA_CLK(clk, 8);   // the next item's phase 1 under the [Wk; -Q'] MMA
        if (t == kStorer) bulk_wait_read();   // the [Tb; M] piece has left the staging buffer
        if (!(ok = wait_all(bar_mma, mma_par, s_abort))) break;
        mma_par ^= 1u;
        tc_fence_after_sync();
        KDA_CLK(clk, 9);   // wait for it
        {   // row L, K = dk columns [32 part, +32).  The Q' rows' lo halves are staged in this
            // item's K_Gamma buffer, which the D2 MMA has finished reading (the next item's phase 1
            // wrote the other one); the buffer's next writer runs after the next item's first
            // bulk_wait_read, so the store below has left it by then.
            float a[32];
            tmem_ld32(tmem_addr(tm, 32 * quarter, TM_D2 + 32 * part), a);
            tmem_wait_ld();
            uint32_t pk[16], pl[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) split_bf16x2(-a[2 * i], -a[2 * i + 1], pk[i], pl[i]);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                st_shared_v4(sbase + A_STAGE + sw128_chunk(L, 4 * part + q, 128), pk[4 * q], pk[4 * q + 1],
                             pk[4 * q + 2], pk[4 * q + 3]);
            if (quarter >= 2) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    st_shared_v4(sbase + kg + sw128_chunk(L - 64, 4 * part + q, 64), pl[4 * q], pl[4 * q + 1],
                                 pl[4 * q + 2], pl[4 * q + 3]);
            }
            fence_proxy_async_smem();
        }
        __syncthreads();
        if (t == kStorer) {   // one bulk group, as the publication count expects three per item
            bulk_store(img + IMG_A1, sm + A_STAGE, 32768);
            bulk_store(img + IMG_QLO, sm + kg, 16384);
            bulk_commit();
        }
        KDA_CLK(clk, 10);   // [-Wk; Q'] hi and Q' lo staged
        KDA_CLK_COUNT(clk, 31);
        cur = nxt;   // the next item's first barrier orders these TMEM reads before its writes
        if (n2 >= 0) {   // its t0 and eos are read at the next item's top
            nxt.gc = n2 / H;
            nxt.h = n2 - nxt.gc * H;
        }
        item = nidx;
        nidx = n2;
    }

    if (t == kStorer) {
        bulk_wait_all();   // the images are written before the CTA's shared memory is reused
        if constexpr (kDyn) {
            if (ok) {
                fence_proxy_async_global();
                if (pub2 >= 0) st_release_gpu(sp.flags + pub2, 1);
                if (pub1 >= 0) st_release_gpu(sp.flags + pub1, 1);
            }
        }
    }
    if (!ok && t == 0) {
        report_status(p.status, kDevTimeout);
        mbar_wait_bounded(bar_mma, mma_par, kWaitNs);
    }
    if (!ok && t == kStorer) {
        if (k_pending) mbar_wait_bounded(bar_k, k_par, kWaitNs);
        if (qg_pending) mbar_wait_bounded(bar_qg, qg_par, kWaitNs);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (t == 0) {
        mbar_inval(bar_k);
        mbar_inval(bar_qg);
        mbar_inval(bar_mma);
    }
    __syncthreads();
}

template <bool kPro>
__global__ void __launch_bounds__(kThreads, 1) kda_chunk_prep_kernel(const __grid_constant__ SplitParams sp)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 32);
    if ((threadIdx.x >> 5) == 0) {
        tmem_alloc(tslot, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = *tslot;
    prep_items<false, kPro>(sp, sm, tm, 0x7fffffff);
    tc_fence_before_sync();
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) tmem_dealloc(tm, TM_COLS);
}

// ---------------------------------------------------------------- step 3: the state scan
// The scan of one (sequence, head) unit by one CTA.  It keeps the state transposed, S^T
// [128 dv lanes][128 dk] fp32 in tensor memory, and forms every product of a chunk step
// transposed, so that the operands the CUDA cores write (S^T hi/lo, W^T hi/lo) are A
// operands in tensor memory and the chunk's images, as they are, are the K-major B operands:
//   D1^T = V^T [Tb; M]^T (hi, lo)            A: v from shared memory (MN-major); B: [Tb; M]
//        + S^T_hi [-Wk; Q']^T + S^T_hi Q'_lo^T (the last into O's columns only, N = 64)
//        + S^T_lo [-Wk; Q']^T                A: S^T hi / lo from tensor memory; B: the images
//   S^T <- gamma_C S^T + W^T_hi K~_hi + W^T_lo K~_hi + W^T_hi K~_lo
//                                            A: W^T hi / lo from tensor memory; B: K~^T
// with D1^T [dv lanes][128]: columns 0-63 W^T (tokens), 64-127 O^T.  Each output element is
// the same sum of the same products as in the one-CTA-per-unit kernel.  Shared memory then
// carries only the images, v and two O staging buffers.  The CTA is split by role:
//   14 CUDA warps (all but kIssuerWarp and kProducerWarp; warp w reads TMEM lanes
//     [32 (w % 4), +32); 4 warps share a lane quarter's columns on lanes 0-63, 3 on lanes
//     64-127): per chunk, S^T_hi, then S^T_lo = bf16(S^T - S^T_hi) and S^T <- S^T gamma_C;
//     once D1 is in, W^T (hi + lo) into tensor memory and O (times sigmoid of the gate
//     logits, which the producer loaded into the same buffer) into staging buffer c % 2, once
//     the producer has taken chunk c-1's O; a sequence's ragged last chunk goes straight
//     from the registers to global memory;
//   lane 0 of kIssuerWarp issues every MMA: the S^T_hi products once S^T_hi is written, the
//     S^T_lo product once S^T_lo is, the state update once W^T is, and right behind it the
//     next chunk's V^T [Tb; M]^T (chunk 0's before the loop), which needs no state;
//   lane 0 of kProducerWarp issues every copy: [Tb; M] of chunk c+1 and v two chunks ahead
//     once chunk c's V^T [Tb; M]^T MMAs are done, the back image of c once the update of c-1
//     (which read the last one) is done, gamma_C of c+1 once S^T_lo of c is formed, [-Wk; Q'] and
//     Q' lo of c+1 once D1 of c is done; the images of chunk c+2 are prefetched into L2; chunk
//     c's staged O goes out by TMA store, after which the gate logits of c+1 go into the
//     buffer that chunk c-1's store has finished reading.
// The roles signal one another through mbarriers (one arrival per warp), never through a
// barrier of the whole CTA: issuing an MMA waits while the tensor pipe's queue is full, which
// then holds up no CUDA warp; the S^T_lo pass runs under the S^T_hi MMAs, the O stores under
// the state update.  Every wait is bounded and gives up early once another role has recorded
// an abort.  With kFlags (the single-launch form) each image is fetched only once its item's
// flag is set.  `tm`: 512 allocated TMEM columns.
constexpr int kIssuerWarp = 10, kProducerWarp = 11;
template <bool kFlags>
__device__ __forceinline__ void scan_unit(const SplitParams& sp, uint8_t* sm, uint32_t tm, int unit)
{
    const TcParams& p = sp.p;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + B_BAR + B_BARS);
    uint64_t* bar_f = bars + B_BAR_FRONT;          // [-Wk; Q'] and Q' lo are in
    uint64_t* bar_tb = bars + B_BAR_TB;            // [Tb; M] hi + lo are in
    uint64_t* bar_b = bars + B_BAR_BACK;           // K~^T hi + lo are in
    uint64_t* bar_v = bars + B_BAR_V;              // v, two, one per buffer
    uint64_t* bar_g = bars + B_BAR_GAMMA;          // gamma_C is in
    uint64_t* bar_mma = bars + B_BAR_MMA;          // D1 is done, then the state update
    uint64_t* bar_vdone = bars + B_BAR_VDONE;      // the V^T [Tb; M]^T MMAs are done
    uint64_t* bar_shi = bars + B_BAR_SHI;          // S^T_hi is written (14 warps)
    uint64_t* bar_slo = bars + B_BAR_SLO;          // S^T_lo is written and S^T decayed (14 warps)
    uint64_t* bar_wready = bars + B_BAR_WREADY;    // W^T is written (14 warps)
    uint64_t* bar_dread = bars + B_BAR_DREAD;      // D1 is read out (14 warps)
    uint64_t* bar_end = bars + B_BAR_END;          // the MMA issuer's last commit
    uint64_t* bar_ostaged = bars + B_BAR_OSTAGED;  // O is staged (14 warps)
    uint64_t* bar_sfree = bars + B_BAR_SFREE;      // a staged O taken; the buffer of the one before free
    uint64_t* bar_z = bars + B_BAR_Z;              // the gate logits are in an O staging buffer, two
    uint64_t* bar_upd = bars + B_BAR_UPD;          // the state update is done (the producer's copy of bar_mma's second phase)
    uint64_t* bar_d1p = bars + B_BAR_D1P;          // D1 is done (the producer's copy of bar_mma's first phase)
    int* s_abort = reinterpret_cast<int*>(sm + B_BAR + B_WORD_ABORT);
    const uint32_t sbase = smem_u32(sm);
    const float* sgam = reinterpret_cast<const float*>(sm + B_GAM);

    const int H = p.num_heads;
    const int n = unit / H, h = unit % H;
    int bos, eos;
    if (!seq_bounds(p.cu_seqlens, n, p.num_seqs, p.total_tokens, p.status, bos, eos)) return;
    const int nchunks = (eos - bos + 63) >> 6;
    const int gc0 = __ldg(sp.chunk_off + n);
    const size_t sbase_g = ((size_t)n * H + h) * 128 * 128;
    auto image = [&](int c) { return sp.ops + ((size_t)(gc0 + c) * H + h) * IMG_BYTES; };

    if (t == 0) {
        for (int i = 0; i < B_BAR_COUNT; ++i) {
            const bool all = i == B_BAR_SHI || i == B_BAR_SLO || i == B_BAR_WREADY || i == B_BAR_DREAD ||
                             i == B_BAR_OSTAGED;
            mbar_init(bars + i, all ? 14u : 1u);
        }
        mbar_fence_init();
        *s_abort = 0;
        tma_prefetch_desc(&p.tm_v);
        tma_prefetch_desc(&p.tm_o);
        if (p.gate) tma_prefetch_desc(&p.tm_z);
    }
    // initial state -> S^T in TMEM, all 16 warps: lane dv = 32 (w % 4) + laneid, dk columns
    // [32 (w / 4), +32); a warp reads one dk row's 32 consecutive dv values at a time
    {
        const int L = 32 * (warp & 3) + lane, c0 = 32 * (warp >> 2);
        float v[32];
        if (p.init_state) {
            const float* src = p.init_state + sbase_g + (size_t)c0 * 128 + L;
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __ldg(src + (size_t)i * 128);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        tmem_st32(tmem_addr(tm, 32 * (warp & 3), B_TM_S + c0), v);
        tmem_wait_st();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    // a snapshot of the state after `done` tokens is due when a full chunk ends there
    auto snapshot_due = [&](int done) {
        return p.checkpoints != nullptr && done > 0 && done % p.ckpt_interval == 0 &&
               done / p.ckpt_interval <= p.ckpt_slots;
    };
    // state element (dk, dv) of a snapshot slot: [dk][dv] fp32
    auto snapshot_at = [&](int done, int dk, int dv) {
        const int slot = done / p.ckpt_interval - 1;
        return p.checkpoints + (((size_t)n * H + h) * p.ckpt_slots + slot) * 128 * 128 + (size_t)dk * 128 + dv;
    };
    auto fail = [&]() { atomicExch(s_abort, 1); };
    KDA_CLK_DECL(clk);

    if (warp != kIssuerWarp && warp != kProducerWarp) {
        // ------------------------------------------------ the CUDA warps
        // a warp's columns as 16-column groups: S^T (dk) groups [sbeg, send) of 8; W^T (token)
        // groups [wbeg, wend) and O^T groups [obeg, oend) of 4 each.  Every warp loads the same
        // number of groups (the spare loads repeat its last one and are not used), which keeps
        // the loaded values in registers.
        const int quarter = warp & 3, slot = warp >> 2;
        const bool four = quarter < 2;   // lanes 0-63: 4 warps; lanes 64-127: 3 (the roles take one each)
        const int s3 = slot == 3 ? 2 : slot;
        const int sbeg = four ? 2 * slot : 3 * s3, send = four ? sbeg + 2 : min(sbeg + 3, 8);
        const int wbeg = four ? slot : (s3 == 0 ? 0 : s3 + 1), wend = four ? slot + 1 : (s3 == 0 ? 2 : s3 + 2);
        const int obeg = four ? slot : (s3 == 0 ? 0 : 2 * s3 - 1), oend = four ? slot + 1 : (s3 == 0 ? 1 : s3 == 1 ? 3 : 4);
        const int L = 32 * quarter + lane;   // dv
        const float* const gate = p.gate;
        uint32_t m_par = 0, g_par = 0, sf_par = 0, z_par = 0;   // z_par: bit b = buffer b's parity
        bool ok = true;
        for (int ci = 0; ci < nchunks && ok; ++ci) {
            const int t0 = bos + 64 * ci;
            const int BT = min(64, eos - t0);
            const bool snap = snapshot_due(64 * ci);   // the state entering this chunk
            if (ci > 0) {   // the last chunk's state update is done
                if (!(ok = role_wait(bar_mma, m_par, s_abort))) break;
                m_par ^= 1u;
            }
            tc_fence_after_sync();
            KDA_CLK(clk, 16);   // the last update waited for
            {
                float a[3][16];
#pragma unroll
                for (int jj = 0; jj < 3; ++jj)
                    tmem_ld16(tmem_addr(tm, 32 * quarter, B_TM_S + 16 * min(sbeg + jj, send - 1)), a[jj]);
                tmem_wait_ld();
#pragma unroll
                for (int jj = 0; jj < 3; ++jj) {   // S^T_hi: bf16 pairs along dk
                    const int j = sbeg + jj;
                    if (j < send) {
                        if (snap) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) *snapshot_at(64 * ci, 16 * j + i, L) = a[jj][i];
                        }
                        uint32_t hi[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) hi[i] = pack_bf16x2(a[jj][2 * i], a[jj][2 * i + 1]);
                        tmem_st8u(tmem_addr(tm, 32 * quarter, B_TM_SH + 8 * j), hi);
                    }
                }
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_shi);
                KDA_CLK(clk, 17);   // S^T_hi
                if (!(ok = role_wait(bar_g, g_par, s_abort))) break;   // gamma_C of this chunk
                g_par ^= 1u;
                // S^T again (nothing is held in registers across the wait)
#pragma unroll
                for (int jj = 0; jj < 3; ++jj)
                    tmem_ld16(tmem_addr(tm, 32 * quarter, B_TM_S + 16 * min(sbeg + jj, send - 1)), a[jj]);
                tmem_wait_ld();
#pragma unroll
                for (int jj = 0; jj < 3; ++jj) {   // S^T_lo = bf16(S^T - S^T_hi), then S^T <- S^T gamma_C
                    const int j = sbeg + jj;
                    if (j < send) {
                        uint32_t lo[8], d[16];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float2 h2 = bf2_to_f2(pack_bf16x2(a[jj][2 * i], a[jj][2 * i + 1]));
                            lo[i] = pack_bf16x2(a[jj][2 * i] - h2.x, a[jj][2 * i + 1] - h2.y);
                        }
                        tmem_st8u(tmem_addr(tm, 32 * quarter, B_TM_SL + 8 * j), lo);
#pragma unroll
                        for (int i = 0; i < 16; ++i) d[i] = __float_as_uint(a[jj][i] * sgam[16 * j + i]);
                        tmem_st16u(tmem_addr(tm, 32 * quarter, B_TM_S + 16 * j), d);
                    }
                }
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_slo);
                KDA_CLK(clk, 18);   // S^T_lo and the decay
            }
            if (!(ok = role_wait(bar_mma, m_par, s_abort))) break;   // D1
            m_par ^= 1u;
            tc_fence_after_sync();
            KDA_CLK(clk, 19);   // D1 waited for
            {
                float w[2][16];
#pragma unroll
                for (int jj = 0; jj < 2; ++jj)
                    tmem_ld16(tmem_addr(tm, 32 * quarter, B_TM_D1 + 16 * min(wbeg + jj, wend - 1)), w[jj]);
                tmem_wait_ld();
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {   // W^T (hi + lo): bf16 pairs along the tokens
                    const int j = wbeg + jj;
                    if (j < wend) {
                        uint32_t hi[8], lo[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) split_bf16x2(w[jj][2 * i], w[jj][2 * i + 1], hi[i], lo[i]);
                        tmem_st8u(tmem_addr(tm, 32 * quarter, B_TM_WH + 8 * j), hi);
                        tmem_st8u(tmem_addr(tm, 32 * quarter, B_TM_WL + 8 * j), lo);
                    }
                }
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_wready);   // W^T written
            }
            KDA_CLK(clk, 20);   // W^T split
            float o[2][16];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj)
                tmem_ld16(tmem_addr(tm, 32 * quarter, B_TM_D1 + 64 + 16 * min(obeg + jj, oend - 1)), o[jj]);
            tmem_wait_ld();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_dread);   // D1 read out: the next chunk's MMAs may overwrite it
            if (BT == 64) {   // O staged for the TMA store: token r, dv L in box L / 32 (a warp: one row per store)
                if (ci >= 1) {   // the last chunk's O is being stored, and the store of two chunks
                                 // back has read this buffer (the producer's arrival for chunk ci - 1)
                    if (!(ok = role_wait(bar_sfree, sf_par, s_abort))) break;
                    sf_par ^= 1u;
                }
                // (the parameters are read once: the asm stores' memory clobbers would reload them)
                const uint32_t box = sbase + B_OST + 32768u * (ci & 1) + 8192u * (L >> 5);
                if (gate) {   // the logits TMA put in the same positions of the buffer
                    if (!(ok = role_wait(bar_z + (ci & 1), (z_par >> (ci & 1)) & 1u, s_abort))) break;
                    z_par ^= 1u << (ci & 1);
                }
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int j = obeg + jj;
                    if (j < oend) {
                        uint32_t at[16];
                        float v[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            at[i] = box + sw128_off_f32(16 * j + i, L & 31, 64);
                            v[i] = o[jj][i];
                        }
                        if (gate) {   // out = o * sigmoid(z)
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] = gate1(v[i], ld_shared_f32(at[i]));
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) st_shared_f32(at[i], v[i]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_ostaged);
            } else {   // a sequence's ragged last chunk: direct stores, token t0 + r, dv L
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int j = obeg + jj;
                    if (j < oend) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int r = 16 * j + i;
                            if (r < BT) {
                                const size_t o0 = ((size_t)(t0 + r) * H + h) * 128 + L;
                                p.out[o0] = p.gate ? gate1(o[jj][i], __ldg(p.gate + o0)) : o[jj][i];
                            }
                        }
                    }
                }
            }
            KDA_CLK(clk, 21);   // O stored
            KDA_CLK_COUNT(clk, 30);
        }
        if (ok && nchunks > 0) {   // the last chunk's state update
            ok = role_wait(bar_mma, m_par, s_abort);
            m_par ^= 1u;
        }
        if (!ok) fail();
    } else if (t == 32 * kIssuerWarp) {
        // ------------------------------------------------ the MMA issuer
        uint32_t shi_par = 0, slo_par = 0, wr_par = 0, dr_par = 0, f_par = 0, tb_par = 0, b_par = 0, v_par = 0;
        bool ok = true;
        const uint32_t idesc_v = idesc_bf16_f32(128, 128, 1, 0);   // A (v) MN-major, B K-major
        const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
        const uint32_t idesc64 = idesc_bf16_f32(128, 64, 0, 0);
        const uint32_t d1 = tm + B_TM_D1;
        // V^T [Tb; M]^T (hi, lo) of chunk c into D1: needs chunk c's [Tb; M] and v, and chunk
        // c-1's D1 read out.  It depends on no state, so chunk c+1's is issued right behind
        // chunk c's state update, and runs while the CUDA warps wait for that update and form
        // S^T_hi: the tensor pipe is then free for the S^T_hi products as soon as they can go.
        auto issue_v = [&](int c) -> bool {
            const int vb = c & 1;
            if (c > 0) {
                if (!role_wait(bar_dread, dr_par, s_abort)) return false;
                dr_par ^= 1u;
            }
            if (!(role_wait(bar_tb, tb_par, s_abort) && role_wait(bar_v + vb, (v_par >> vb) & 1u, s_abort)))
                return false;
            tb_par ^= 1u;
            v_par ^= 1u << vb;
            tc_fence_after_sync();
            const uint32_t vt = sbase + (vb ? B_V1 : B_V0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16(d1, desc_mnmajor(vt, 64, ks), desc_kmajor(sbase + B_TBH, 128, ks), idesc_v, ks > 0 ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16(d1, desc_mnmajor(vt, 64, ks), desc_kmajor(sbase + B_TBL, 128, ks), idesc_v, 1u);
            umma_commit(bar_vdone);
            return true;
        };
        if (nchunks > 0) ok = issue_v(0);
        for (int ci = 0; ci < nchunks && ok; ++ci) {
            // S^T_hi [-Wk; Q']^T, and S^T_hi Q'_lo^T into O's columns, once S^T_hi is written
            if (!(ok = role_wait(bar_shi, shi_par, s_abort) && role_wait(bar_f, f_par, s_abort))) break;
            shi_par ^= 1u;
            f_par ^= 1u;
            tc_fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                umma_bf16_tmem_a(d1, tm + B_TM_SH + 8 * ks, desc_kmajor(sbase + B_A1, 128, ks), idesc, 1u);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                umma_bf16_tmem_a(d1 + 64, tm + B_TM_SH + 8 * ks, desc_kmajor(sbase + B_QLO, 64, ks), idesc64, 1u);
            // S^T_lo [-Wk; Q']^T, once S^T_lo is written
            if (!(ok = role_wait(bar_slo, slo_par, s_abort))) break;
            slo_par ^= 1u;
            tc_fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                umma_bf16_tmem_a(d1, tm + B_TM_SL + 8 * ks, desc_kmajor(sbase + B_A1, 128, ks), idesc, 1u);
            umma_commit(bar_mma);
            umma_commit(bar_d1p);   // the same MMAs, for the producer
            // S^T += W^T_hi K~_hi + W^T_lo K~_hi + W^T_hi K~_lo, once W^T is written
            if (!(ok = role_wait(bar_wready, wr_par, s_abort) && role_wait(bar_b, b_par, s_abort))) break;
            wr_par ^= 1u;
            b_par ^= 1u;
            tc_fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + B_TM_S, tm + B_TM_WH + 8 * ks, desc_kmajor(sbase + B_KTH, 128, ks), idesc, 1u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + B_TM_S, tm + B_TM_WL + 8 * ks, desc_kmajor(sbase + B_KTH, 128, ks), idesc, 1u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16_tmem_a(tm + B_TM_S, tm + B_TM_WH + 8 * ks, desc_kmajor(sbase + B_KTL, 128, ks), idesc, 1u);
            umma_commit(bar_mma);
            umma_commit(bar_upd);   // the same MMAs, for the producer
            if (ci + 1 < nchunks && !(ok = issue_v(ci + 1))) break;
        }
        if (!ok) fail();
        // every MMA issued has completed before the CTA moves on (bounded)
        umma_commit(bar_end);
        if (!mbar_wait_bounded(bar_end, 0u, kWaitNs)) fail();
    } else if (t == 32 * kProducerWarp) {
        // ------------------------------------------------ the copy producer
        // kFlags: chunk c's images are fetched only once its item is published.  The flags of up
        // to 16 chunks ahead are read with relaxed loads and one acquire (and proxy) fence covers
        // all that are set, so that a fence is paid per batch, not per fetch; the producer
        // blocks (bounded) only when chunk c itself is not yet published.
        int known = -1;   // chunks <= known are published and acquired
        auto ready = [&](int c) {
            if constexpr (kFlags) {
                if (c <= known) return true;
                const int* f = sp.flags + (size_t)gc0 * H + h;
                if (!ld_relaxed_gpu(f + (size_t)c * H) && !wait_flag(f + (size_t)c * H)) return false;
                int fl[15];   // the next 15 chunks' flags, loaded together
#pragma unroll
                for (int i = 0; i < 15; ++i)
                    fl[i] = (c + 1 + i < nchunks) ? ld_relaxed_gpu(f + (size_t)(c + 1 + i) * H) : 0;
                int k = c;
#pragma unroll
                for (int i = 0; i < 15; ++i)
                    if (k == c + i && fl[i]) k = c + 1 + i;
                fence_acquire_gpu();
                fence_proxy_async_global();
                known = k;
            }
            return true;
        };
        int n_front = 0, n_tb = 0, n_back = 0, n_gam = 0, n_v[2] = {0, 0}, n_z[2] = {0, 0};
        auto fetch_z = [&](int c) {   // a full chunk's gate logits into its O staging buffer (free by now)
            if (p.gate && c < nchunks && eos - (bos + 64 * c) >= 64) {
                uint64_t* bar = bar_z + (c & 1);
                mbar_arrive_expect_tx(bar, 32768u);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    tma_load_3d(sm + B_OST + 32768u * (c & 1) + 8192 * j, &p.tm_z, bar, 32 * j, h, bos + 64 * c);
                if (c & 1) ++n_z[1];
                else ++n_z[0];
            }
        };
        auto fetch_gamma = [&](int c) {   // gamma_C: read by the S^T_lo pass
            if (!ready(c)) return false;
            mbar_arrive_expect_tx(bar_g, 512u);
            bulk_load(sm + B_GAM, image(c) + IMG_GAM, 512u, bar_g);
            ++n_gam;
            return true;
        };
        auto fetch_tb = [&](int c) {   // [Tb; M] hi + lo: read by the V^T [Tb; M]^T MMAs
            if (!ready(c)) return false;
            mbar_arrive_expect_tx(bar_tb, 32768u);
            bulk_load(sm + B_TBH, image(c) + IMG_TBH, 32768u, bar_tb);
            ++n_tb;
            return true;
        };
        auto fetch_front = [&](int c) {   // [-Wk; Q'] and Q' lo: read by the S^T MMAs of D1
            if (!ready(c)) return false;
            mbar_arrive_expect_tx(bar_f, 32768u + 16384u);
            bulk_load(sm + B_A1, image(c), 32768u, bar_f);
            bulk_load(sm + B_QLO, image(c) + IMG_QLO, 16384u, bar_f);
            ++n_front;
            return true;
        };
        auto fetch_back = [&](int c) {   // K~^T hi + lo: read by the state update
            if (!ready(c)) return false;
            mbar_arrive_expect_tx(bar_b, IMG_BACK);
            bulk_load(sm + B_KTH, image(c) + IMG_KTH, IMG_BACK, bar_b);
            ++n_back;
            return true;
        };
        auto fetch_v = [&](int c) {   // [64 tok][128 ch] as two 64-channel TMA boxes
            uint64_t* bar = bar_v + (c & 1);
            uint8_t* dst = sm + ((c & 1) ? B_V1 : B_V0);
            mbar_arrive_expect_tx(bar, 16384u);
            tma_load_3d(dst, &p.tm_v, bar, 0, h, bos + 64 * c);
            tma_load_3d(dst + 8192, &p.tm_v, bar, 64, h, bos + 64 * c);
            if (c & 1) ++n_v[1];
            else ++n_v[0];
        };
        bool ok = true;
        if (nchunks > 0) {
            ok = fetch_tb(0) && fetch_gamma(0) && fetch_front(0) && fetch_back(0);
            fetch_v(0);
            fetch_z(0);
            fetch_z(1);
            if (nchunks > 1) {
                fetch_v(1);
                prefetch_l2(image(1), IMG_BYTES);
            }
        }
        uint32_t vd_par = 0, slo_par = 0, d1_par = 0, os_par = 0, upd_par = 0;
        for (int ci = 0; ci < nchunks && ok; ++ci) {
            const int t0 = bos + 64 * ci;
            const bool full = eos - t0 >= 64;
            // the last chunk's state update is done: it has read the back image, whose copy for
            // this chunk goes out first (the update waits for it at the end of the chunk).
            // Chunk ci's update needs this copy, so bar_upd cannot run a phase ahead of here.
            if (ci > 0) {
                if (!(ok = role_wait(bar_upd, upd_par, s_abort))) break;
                upd_par ^= 1u;
                if (!(ok = fetch_back(ci))) break;
            }
            // the V^T [Tb; M]^T MMAs are done: [Tb; M] and this v buffer have been read
            if (!(ok = role_wait(bar_vdone, vd_par, s_abort))) break;
            vd_par ^= 1u;
            if (ci + 1 < nchunks && !(ok = fetch_tb(ci + 1))) break;
            if (ci + 2 < nchunks) {
                fetch_v(ci + 2);
                prefetch_l2(image(ci + 2), IMG_BYTES);   // so that the next fetches come from L2
            }
            // S^T_lo is formed: gamma_C has been read
            if (!(ok = role_wait(bar_slo, slo_par, s_abort))) break;
            slo_par ^= 1u;
            if (ci + 1 < nchunks && !(ok = fetch_gamma(ci + 1))) break;
            // D1 is done: [-Wk; Q'] and Q' lo have been read.  (Chunk ci+1's D1 needs the copy
            // made here, so bar_d1p cannot run a phase ahead of this wait.)
            if (!(ok = role_wait(bar_d1p, d1_par, s_abort))) break;
            d1_par ^= 1u;
            if (ci + 1 < nchunks && !(ok = fetch_front(ci + 1))) break;
            if (p.gate && ci + 2 < nchunks) {   // the gate logits of two chunks ahead into L2
#pragma unroll
                for (int j = 0; j < 4; ++j) tma_prefetch_3d(&p.tm_z, 32 * j, h, t0 + 128);
            }
            if (full) {   // O staged: stored from its buffer; the last chunk's buffer is then free once read
                if (!(ok = role_wait(bar_ostaged, os_par, s_abort))) break;
                os_par ^= 1u;
                uint8_t* buf = sm + B_OST + 32768u * (ci & 1);
#pragma unroll
                for (int j = 0; j < 4; ++j) tma_store_3d(&p.tm_o, buf + 8192 * j, 32 * j, h, t0);
                bulk_commit();
                if (ci >= 1) {
                    bulk_wait_read_group<1>();
                    fetch_z(ci + 1);   // into the buffer the store of chunk ci - 1 has just read
                }
                // one arrival per full chunk, waited for by the CUDA warps before they stage the
                // next chunk: they never stage chunk ci + 1 (and arrive on ostaged again) before
                // this thread has taken chunk ci's arrivals, so neither barrier runs two phases
                // ahead of its waiter
                mbar_arrive(bar_sfree);
            }
        }
        bulk_wait_all();   // the staged O fully written before the CTA's shared memory goes away
        if (!ok) {   // record it, and let the copies in flight land (bounded): the last on each barrier
            fail();
            if (n_front > 0) mbar_wait_bounded(bar_f, (uint32_t)(n_front - 1) & 1u, kWaitNs);
            if (n_tb > 0) mbar_wait_bounded(bar_tb, (uint32_t)(n_tb - 1) & 1u, kWaitNs);
            if (n_back > 0) mbar_wait_bounded(bar_b, (uint32_t)(n_back - 1) & 1u, kWaitNs);
            if (n_gam > 0) mbar_wait_bounded(bar_g, (uint32_t)(n_gam - 1) & 1u, kWaitNs);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                if (n_v[i] > 0) mbar_wait_bounded(bar_v + i, (uint32_t)(n_v[i] - 1) & 1u, kWaitNs);
                if (n_z[i] > 0) mbar_wait_bounded(bar_z + i, (uint32_t)(n_z[i] - 1) & 1u, kWaitNs);
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const bool ok = *reinterpret_cast<volatile int*>(s_abort) == 0;
    if (ok) {   // the last chunk's snapshot, if due, and the final state: all 16 warps
        const int L = 32 * (warp & 3) + lane, c0 = 32 * (warp >> 2);
        const bool snap = nchunks > 0 && eos - bos == 64 * nchunks && snapshot_due(64 * nchunks);
        if (snap || p.final_state) {
            float v[32];
            tmem_ld32(tmem_addr(tm, 32 * (warp & 3), B_TM_S + c0), v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (snap) *snapshot_at(64 * nchunks, c0 + i, L) = v[i];
                if (p.final_state) p.final_state[sbase_g + (size_t)(c0 + i) * 128 + L] = v[i];
            }
        }
    } else if (t == 0) {
        report_status(p.status, kDevTimeout);
    }
    tc_fence_before_sync();
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1) kda_state_scan_kernel(const __grid_constant__ SplitParams sp)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + B_BAR + B_WORD_TSLOT);
    if ((threadIdx.x >> 5) == 0) {
        tmem_alloc(tslot, B_TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = *tslot;
    // the units longest sequence first (the scratch: the O staging, unused until the scan)
    const int H = sp.p.num_heads;
    const int n = unit_sequence(sp.p.cu_seqlens, sp.p.num_seqs, (int)blockIdx.x / H, reinterpret_cast<int*>(sm + B_OST));
    scan_unit<false>(sp, sm, tm, n * H + (int)blockIdx.x % H);
    tc_fence_before_sync();
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) tmem_dealloc(tm, B_TM_COLS);
}

// The single-launch form (cooperative: every CTA resident, one per SM).  Every CTA claims
// chunk-prep items in increasing order; CTAs b < units stop claiming at `switch_item` and
// then scan unit b, fetching each chunk's images once its flag is set, while the others
// keep claiming until the items run out.  A CTA waits only on items that other CTAs have
// already claimed or will claim, and the CTAs that never scan finish every item left, so
// every wait ends.
template <bool kPro>
__global__ void __launch_bounds__(kThreads, 1) kda_prep_scan_kernel(const __grid_constant__ SplitParams sp, int units,
                                                                    int switch_item)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + B_BAR + B_WORD_TSLOT1);   // used by neither layout
    if ((threadIdx.x >> 5) == 0) {
        tmem_alloc(tslot, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = *tslot;
    const bool scans = (int)blockIdx.x < units;
    prep_items<true, kPro>(sp, sm, tm, scans ? switch_item : 0x7fffffff);
    if (scans) scan_unit<true>(sp, sm, tm, blockIdx.x);
    tc_fence_before_sync();
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) tmem_dealloc(tm, TM_COLS);
}

// workspace: chunk_off [N + 1] int32, chunk_info [chunks] int2, the claim counter, the item
// flags [chunks * H] int32, then the operand images
struct SplitWorkspace {
    size_t chunks, off_bytes, info_bytes, ctr_bytes, flag_bytes, total;
};

SplitWorkspace split_workspace(int num_seqs, int total_tokens, int num_heads)
{
    SplitWorkspace w;
    w.chunks = (size_t)total_tokens / 64 + (size_t)num_seqs;   // >= the sum of ceil(len / 64)
    w.off_bytes = ((size_t)(num_seqs + 1) * sizeof(int32_t) + 255) & ~(size_t)255;
    w.info_bytes = (w.chunks * sizeof(int2) + 255) & ~(size_t)255;
    w.ctr_bytes = 256;
    w.flag_bytes = (w.chunks * (size_t)num_heads * sizeof(int) + 255) & ~(size_t)255;
    w.total = w.off_bytes + w.info_bytes + w.ctr_bytes + w.flag_bytes + w.chunks * (size_t)num_heads * IMG_BYTES;
    return w;
}

}  // namespace

size_t prefill_split_workspace_bytes(int num_seqs, int total_tokens, int num_heads)
{
    return split_workspace(num_seqs, total_tokens, num_heads).total;
}

// Per-device facts the launch needs, found once: SM count and whether the single-launch
// form can run (cooperative launch, one resident CTA per SM).
struct SplitDevice {
    int sms = 0;
    bool single = false;
};

cudaError_t split_device(SplitDevice* out)
{
    static SplitDevice cache[64];
    static std::once_flag once[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [dev] {
        SplitDevice d;
        int coop = 0, per_sm = 0, per_sm_pro = 0;
        bool ok = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess &&
                  cudaFuncSetAttribute(kda_chunk_prep_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)A_SMEM_BYTES) == cudaSuccess &&
                  cudaFuncSetAttribute(kda_chunk_prep_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)A_SMEM_BYTES) == cudaSuccess &&
                  cudaFuncSetAttribute(kda_state_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)B_SMEM_BYTES) == cudaSuccess &&
                  cudaFuncSetAttribute(kda_prep_scan_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)B_SMEM_BYTES) == cudaSuccess &&
                  cudaFuncSetAttribute(kda_prep_scan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)B_SMEM_BYTES) == cudaSuccess &&
                  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_prep_scan_kernel<false>, kThreads,
                                                                B_SMEM_BYTES) == cudaSuccess &&
                  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_pro, kda_prep_scan_kernel<true>, kThreads,
                                                                B_SMEM_BYTES) == cudaSuccess;
        d.single = ok && coop && per_sm >= 1 && per_sm_pro >= 1;
        if (!ok) d.sms = 0;
        cache[dev] = d;
    });
    *out = cache[dev];
    return out->sms > 0 ? cudaSuccess : cudaErrorUnknown;
}

cudaError_t launch_prefill_split(const PrefillArgs& a, cudaStream_t stream)
{
    SplitParams sp;
    memset(&sp, 0, sizeof(sp));
    TcParams& p = sp.p;
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
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    const SplitWorkspace wl = split_workspace(a.num_seqs, a.total_tokens, a.num_heads);
    sp.chunk_off = reinterpret_cast<int32_t*>(ws);
    sp.chunk_info = reinterpret_cast<int2*>(ws + wl.off_bytes);
    sp.counter = reinterpret_cast<int*>(ws + wl.off_bytes + wl.info_bytes);
    sp.flags = reinterpret_cast<int*>(ws + wl.off_bytes + wl.info_bytes + wl.ctr_bytes);
    sp.num_flags = (int)(wl.chunks * (size_t)a.num_heads);
    sp.ops = ws + wl.off_bytes + wl.info_bytes + wl.ctr_bytes + wl.flag_bytes;

    SplitDevice dv;
    cudaError_t e = split_device(&dv);
    if (e != cudaSuccess) return e;

    kda_chunk_offsets_kernel<<<1, 1024, 0, stream>>>(a.cu_seqlens, a.num_seqs, a.total_tokens, sp.chunk_off,
                                                      sp.chunk_info, sp.counter, sp.flags, sp.num_flags, a.status);
    const long long units = (long long)a.num_seqs * a.num_heads;
    if (dv.single && units + kSingleMinProducers <= dv.sms) {
        // Scanning CTAs stop claiming items once (grid - units) producers alone can finish the
        // rest in the time the scan takes: rest = (grid - units) x chunks x scan / prep per item.
        const long long chunks = ((long long)a.total_tokens / a.num_seqs + 63) / 64;
        const long long items = chunks * a.num_seqs * a.num_heads;
        const long long prep = a.prologue ? kPrepCyclesPerItemPrologue : kPrepCyclesPerItem;
        const long long rest = (dv.sms - units) * chunks * kScanCyclesPerChunk / prep;
        int units_i = (int)units, switch_item = (int)std::max(0LL, items - rest);
        void* args[] = {&sp, &units_i, &switch_item};
        const void* kern = a.prologue ? (const void*)kda_prep_scan_kernel<true> : (const void*)kda_prep_scan_kernel<false>;
        e = cudaLaunchCooperativeKernel(kern, dim3((unsigned)dv.sms), dim3(kThreads), args, B_SMEM_BYTES, stream);
        if (e == cudaSuccess) return cudaGetLastError();
        if (e != cudaErrorCooperativeLaunchTooLarge) return e;
        (void)cudaGetLastError();   // not all CTAs can be resident here: the separate launches below
    }
    const long long items_max = ((long long)a.total_tokens / 64 + a.num_seqs) * a.num_heads;
    const long long prep_grid = std::max(1LL, std::min<long long>(dv.sms, items_max));
    if (a.prologue)
        kda_chunk_prep_kernel<true><<<(unsigned)prep_grid, kThreads, A_SMEM_BYTES, stream>>>(sp);
    else
        kda_chunk_prep_kernel<false><<<(unsigned)prep_grid, kThreads, A_SMEM_BYTES, stream>>>(sp);
    kda_state_scan_kernel<<<(unsigned)units, kThreads, B_SMEM_BYTES, stream>>>(sp);
    return cudaGetLastError();
}

}  // namespace kda

#ifdef KDA_PHASE_CLOCKS
// Instrumented build only: copy out and clear this file's cycle marks (kClockSlots values).
extern "C" int kda_phase_clocks_split(unsigned long long* out)
{
    if (cudaMemcpyFromSymbol(out, kda::phase_clock_slots, sizeof(kda::phase_clock_slots)) != cudaSuccess) return -1;
    static const unsigned long long zero[kda::kClockSlots] = {};
    return cudaMemcpyToSymbol(kda::phase_clock_slots, zero, sizeof(zero)) == cudaSuccess ? 0 : -1;
}
#endif
