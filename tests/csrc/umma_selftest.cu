// Self-test of the library's tcgen05 primitives: one 128x128 tile D = C (+/-) A*B with
// A, B staged in 128-byte-swizzled shared memory in K-major or MN-major form, the
// accumulator in TMEM, read back with tcgen05.ld.  Test infrastructure only.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_sm100.cuh"

using namespace kda::sm100;

// mode 0: A K-major [128][K], B K-major [128][K]      (D = A * B_nk^T)
// mode 1: A K-major [128][K], B MN-major [K][128]
// mode 2: A MN-major [K][128], B MN-major [K][128]
// mode 3: as mode 1, with D preloaded from C through tcgen05.st and A negated: D = C - A*B
// mode 4: as mode 1, with A read from TMEM (row m in lane m, bf16 pairs per column)
// mode 5: M = 64, A K-major [64][K], B MN-major; all 128 lanes are read back so the
//         test can locate the 64 result rows
__global__ void __launch_bounds__(128, 1) umma_selftest_kernel(const __nv_bfloat16* A, const __nv_bfloat16* B,
                                                               const float* C, float* D, int K, int mode, int* err)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + 128 * K * 2;
    __shared__ uint64_t bar;
    __shared__ uint32_t tslot;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const bool a_mn = (mode == 2), b_mn = (mode != 0);
    const int M = (mode == 5) ? 64 : 128;

    for (int idx = t; idx < 128 * K; idx += 128) {
        // A(m, k)
        const int m = idx / K, k = idx % K;
        if (m < M) {
            const __nv_bfloat16 av = a_mn ? A[k * 128 + m] : A[m * K + k];
            const uint32_t aoff = a_mn ? sw128_off(k, m, K) : sw128_off(m, k, M);
            *reinterpret_cast<__nv_bfloat16*>(sA + aoff) = av;
        }
        // B(n, k)
        const int n = m;
        const __nv_bfloat16 bv = b_mn ? B[k * 128 + n] : B[n * K + k];
        const uint32_t boff = b_mn ? sw128_off(k, n, K) : sw128_off(n, k, 128);
        *reinterpret_cast<__nv_bfloat16*>(sB + boff) = bv;
    }
    fence_proxy_async_smem();
    if (t == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(&tslot, 256);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t base = tslot;
    const uint32_t row = 32 * warp + lane;

    if (mode == 3) {
        for (int c0 = 0; c0 < 128; c0 += 32) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = C[row * 128 + c0 + i];
            tmem_st32(tmem_addr(base, 32 * warp, c0), v);
        }
        tmem_wait_st();
    }
    if (mode == 4) {
        // A row `row` into TMEM columns [128, 128 + K/2) of lane `row`
        for (int c0 = 0; c0 < K / 2; c0 += 16) {
            uint32_t r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int k = 2 * (c0 + i);
                r[i] = pack_bf16x2(__bfloat162float(A[row * K + k]), __bfloat162float(A[row * K + k + 1]));
            }
            tmem_st16u(tmem_addr(base, 32 * warp, 128 + c0), r);
        }
        tmem_wait_st();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    if (t == 0) {
        const uint32_t idesc = idesc_bf16_f32(M, 128, a_mn ? 1 : 0, b_mn ? 1 : 0, mode == 3 ? 1 : 0);
        const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
        for (int ks = 0; ks < K / 16; ++ks) {
            const uint64_t ad = a_mn ? desc_mnmajor(a0, K, ks) : desc_kmajor(a0, M, ks);
            const uint64_t bd = b_mn ? desc_mnmajor(b0, K, ks) : desc_kmajor(b0, 128, ks);
            if (mode == 4)
                umma_bf16_tmem_a(base, base + 128 + 8 * ks, bd, idesc, ks > 0 ? 1u : 0u);
            else
                umma_bf16(base, ad, bd, idesc, (ks > 0 || mode == 3) ? 1u : 0u);
        }
        umma_commit(&bar);
    }
    if (!mbar_wait_bounded(&bar, 0, 1000000000ull)) atomicExch(err, 1);
    tc_fence_after_sync();
    for (int c0 = 0; c0 < 128; c0 += 32) {
        float v[32];
        tmem_ld32(tmem_addr(base, 32 * warp, c0), v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) D[row * 128 + c0 + i] = v[i];
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(base, 256);
}

// kind::tf32 self-test: A [128][K] fp32, B [128][K] fp32 (both K-major, B given as N x K),
// D = A * B_nk^T.  a_tmem: A read from TMEM (one fp32 per column) instead of shared memory.
__global__ void __launch_bounds__(128, 1) umma_tf32_kernel(const float* A, const float* B, float* D, int K,
                                                           int a_tmem, int* err)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + 128 * K * 4;
    __shared__ uint64_t bar;
    __shared__ uint32_t tslot;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    for (int idx = t; idx < 128 * K; idx += 128) {
        const int m = idx / K, k = idx % K;
        *reinterpret_cast<float*>(sA + sw128_off_f32(m, k, 128)) = A[m * K + k];
        *reinterpret_cast<float*>(sB + sw128_off_f32(m, k, 128)) = B[m * K + k];
    }
    fence_proxy_async_smem();
    if (t == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(&tslot, 256);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t base = tslot;
    const uint32_t row = 32 * warp + lane;
    if (a_tmem) {
        for (int c0 = 0; c0 < K; c0 += 32) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = A[row * K + c0 + i];
            tmem_st32(tmem_addr(base, 32 * warp, 128 + c0), v);
        }
        tmem_wait_st();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (t == 0) {
        const uint32_t idesc = idesc_tf32_f32(128, 128);
        const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
        for (int ks = 0; ks < K / 8; ++ks) {
            const uint64_t bd = desc_kmajor(b0, 128, ks);
            if (a_tmem)
                umma_tf32_tmem_a(base, base + 128 + 8 * ks, bd, idesc, ks > 0 ? 1u : 0u);
            else
                umma_tf32(base, desc_kmajor(a0, 128, ks), bd, idesc, ks > 0 ? 1u : 0u);
        }
        umma_commit(&bar);
    }
    if (!mbar_wait_bounded(&bar, 0, 1000000000ull)) atomicExch(err, 1);
    tc_fence_after_sync();
    for (int c0 = 0; c0 < 128; c0 += 32) {
        float v[32];
        tmem_ld32(tmem_addr(base, 32 * warp, c0), v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) D[row * 128 + c0 + i] = v[i];
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(base, 256);
}

extern "C" int umma_tf32_selftest(const void* A, const void* B, void* D, int K, int a_tmem, int* err)
{
    const size_t smem = 2 * 128 * K * 4 + 1024;
    if (cudaFuncSetAttribute(umma_tf32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return -1;
    umma_tf32_kernel<<<1, 128, smem>>>(static_cast<const float*>(A), static_cast<const float*>(B),
                                       static_cast<float*>(D), K, a_tmem, err);
    if (cudaGetLastError() != cudaSuccess) return -2;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -3;
}

extern "C" int umma_selftest(const void* A, const void* B, const void* C, void* D, int K, int mode, int* err)
{
    const size_t smem = 2 * 128 * K * 2 + 1024;
    if (cudaFuncSetAttribute(umma_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return -1;
    umma_selftest_kernel<<<1, 128, smem>>>(static_cast<const __nv_bfloat16*>(A),
                                           static_cast<const __nv_bfloat16*>(B), static_cast<const float*>(C),
                                           static_cast<float*>(D), K, mode, err);
    if (cudaGetLastError() != cudaSuccess) return -2;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -3;
}
