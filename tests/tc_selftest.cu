// Self-test of the tcgen05 helpers (kda_tcgen05.cuh): one CTA issues an
// M x N x K tensor-core MMA (M = 64 or 128) from shared-memory tiles in the
// no-swizzle core-matrix layouts and writes all 128 TMEM lanes of the first
// N columns back, so that the test sees where each row of D lands. Built and
// called only by tests/test_tcgen05_layouts.py.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_common.cuh"
#include "kda_tcgen05.cuh"

using namespace kda;
using namespace kda::tc;

__global__ void __launch_bounds__(128, 1)
    tc_selftest_kernel(const uint16_t *__restrict__ A, const uint16_t *__restrict__ B,
                       float *__restrict__ D, int M, int N, int K, int a_mn, int b_mn, int f16,
                       int mn_swap, int *err) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_base;
    unsigned char *sA = smem;
    unsigned char *sB = smem + 128 * 128 * 2;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    uint32_t lboA = 128, sboA = (uint32_t)(K / 8) * 128;      // K-major A (M x K)
    if (a_mn) { lboA = (uint32_t)(M / 8) * 128; sboA = 128; } // MN-major: M groups adjacent
    uint32_t lboB = 128, sboB = (uint32_t)(K / 8) * 128;     // K-major B (N x K)
    if (b_mn) { lboB = (uint32_t)(N / 8) * 128; sboB = 128; } // MN-major: N groups adjacent
    if (!a_mn) {
        for (int i = tid; i < M * K; i += blockDim.x) {  // A given as A[M][K]
            const int r = i / K, k = i % K;
            *reinterpret_cast<uint16_t *>(sA + kmajor_off(r, k, lboA, sboA)) = A[i];
        }
    } else {
        for (int i = tid; i < K * M; i += blockDim.x) {  // A given as At[K][M]
            const int k = i / M, r = i % M;
            *reinterpret_cast<uint16_t *>(sA + mnmajor_off(k, r, lboA, sboA)) = A[i];
        }
    }
    if (!b_mn) {
        for (int i = tid; i < N * K; i += blockDim.x) {  // B given as Bt[N][K]
            const int n = i / K, k = i % K;
            *reinterpret_cast<uint16_t *>(sB + kmajor_off(n, k, lboB, sboB)) = B[i];
        }
    } else {
        for (int i = tid; i < K * N; i += blockDim.x) {  // B given as B[K][N]
            const int k = i / N, n = i % N;
            *reinterpret_cast<uint16_t *>(sB + mnmajor_off(k, n, lboB, sboB)) = B[i];
        }
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_base), 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = tmem_base;
    {  // zero every lane of the N result columns: lanes the MMA does not write
       // (M = 64) then read as 0, not as what an earlier kernel left in TMEM
        const float zero[16] = {};
        for (int c = 0; c < N; c += 16) tmem_st16(tm + ((uint32_t)(32 * warp) << 16) + (uint32_t)c, zero);
        tmem_wait_st();
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
        const uint32_t idesc = idesc_f16(M, N, f16, a_mn, b_mn);
        // descriptor fields for B; mn_swap = 1 passes them in the opposite
        // order (the test shows that order is wrong)
        const uint32_t dlbo = (b_mn && mn_swap) ? sboB : lboB;
        const uint32_t dsbo = (b_mn && mn_swap) ? lboB : sboB;
        for (int ks = 0; ks < K / 16; ++ks) {
            const uint64_t da = smem_desc(smem_u32(sA) + ks * 2 * lboA, lboA, sboA);  // 2 k groups
            const uint32_t bstep = 2 * lboB;  // two core matrices along K
            const uint64_t db = smem_desc(smem_u32(sB) + ks * bstep, dlbo, dsbo);
            mma_f16(tm, da, db, idesc, ks > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&bar));
    }
    const bool ok = mbar_wait(smem_u32(&bar), 0, 1000000000ull);
    if (!ok && lane == 0) atomicOr(err, 1);
    fence_after_sync();
    if (ok) {
        for (int c = 0; c < N; c += 16) {
            float v[16];
            tmem_ld16(tm + ((uint32_t)(32 * warp) << 16) + (uint32_t)c, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) D[(32 * warp + lane) * N + c + j] = v[j];
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 256);
}

extern "C" int tc_selftest(const void *A, const void *B, float *D, int M, int N, int K, int a_mn,
                           int b_mn, int f16, int mn_swap, int *err) {
    if (M != 64 && M != 128) return 1;
    if (N < 16 || N > 256 || N % 16 || K < 16 || K > 128 || K % 16) return 1;
    // The whole 227 KB window is allocated so that a descriptor read with the
    // byte-offset fields in either order stays inside this CTA's shared memory.
    const int smem = 220 * 1024;
    if (cudaFuncSetAttribute(tc_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
        return 2;
    tc_selftest_kernel<<<1, 128, smem>>>(static_cast<const uint16_t *>(A),
                                         static_cast<const uint16_t *>(B), D, M, N, K, a_mn, b_mn,
                                         f16, mn_swap, err);
    if (cudaGetLastError() != cudaSuccess) return 3;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : 4;
}
