// Shared device helpers of libkda: warp-level bf16 tensor-core fragments,
// ldmatrix loads, bf16 packing, and the status word of a call.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

constexpr int kD = 128;          // head dimension (d_k = d_v)
constexpr float kGMin = -5.0f;   // log-decay lower bound
constexpr float kGMax = 0.0f;

// Device-side status bits written into the first word of a workspace.
constexpr uint32_t kStatusBadSeqlens = 1u;
constexpr uint32_t kStatusTimeout = 2u;
constexpr uint32_t kStatusRange = 4u;  // a result of the bf16 prefill is not finite

__device__ __forceinline__ float clamp_g(float g) { return fminf(fmaxf(g, kGMin), kGMax); }

// How the bf16 prefill runs for given sizes (host side): schedule 1 = fused
// (groups of group_chains chains, `groups` cooperative launches; ring > 0:
// blocks in per-chain rings of that length; lead_items > 0: that many blocks
// are prepared by a launch of producers only before the chains start), 0 =
// split; bytes of workspace.
struct PrefillPlan {
    int schedule = 0, groups = 0, group_chains = 0, ring = 0;
    size_t bytes = 0;
    long long lead_items = 0;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ---- ldmatrix -------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t r[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t r[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D(16x8, fp32) += A(16x16, bf16) * B(16x8, bf16)
__device__ __forceinline__ void mma_bf16_16816(float c[4], const uint32_t a[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D(16x8, fp32) += A(16x16, f16) * B(16x8, f16)
__device__ __forceinline__ void mma_f16_16816(float c[4], const uint32_t a[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Fragment loaders. `base` is a shared-memory byte address of a bf16 matrix
// with leading dimension `ld` (elements); (r0, k0) are the tile origin.
//
// A (16 x 16) from row-major storage A[m][k].
__device__ __forceinline__ void frag_a_rowmajor(uint32_t a[4], uint32_t base, int ld, int m0,
                                                int k0, int lane) {
    const int r = m0 + (lane & 15);
    const int c = k0 + ((lane >> 4) << 3);
    ldsm_x4(a, base + (uint32_t)(r * ld + c) * 2u);
}
// A (16 x 16) from storage of its transpose, At[k][m].
__device__ __forceinline__ void frag_a_colmajor(uint32_t a[4], uint32_t base, int ld, int m0,
                                                int k0, int lane) {
    const int idx = lane >> 3;
    const int r = k0 + (lane & 7) + ((idx >> 1) << 3);
    const int c = m0 + ((idx & 1) << 3);
    ldsm_x4_t(a, base + (uint32_t)(r * ld + c) * 2u);
}
// B (16 x 16 = two n8 tiles) from storage Bt[n][k] (k contiguous).
// Result: {b0(n0), b1(n0), b0(n0+8), b1(n0+8)}.
__device__ __forceinline__ void frag_b_nk(uint32_t b[4], uint32_t base, int ld, int n0, int k0,
                                          int lane) {
    const int idx = lane >> 3;
    const int r = n0 + (lane & 7) + ((idx >> 1) << 3);
    const int c = k0 + ((idx & 1) << 3);
    ldsm_x4(b, base + (uint32_t)(r * ld + c) * 2u);
}
// B (16 x 16 = two n8 tiles) from storage B[k][n] (n contiguous).
__device__ __forceinline__ void frag_b_kn(uint32_t b[4], uint32_t base, int ld, int n0, int k0,
                                          int lane) {
    const int idx = lane >> 3;
    const int r = k0 + (lane & 7) + ((idx & 1) << 3);
    const int c = n0 + ((idx >> 1) << 3);
    ldsm_x4_t(b, base + (uint32_t)(r * ld + c) * 2u);
}

// I/O element conversions.
template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Sequence bounds: either equal-length sequences (cu == nullptr) or packed
// offsets. Returns false (and flags the status word) on malformed offsets.
__device__ __forceinline__ bool seq_bounds(const int32_t *cu, int n, int T, int T_total,
                                           int &t0, int &t1, uint32_t *status) {
    if (cu == nullptr) {
        t0 = n * T;
        t1 = t0 + T;
        return true;
    }
    t0 = cu[n];
    t1 = cu[n + 1];
    const bool ok = (t0 >= 0) && (t1 >= t0) && (t1 <= T_total) && (n != 0 || t0 == 0);
    if (!ok && status != nullptr) atomicOr(status, kStatusBadSeqlens);
    return ok;
}

}  // namespace kda
