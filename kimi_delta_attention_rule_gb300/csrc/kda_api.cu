// C ABI of libkda (declared in include/kda.h): argument validation and
// kernel dispatch. No allocation, no host synchronisation except in
// kda_workspace_status().
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>  // header-only: ranges are free unless a profiler is attached

#include "kda.h"
#include "kda_testing.h"
#include "kda_common.cuh"

namespace kda {
template <typename IO>
cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *g,
                          const void *beta, float scale, int B, int T, int H, int g_per_channel,
                          float *pool, int pool_size, const int32_t *idx, void *out,
                          cudaStream_t stream);
cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, const float *g,
                               const float *beta, float scale, const float *init,
                               const int32_t *cu, int N, int T, int T_total, int H, int chunk,
                               int g_per_channel, int snap_interval, int snap_max, float *snaps,
                               float *out, float *fin, uint32_t *status, cudaStream_t stream);
size_t prefill_tc_workspace(int N, long long T, long long T_total, int H, bool varlen, int kind);
cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const float *g,
                              const void *beta, float scale, const float *init,
                              const int32_t *cu, int N, int T, int T_total, int H,
                              int g_per_channel, int snap_interval, int snap_max, float *snaps,
                              void *out, float *fin, unsigned char *ws, size_t ws_bytes,
                              unsigned test_wait_ms, cudaStream_t stream);
void prefill_tc_query(int N, long long T, long long T_total, int H, bool varlen, size_t budget,
                      PrefillPlan &p);
int prefill_tc_set_schedule(int s);
bool prefill_tc_plan_for(int N, long long T, long long T_total, int H, bool varlen, int nsm,
                         int coop, int force, size_t budget, int kind, PrefillPlan &p);
template <typename IO>
cudaError_t launch_layer_prologue(const void *q_raw, const void *k_raw, const void *v_raw,
                                  const void *alpha_raw, const void *beta_raw, const float *wq,
                                  const float *wk, const float *wv, int W, const int32_t *cu,
                                  int N, long long T_total, int H, void *q, void *k, void *v,
                                  float *g, void *beta, cudaStream_t stream);
template <typename IO>
cudaError_t launch_layer_epilogue(const void *o, const void *gate_raw, const float *w,
                                  long long T_total, int H, void *y, cudaStream_t stream);
template <typename IO>
cudaError_t launch_layer_prologue_decode(const void *q_raw, const void *k_raw, const void *v_raw,
                                         const void *alpha_raw, const void *beta_raw,
                                         const float *wq, const float *wk, const float *wv, int W,
                                         int B, int T, int H, void *conv_state, int pool_size,
                                         const int32_t *idx, void *q, void *k, void *v, float *g,
                                         void *beta, cudaStream_t stream);
}  // namespace kda

namespace {

constexpr size_t kWorkspaceBytes = 256;  // device status word, padded to 256 B
constexpr int32_t kMaxDecodeTokens = 64;  // beyond a chunk, the prefill path is the better one

// Workspace of one call: status word, plus (bf16 path) the chunk schedule,
// the fused schedule's flags and the 74,368-byte prepared blocks. kind 1: the
// fastest plan's size (one block per chunk and head); 2: the ring plan's
// (blocks in flight per chain, bounded by the group, not the length); 3: the
// smallest size kda_prefill accepts.
size_t workspace_bytes_for(int32_t N, int32_t T, int32_t H, int32_t io, bool varlen, int kind) {
    if (io == KDA_F32) return kWorkspaceBytes;
    return kda::prefill_tc_workspace(N, T, T, H, varlen, kind);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// An NVTX range around the launches of one call (seen by nsys / ncu --nvtx).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

// Validates the prefill sizes; writes T_total on success.
int check_prefill_dims(int32_t N, int32_t T, int32_t H, int32_t D, int32_t chunk, int32_t io,
                       bool varlen, long long *T_total) {
    if (N < 0 || T < 0 || H <= 0 || D <= 0) return KDA_ERR_INVALID_ARG;
    if (io != KDA_BF16 && io != KDA_F32) return KDA_ERR_UNSUPPORTED;
    if (D != kda::kD) return KDA_ERR_UNSUPPORTED;
    if (io == KDA_BF16 && chunk != 64) return KDA_ERR_UNSUPPORTED;
    if (io == KDA_F32 && chunk != 16 && chunk != 64) return KDA_ERR_UNSUPPORTED;
    const long long tt = varlen ? (long long)T : (long long)N * T;
    // element offsets (t * H + h) * D must fit in 64 bits and grid sizes in 32 bits
    if (tt > (1LL << 31) - 1 || tt * H > (1LL << 40)) return KDA_ERR_INVALID_ARG;
    if ((long long)N * H * 4 > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    *T_total = tt;
    return KDA_OK;
}

}  // namespace

extern "C" {

const char *kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
        case KDA_ERR_DEVICE: return "KDA_ERR_DEVICE";
        case KDA_ERR_TOO_LARGE: return "KDA_ERR_TOO_LARGE";
        case KDA_ERR_RANGE: return "KDA_ERR_RANGE";
        default: return "KDA_ERR_UNKNOWN";
    }
}

int kda_abi_version(void) { return 101; }

size_t kda_prefill_workspace_size(int32_t N, int32_t T, int32_t H, int32_t D, int32_t chunk,
                                  int32_t io, int32_t varlen) {
    long long tt = 0;
    if (check_prefill_dims(N, T, H, D, chunk, io, varlen != 0, &tt) != KDA_OK) return 0;
    return workspace_bytes_for(N, T, H, io, varlen != 0, 1);
}

size_t kda_prefill_workspace_size_ring(int32_t N, int32_t T, int32_t H, int32_t D, int32_t chunk,
                                       int32_t io, int32_t varlen) {
    long long tt = 0;
    if (check_prefill_dims(N, T, H, D, chunk, io, varlen != 0, &tt) != KDA_OK) return 0;
    return workspace_bytes_for(N, T, H, io, varlen != 0, 2);
}

size_t kda_prefill_workspace_size_min(int32_t N, int32_t T, int32_t H, int32_t D, int32_t chunk,
                                      int32_t io, int32_t varlen) {
    long long tt = 0;
    if (check_prefill_dims(N, T, H, D, chunk, io, varlen != 0, &tt) != KDA_OK) return 0;
    return workspace_bytes_for(N, T, H, io, varlen != 0, 3);
}

int kda_prefill_plan(int32_t N, int32_t T, int32_t H, int32_t D, int32_t chunk, int32_t io,
                     int32_t varlen, size_t workspace_bytes, kda_prefill_plan_info *plan) {
    if (plan == nullptr) return KDA_ERR_INVALID_ARG;
    long long tt = 0;
    const int rc = check_prefill_dims(N, T, H, D, chunk, io, varlen != 0, &tt);
    if (rc != KDA_OK) return rc;
    if (io == KDA_F32) {
        if (workspace_bytes < kWorkspaceBytes) return KDA_ERR_INVALID_ARG;
        *plan = kda_prefill_plan_info{KDA_SCHEDULE_DIRECT, 0, 0, 0, kWorkspaceBytes, 0};
        return KDA_OK;
    }
    kda::PrefillPlan p;
    kda::prefill_tc_query(N, T, tt, H, varlen != 0, workspace_bytes, p);
    if (p.schedule == -2) return KDA_ERR_INVALID_ARG;
    if (p.schedule < 0) return KDA_ERR_CUDA;
    *plan = kda_prefill_plan_info{p.schedule == 1 ? KDA_SCHEDULE_FUSED : KDA_SCHEDULE_SPLIT,
                                  p.groups, p.group_chains, p.ring, p.bytes, p.lead_items};
    return KDA_OK;
}

int kda_prefill_schedule(int32_t N, int32_t T, int32_t H, int32_t D, int32_t chunk, int32_t io,
                         int32_t varlen) {
    kda_prefill_plan_info p;
    const int rc = kda_prefill_plan(N, T, H, D, chunk, io, varlen, SIZE_MAX, &p);
    return rc == KDA_OK ? p.schedule : -rc;
}

int kda_check_cu_seqlens(const int32_t *cu, int32_t N, int32_t T_total) {
    if (cu == nullptr || N < 0 || T_total < 0) return KDA_ERR_INVALID_ARG;
    if (cu[0] != 0 || cu[N] != T_total) return KDA_ERR_INVALID_ARG;
    for (int32_t n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

}  // extern "C"

namespace {

// kda_prefill_ex, plus the failure-detection test mode (test_wait_ms > 0:
// bf16 chains launched without producers, each wait bounded by test_wait_ms).
int prefill_impl(const void *q, const void *k, const void *v, const float *g, const void *beta,
                 float scale, const float *init_state, const int32_t *cu_seqlens, int32_t N,
                 int32_t T, int32_t H, int32_t D, int32_t chunk, int32_t io, int32_t g_per_channel,
                 int32_t snapshot_interval, int32_t max_snapshots, float *snapshots, void *out,
                 float *final_state, void *workspace, size_t workspace_bytes, unsigned test_wait_ms,
                 void *stream) {

    long long T_total = 0;
    const int rc = check_prefill_dims(N, T, H, D, chunk, io, cu_seqlens != nullptr, &T_total);
    if (rc != KDA_OK) return rc;
    if (g_per_channel != 0 && g_per_channel != 1) return KDA_ERR_INVALID_ARG;
    if (snapshot_interval < 0) return KDA_ERR_INVALID_ARG;
    if (snapshot_interval > 0) {
        if (snapshot_interval % chunk != 0) return KDA_ERR_UNSUPPORTED;
        if (snapshots == nullptr || max_snapshots <= 0 || !aligned16(snapshots))
            return KDA_ERR_INVALID_ARG;
        if ((long long)N * max_snapshots * H > (1LL << 40)) return KDA_ERR_INVALID_ARG;
    }
    if (workspace == nullptr ||
        workspace_bytes < workspace_bytes_for(N, T, H, io, cu_seqlens != nullptr, 3) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return KDA_ERR_INVALID_ARG;
    if (N == 0) return KDA_OK;
    if (T_total > 0) {
        if (!q || !k || !v || !g || !beta || !out) return KDA_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(out))
            return KDA_ERR_INVALID_ARG;
    }
    if ((init_state && !aligned16(init_state)) || (final_state && !aligned16(final_state)))
        return KDA_ERR_INVALID_ARG;
    const int si = snapshot_interval, sm = snapshot_interval > 0 ? max_snapshots : 0;
    NvtxRange range(io == KDA_F32 ? "kda_prefill (fp32)" : "kda_prefill");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t *status = static_cast<uint32_t *>(workspace);
    // the status word reports this call only
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    if (io == KDA_F32) {
        e = kda::launch_prefill_f32(static_cast<const float *>(q), static_cast<const float *>(k),
                                    static_cast<const float *>(v), g,
                                    static_cast<const float *>(beta), scale, init_state,
                                    cu_seqlens, N, T, (int)T_total, H, chunk, g_per_channel, si,
                                    sm, snapshots, static_cast<float *>(out), final_state,
                                    status, st);
    } else {
        e = kda::launch_prefill_tc(q, k, v, g, beta, scale, init_state, cu_seqlens, N, T,
                                   (int)T_total, H, g_per_channel, si, sm, snapshots, out,
                                   final_state, static_cast<unsigned char *>(workspace),
                                   workspace_bytes, test_wait_ms, st);
    }
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}


}  // namespace

extern "C" {

int kda_prefill_ex(const void *q, const void *k, const void *v, const float *g,
                   const void *beta, float scale, const float *init_state,
                   const int32_t *cu_seqlens, int32_t N, int32_t T, int32_t H, int32_t D,
                   int32_t chunk, int32_t io, int32_t g_per_channel, int32_t snapshot_interval,
                   int32_t max_snapshots, float *snapshots, void *out, float *final_state,
                   void *workspace, size_t workspace_bytes, void *stream) {
    return prefill_impl(q, k, v, g, beta, scale, init_state, cu_seqlens, N, T, H, D, chunk, io,
                        g_per_channel, snapshot_interval, max_snapshots, snapshots, out,
                        final_state, workspace, workspace_bytes, 0u, stream);
}

int kda_prefill_set_schedule(int schedule) {
    if (schedule != -1 && schedule != KDA_SCHEDULE_SPLIT && schedule != KDA_SCHEDULE_FUSED)
        return -KDA_ERR_INVALID_ARG;
    return kda::prefill_tc_set_schedule(schedule);
}

int kda_testing_prefill_chain_timeout(const void *q, const void *k, const void *v,
                                      const float *g, const void *beta, float scale,
                                      const float *init_state, const int32_t *cu_seqlens,
                                      int32_t N, int32_t T, int32_t H, int32_t D, int32_t chunk,
                                      int32_t io, void *out, float *final_state, void *workspace,
                                      size_t workspace_bytes, int32_t wait_ms, void *stream) {
    if (io != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (wait_ms <= 0 || wait_ms > 10000) return KDA_ERR_INVALID_ARG;
    return prefill_impl(q, k, v, g, beta, scale, init_state, cu_seqlens, N, T, H, D, chunk, io, 1,
                        0, 0, nullptr, out, final_state, workspace, workspace_bytes,
                        (unsigned)wait_ms, stream);
}

int kda_testing_prefill_plan(int32_t N, int32_t T, int32_t H, int32_t varlen, int32_t sm_count,
                             int32_t cooperative, int32_t schedule_override, int32_t kind,
                             size_t workspace_bytes, kda_prefill_plan_info *plan) {
    if (plan == nullptr || kind < 0 || kind > 3 || schedule_override < -1 || schedule_override > 1)
        return KDA_ERR_INVALID_ARG;
    long long tt = 0;
    const int rc = check_prefill_dims(N, T, H, kda::kD, 64, KDA_BF16, varlen != 0, &tt);
    if (rc != KDA_OK) return rc;
    kda::PrefillPlan p;
    if (!kda::prefill_tc_plan_for(N, T, tt, H, varlen != 0, sm_count, cooperative != 0,
                                  schedule_override, workspace_bytes, kind, p))
        return KDA_ERR_INVALID_ARG;
    *plan = kda_prefill_plan_info{p.schedule == 1 ? KDA_SCHEDULE_FUSED : KDA_SCHEDULE_SPLIT,
                                  p.groups, p.group_chains, p.ring, p.bytes, p.lead_items};
    return KDA_OK;
}

int kda_prefill(const void *q, const void *k, const void *v, const float *g, const void *beta,
                float scale, const float *init_state, const int32_t *cu_seqlens, int32_t N,
                int32_t T, int32_t H, int32_t D, int32_t chunk, int32_t io, void *out,
                float *final_state, void *workspace, size_t workspace_bytes, void *stream) {
    return kda_prefill_ex(q, k, v, g, beta, scale, init_state, cu_seqlens, N, T, H, D, chunk, io,
                          1, 0, 0, nullptr, out, final_state, workspace, workspace_bytes, stream);
}

int kda_decode(const void *q, const void *k, const void *v, const float *g, const void *beta,
               float scale, int32_t B, int32_t T, int32_t H, int32_t D, int32_t io,
               int32_t g_per_channel, float *state_pool, int32_t pool_size,
               const int32_t *state_indices, void *out, void *stream) {
    if (B < 0 || T < 0 || H <= 0 || D <= 0 || pool_size < 0) return KDA_ERR_INVALID_ARG;
    if (io != KDA_BF16 && io != KDA_F32) return KDA_ERR_UNSUPPORTED;
    if (D != kda::kD) return KDA_ERR_UNSUPPORTED;
    if (T > kMaxDecodeTokens) return KDA_ERR_UNSUPPORTED;
    if (g_per_channel != 0 && g_per_channel != 1) return KDA_ERR_INVALID_ARG;
    if ((long long)B * H > 0x7fffffffLL || (long long)B * T * H > (1LL << 40))
        return KDA_ERR_INVALID_ARG;
    if (state_indices == nullptr && pool_size < B) return KDA_ERR_INVALID_ARG;
    if (B == 0 || T == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !state_pool || !out) return KDA_ERR_INVALID_ARG;
    // rows of q, k, v (and g per channel) are copied in 16-byte pieces
    if (!aligned16(state_pool) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !aligned16(out) || (g_per_channel && !aligned16(g)))
        return KDA_ERR_INVALID_ARG;
    NvtxRange range("kda_decode");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e =
        io == KDA_F32
            ? kda::launch_decode<float>(q, k, v, g, beta, scale, B, T, H, g_per_channel,
                                        state_pool, pool_size, state_indices, out, st)
            : kda::launch_decode<__nv_bfloat16>(q, k, v, g, beta, scale, B, T, H, g_per_channel,
                                                state_pool, pool_size, state_indices, out, st);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_decode_step(const void *q, const void *k, const void *v, const float *g,
                    const void *beta, float scale, int32_t B, int32_t H, int32_t D, int32_t io,
                    float *state_inout, void *out, void *stream) {
    return kda_decode(q, k, v, g, beta, scale, B, 1, H, D, io, 1, state_inout, B, nullptr, out,
                      stream);
}

int kda_layer_prologue(const void *q_raw, const void *k_raw, const void *v_raw,
                       const void *alpha_raw, const void *beta_raw, const float *conv_q,
                       const float *conv_k, const float *conv_v, int32_t W,
                       const int32_t *cu_seqlens, int32_t N, int32_t T_total, int32_t H, int32_t D,
                       int32_t io, void *q, void *k, void *v, float *g, void *beta, void *stream) {
    if (N < 0 || T_total < 0 || H <= 0 || D <= 0) return KDA_ERR_INVALID_ARG;
    if (io != KDA_BF16 && io != KDA_F32) return KDA_ERR_UNSUPPORTED;
    if (D != kda::kD || W < 1 || W > 4) return KDA_ERR_UNSUPPORTED;
    if ((long long)T_total * H > (1LL << 33)) return KDA_ERR_INVALID_ARG;
    if (T_total == 0) return KDA_OK;
    if (!q_raw || !k_raw || !v_raw || !alpha_raw || !beta_raw || !conv_q || !conv_k || !conv_v ||
        !q || !k || !v || !g || !beta)
        return KDA_ERR_INVALID_ARG;
    const unsigned a = io == KDA_F32 ? 15u : 7u;  // row pieces of 4 channels
    for (const void *p : {q_raw, k_raw, v_raw, alpha_raw, static_cast<const void *>(q),
                          static_cast<const void *>(k), static_cast<const void *>(v)})
        if (reinterpret_cast<uintptr_t>(p) & a) return KDA_ERR_INVALID_ARG;
    if (!aligned16(g)) return KDA_ERR_INVALID_ARG;
    // a lane reads its 4 channels x W taps of [H, D, W] weights as float4
    if (!aligned16(conv_q) || !aligned16(conv_k) || !aligned16(conv_v)) return KDA_ERR_INVALID_ARG;
    NvtxRange range("kda_layer_prologue");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e =
        io == KDA_F32
            ? kda::launch_layer_prologue<float>(q_raw, k_raw, v_raw, alpha_raw, beta_raw, conv_q,
                                                conv_k, conv_v, W, cu_seqlens, N, T_total, H, q,
                                                k, v, g, beta, st)
            : kda::launch_layer_prologue<__nv_bfloat16>(q_raw, k_raw, v_raw, alpha_raw, beta_raw,
                                                        conv_q, conv_k, conv_v, W, cu_seqlens, N,
                                                        T_total, H, q, k, v, g, beta, st);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_layer_prologue_decode(const void *q_raw, const void *k_raw, const void *v_raw,
                              const void *alpha_raw, const void *beta_raw, const float *conv_q,
                              const float *conv_k, const float *conv_v, int32_t W, int32_t B,
                              int32_t T, int32_t H, int32_t D, int32_t io, void *conv_state,
                              int32_t pool_size, const int32_t *state_indices, void *q, void *k,
                              void *v, float *g, void *beta, void *stream) {
    if (B < 0 || T < 0 || H <= 0 || D <= 0 || pool_size < 0) return KDA_ERR_INVALID_ARG;
    if (io != KDA_BF16 && io != KDA_F32) return KDA_ERR_UNSUPPORTED;
    if (D != kda::kD || W < 1 || W > 4) return KDA_ERR_UNSUPPORTED;
    if ((long long)B * T * H > (1LL << 33)) return KDA_ERR_INVALID_ARG;
    if (state_indices == nullptr && pool_size < B) return KDA_ERR_INVALID_ARG;
    if (B == 0 || T == 0) return KDA_OK;
    if (!q_raw || !k_raw || !v_raw || !alpha_raw || !beta_raw || !conv_q || !conv_k || !conv_v ||
        !q || !k || !v || !g || !beta || (W > 1 && !conv_state))
        return KDA_ERR_INVALID_ARG;
    const unsigned a = io == KDA_F32 ? 15u : 7u;  // row pieces of 4 channels
    for (const void *p : {q_raw, k_raw, v_raw, alpha_raw, static_cast<const void *>(q),
                          static_cast<const void *>(k), static_cast<const void *>(v),
                          static_cast<const void *>(conv_state)})
        if (reinterpret_cast<uintptr_t>(p) & a) return KDA_ERR_INVALID_ARG;
    if (!aligned16(g) || !aligned16(conv_q) || !aligned16(conv_k) || !aligned16(conv_v))
        return KDA_ERR_INVALID_ARG;
    NvtxRange range("kda_layer_prologue_decode");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e =
        io == KDA_F32
            ? kda::launch_layer_prologue_decode<float>(q_raw, k_raw, v_raw, alpha_raw, beta_raw,
                                                       conv_q, conv_k, conv_v, W, B, T, H,
                                                       conv_state, pool_size, state_indices, q, k,
                                                       v, g, beta, st)
            : kda::launch_layer_prologue_decode<__nv_bfloat16>(
                  q_raw, k_raw, v_raw, alpha_raw, beta_raw, conv_q, conv_k, conv_v, W, B, T, H,
                  conv_state, pool_size, state_indices, q, k, v, g, beta, st);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_layer_epilogue(const void *o, const void *gate_raw, const float *norm_weight,
                       int32_t T_total, int32_t H, int32_t D, int32_t io, void *y, void *stream) {
    if (T_total < 0 || H <= 0 || D <= 0) return KDA_ERR_INVALID_ARG;
    if (io != KDA_BF16 && io != KDA_F32) return KDA_ERR_UNSUPPORTED;
    if (D != kda::kD) return KDA_ERR_UNSUPPORTED;
    if ((long long)T_total * H > (1LL << 33)) return KDA_ERR_INVALID_ARG;
    if (T_total == 0) return KDA_OK;
    if (!o || !gate_raw || !norm_weight || !y) return KDA_ERR_INVALID_ARG;
    // rows are read and written 8 channels (16 or 32 bytes) per lane
    for (const void *p : {o, gate_raw, static_cast<const void *>(y)})
        if (!aligned16(p)) return KDA_ERR_INVALID_ARG;
    if (!aligned16(norm_weight)) return KDA_ERR_INVALID_ARG;
    NvtxRange range("kda_layer_epilogue");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e =
        io == KDA_F32 ? kda::launch_layer_epilogue<float>(o, gate_raw, norm_weight, T_total, H, y, st)
                      : kda::launch_layer_epilogue<__nv_bfloat16>(o, gate_raw, norm_weight, T_total,
                                                                  H, y, st);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_workspace_status(void *workspace, void *stream) {
    if (workspace == nullptr) return KDA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof(word), st) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KDA_ERR_CUDA;
    if (word & kda::kStatusTimeout) return KDA_ERR_TIMEOUT;
    if (word & kda::kStatusBadSeqlens) return KDA_ERR_DEVICE;
    if (word & kda::kStatusRange) return KDA_ERR_RANGE;
    return KDA_OK;
}

}  // extern "C"
