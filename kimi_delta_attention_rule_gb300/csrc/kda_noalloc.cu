// kda_prefill_noalloc: the prefill entry point for callers that cannot
// allocate device memory themselves.
//
// Some callers have no way to call cudaMalloc before the call: code running
// inside a captured region that must not allocate, plug-in hosts that hand
// over only the tensors they own, or runtimes whose allocator is not exposed
// to the library. kda_prefill needs a caller-provided workspace (its device
// status word and schedule data); this variant takes its scratch from a
// file-scope device array instead, so the caller passes only inputs and
// outputs.
//
// The array is kNoallocScratchBytes long and lives on every GPU that loads
// the library until the process exits. Host code cannot use the array's name
// as a device address, so at the first call on each device (with that
// device current) the address is looked up with cudaGetSymbolAddress and
// cached. That first call should therefore come before any stream capture.
// Every call shares the one array: calls that overlap on the GPU (other
// streams, or other threads) race on it and must be serialised by the
// caller. The status word it holds is cleared by each call before its
// kernels run, and kda_noalloc_status() reads it: the caller has no address
// of the array, so device-side errors of these calls (malformed offsets, a
// timed-out wait) are reported through that query instead of
// kda_workspace_status().
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

#include "kda.h"

namespace {

constexpr size_t kNoallocScratchBytes = 16u << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
int scratch_for_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return KDA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" {

int kda_prefill_noalloc(const void *q, const void *k, const void *v, const float *g,
                        const void *beta, float scale, const float *init_state,
                        const int32_t *cu_seqlens, int32_t N, int32_t T, int32_t H, int32_t D,
                        int32_t chunk, int32_t io, void *out, float *final_state, void *stream) {
    // the smallest workspace the call accepts; kda_prefill then runs the
    // fastest plan that the array holds (the ring plan when the one with a
    // block per chunk does not fit)
    const size_t need =
        kda_prefill_workspace_size_min(N, T, H, D, chunk, io, cu_seqlens != nullptr ? 1 : 0);
    if (need == 0) {
        // same validation (and error code) as kda_prefill
        return kda_prefill(q, k, v, g, beta, scale, init_state, cu_seqlens, N, T, H, D, chunk,
                           io, out, final_state, nullptr, 0, stream);
    }
    if (need > kNoallocScratchBytes) return KDA_ERR_TOO_LARGE;  // beyond the static scratch
    void *scratch = nullptr;
    const int rc = scratch_for_current_device(&scratch);
    if (rc != KDA_OK) return rc;
    return kda_prefill(q, k, v, g, beta, scale, init_state, cu_seqlens, N, T, H, D, chunk, io,
                       out, final_state, scratch, kNoallocScratchBytes, stream);
}

int kda_noalloc_status(void *stream) {
    void *scratch = nullptr;
    const int rc = scratch_for_current_device(&scratch);
    if (rc != KDA_OK) return rc;
    // the status word is the first word of the array, as of any workspace
    return kda_workspace_status(scratch, stream);
}

}  // extern "C"
