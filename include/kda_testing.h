/*
 * kda_testing.h -- entry points of libkda.so that exist only for tests of its
 * failure detection. Production code never calls them; nothing in kda.h
 * reaches them, and no environment variable switches them on.
 */
#ifndef KDA_TESTING_H
#define KDA_TESTING_H

#include <stddef.h>
#include <stdint.h>

#include "kda.h"  /* kda_prefill_plan_info */

#ifdef __cplusplus
extern "C" {
#endif

/*
 * kda_prefill (bf16 I/O only, arguments as there) with its recurrence chains
 * launched WITHOUT the chunk-preparation producers of the fused schedule and
 * with every wait of a chain bounded by wait_ms milliseconds (1..10000). No
 * ready flag is ever set, so each chain gives up after wait_ms, records
 * KDA_ERR_TIMEOUT in the workspace status word (read it with
 * kda_workspace_status) and returns; the outputs are garbage. It shows that a
 * missing producer ends in an error status and a usable context, never in a
 * hang. Needs fewer chains (N * H) than SMs. Returns KDA_OK once enqueued,
 * KDA_ERR_UNSUPPORTED for fp32 I/O, KDA_ERR_INVALID_ARG for a bad wait_ms or
 * invalid arguments, KDA_ERR_CUDA if the launch fails (e.g. too many chains).
 * The pages have no counterpart to this entry point.
 */
int kda_testing_prefill_chain_timeout(const void *q, const void *k, const void *v,
                                      const float *g, const void *beta, float scale,
                                      const float *init_state, const int32_t *cu_seqlens,
                                      int32_t N, int32_t T, int32_t H, int32_t D, int32_t chunk,
                                      int32_t io, void *out, float *final_state, void *workspace,
                                      size_t workspace_bytes, int32_t wait_ms, void *stream);

/*
 * The workspace-plan selection of the bf16 prefill (the host logic behind
 * kda_prefill_plan) for given device properties instead of the current
 * device's, so that it can be checked without a GPU: sm_count SMs,
 * cooperative != 0 if cooperative launches are supported, schedule_override
 * -1 (automatic), KDA_SCHEDULE_SPLIT or KDA_SCHEDULE_FUSED. kind 0: the plan
 * that a workspace of workspace_bytes gets; 1: the fastest plan; 2: the ring
 * plan with the modelled best group; 3: the smallest accepted plan (kinds 1-3
 * ignore workspace_bytes). Sizes as in kda_prefill_workspace_size (D = 128,
 * chunk 64). Writes *plan and returns KDA_OK; KDA_ERR_INVALID_ARG when the
 * arguments are invalid or no plan fits. Launches nothing, needs no device.
 */
int kda_testing_prefill_plan(int32_t N, int32_t T, int32_t H, int32_t varlen, int32_t sm_count,
                             int32_t cooperative, int32_t schedule_override, int32_t kind,
                             size_t workspace_bytes, kda_prefill_plan_info *plan);

#ifdef __cplusplus
}
#endif

#endif /* KDA_TESTING_H */
