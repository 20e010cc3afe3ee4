// Host-side helpers shared by the translation units of libspecverify.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/specverify.h"

namespace sv {
int sm_count();                    // SMs of the current device
void prof_begin(cudaStream_t s);   // profiling hook around the dominant kernel
void prof_end(cudaStream_t s);
void set_launches(int n);          // kernels launched by the last call (this thread)
long long wait_budget();           // spec_set_wait_budget's current value (SM cycles)
void counter_region(int B, int rows, int V, size_t *offset, size_t *bytes);  // per-request counters
// Host-side argument rules of the verification calls (the workspace aside):
// SV_ERR_INVALID if one is broken, else SV_OK.  `rows` is taken in 64 bits so
// that a product B (K + 1) past INT_MAX is refused rather than wrapped.
sv_status check_verify_args(const void *logits, sv_dtype dt, const float *q, const int32_t *row_offsets,
                            int B, int K, long long rows, int V, float temperature, bool sample,
                            const int32_t *draft, const float *uniforms, const int32_t *out_tokens,
                            const int32_t *accept_len);
size_t finish_workspace_size(int B, int rows, int V);
// Decide (+ residual draw when `sample`) over fp32 logits and chunk partials
// produced by a previous kernel on `s` (see verify.cu).
sv_status finish_from_partials(const float *logits, const float2 *partials, int n_parts, const float *q, int B,
                               int K, int V, float temperature, bool sample, const int32_t *draft,
                               const float *uniforms, int32_t *out_tokens, int32_t *accept_len, float *diag,
                               void *ws, size_t ws_bytes, cudaStream_t s, int *launches);
struct Args;
// One cluster of CTAs per request over the call in `a` (cluster.cu); nr_cap rows per request at most.
cudaError_t launch_cluster_kernel(const Args &a, int nr_cap, bool sample, bool bf16, cudaStream_t s);
// One CTA per request over the call in `a` (small.cu); nr_cap rows per request at most.
cudaError_t launch_small_kernel(const Args &a, int nr_cap, bool sample, bool bf16, cudaStream_t s);
}  // namespace sv
