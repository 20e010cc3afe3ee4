// Sampling verification for callers that cannot allocate device memory.
//
// Some host programs have no device allocator to hand: a plugin loaded into
// an inference server whose device memory is all reserved by the server's
// own caching allocator, or a latency-critical loop that must not call
// cudaMalloc (it can synchronise the whole device).  Such callers still own
// their inputs and outputs but cannot provide the workspace that
// spec_verify_sample needs.  spec_verify_sample_noalloc runs the same
// kernels with a scratch area that this library keeps in a fixed device
// array instead.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/specverify.h"
#include "sv_host.h"

namespace {

// Scratch of every spec_verify_sample_noalloc call on a device.  It occupies
// SV_NOALLOC_SCRATCH_BYTES of every GPU that loads this library until the
// process exits.  In host code the name is only a stand-in: its device
// address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_scratch[SV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_dev[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per
// device (with that device current) and cached.
sv_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_dev[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return SV_ERR_CUDA;
        g_scratch_dev[dev] = p;
    }
    *out = g_scratch_dev[dev];
    return SV_OK;
}

}  // namespace

extern "C" sv_status spec_verify_sample_noalloc(const void *logits, sv_dtype dt, const float *q, int B, int K,
                                                int V, float temperature, const int32_t *draft,
                                                const float *uniforms, int32_t *out_tokens,
                                                int32_t *accept_len, float *diag, void *stream) {
    if (B < 0 || K < 0 || K > SV_MAX_K) return SV_ERR_INVALID;
    // Every argument rule is checked before anything touches the shared
    // scratch, so a refused call enqueues nothing.
    const long long rows64 = static_cast<long long>(B) * (K + 1);
    const sv_status arg = sv::check_verify_args(logits, dt, q, nullptr, B, K, rows64, V, temperature, true,
                                                draft, uniforms, out_tokens, accept_len);
    if (arg != SV_OK) return arg;
    if (B == 0) return spec_verify_sample(logits, dt, q, B, K, V, temperature, draft, uniforms, out_tokens,
                                          accept_len, diag, nullptr, 0, stream);
    const int rows = static_cast<int>(rows64);
    if (spec_verify_workspace_size(B, rows, V) > SV_NOALLOC_SCRATCH_BYTES) return SV_ERR_WORKSPACE;
    // The scratch keeps whatever the last call left in it; the per-request
    // counters must start this call at zero.
    size_t off = 0, bytes = 0;
    sv::counter_region(B, rows, V, &off, &bytes);
    if (off > SV_NOALLOC_SCRATCH_BYTES || bytes > SV_NOALLOC_SCRATCH_BYTES - off) return SV_ERR_WORKSPACE;
    void *scratch = nullptr;
    const sv_status st = scratch_address(&scratch);
    if (st != SV_OK) return st;
    if (cudaMemsetAsync(static_cast<char *>(scratch) + off, 0, bytes, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return SV_ERR_CUDA;
    return spec_verify_sample(logits, dt, q, B, K, V, temperature, draft, uniforms, out_tokens, accept_len,
                              diag, scratch, SV_NOALLOC_SCRATCH_BYTES, stream);
}
