// Model-free n-gram (prompt lookup) drafter: proposes the tokens that
// followed the latest earlier occurrence of the context's longest matching
// suffix.  "Co-Designing AI Models Using Speculative Decoding for Faster LLM
// Inference", Table 1 (suffix / n-gram: string matching over the token
// stream, no model, one lookup), and the model-free passage of "Speculative
// Decoding" (glossary), section "Variants: Draft Models, EAGLE, Medusa, and
// Model-Free Methods" (prompt lookup matches strings already in the context).
//
// One CTA per request.  The context's last n_max tokens sit in shared memory,
// and the context passes through shared memory in tiles of 8192 tokens (with
// the 32 tokens before each tile kept as a halo); every thread takes
// candidate end positions e <= L - 2 and measures m(e),
// the length of the common suffix of ctx[..e] and ctx[..L-1] (at most
// min(n_max, e + 1)).  The winner maximises (m, e) with m >= n_min: the
// longest suffix first, then its latest occurrence -- the order in which the
// method tries n = n_max .. n_min and scans back from the end.
#include <cstdint>

#include "../../include/specverify.h"
#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {
namespace ng {

constexpr int kThreads = 512;
constexpr int kMaxN = 32;
constexpr int kTile = 8192;            // context tokens staged in shared memory at a time
constexpr int kPerThread = kTile / kThreads;

__global__ void __launch_bounds__(kThreads) ngram_kernel(const int32_t *tokens, const int32_t *ctx_offsets, int K,
                                                         int n_min, int n_max, int32_t *draft_out, int32_t *k_out) {
    pdl_wait_prior_grid();
    pdl_launch_dependents();
    // buf[kMaxN + i] = ctx[t0 + i]; buf[0 .. kMaxN) holds the kMaxN tokens before the tile (the halo)
    __shared__ int32_t buf[kMaxN + kTile];
    __shared__ int32_t suf[kMaxN];
    __shared__ unsigned long long s_best[kThreads / 32];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long s0 = ctx_offsets[b];
    long long L = static_cast<long long>(ctx_offsets[b + 1]) - s0;
    if (L < 0) L = 0;  // decreasing offsets: an empty context, nothing proposed
    const int32_t *ctx = tokens + s0;
    if (tid < n_max && tid < L) suf[tid] = ctx[L - 1 - tid];
    // key = m << 32 | e, 0 = no candidate (m >= n_min >= 1 makes every real key nonzero)
    unsigned long long best = 0ull;
    int32_t v[kPerThread];  // the next tile, loaded while the current one is compared
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
        const long long i = j * kThreads + tid;
        v[j] = i < L ? ctx[i] : 0;
    }
    for (long long t0 = 0; t0 <= L - 2; t0 += kTile) {
        const long long n_here = (L - 1 - t0) < kTile ? (L - 1 - t0) : kTile;  // candidate ends t0 .. t0 + n_here - 1
        __syncthreads();  // the previous tile's compares are done
        if (tid < kMaxN) {
            const long long i = t0 - kMaxN + tid;
            buf[tid] = (t0 > 0 && i >= 0) ? buf[kTile + tid] : 0;  // last kMaxN tokens of the previous tile
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kPerThread; ++j) buf[kMaxN + j * kThreads + tid] = v[j];
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kPerThread; ++j) {  // independent loads of the next tile, in flight during the compares
            const long long i = t0 + kTile + j * kThreads + tid;
            v[j] = i < L ? ctx[i] : 0;
        }
        for (int i = tid; i < n_here; i += kThreads) {
            const long long e = t0 + i;
            const int lim = static_cast<int>(e + 1 < n_max ? e + 1 : n_max);
            int m = 0;
            while (m < lim && buf[kMaxN + i - m] == suf[m]) ++m;
            if (m >= n_min) {
                const unsigned long long key = (static_cast<unsigned long long>(m) << 32) | static_cast<unsigned long long>(e);
                best = key > best ? key : best;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
        best = y > best ? y : best;
    }
    if (lane == 0) s_best[warp] = best;
    __syncthreads();
    if (warp == 0) {
        best = lane < kThreads / 32 ? s_best[lane] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
            best = y > best ? y : best;
        }
        if (lane == 0) s_best[0] = best;
    }
    __syncthreads();
    best = s_best[0];
    long long k = 0, e_w = -1;
    if (best != 0ull) {
        e_w = static_cast<long long>(best & 0xffffffffull);
        k = L - 1 - e_w;
        if (k > K) k = K;
    }
    for (int j = tid; j < K; j += kThreads)
        draft_out[static_cast<size_t>(b) * K + j] = (j < k) ? ctx[e_w + 1 + j] : -1;
    if (tid == 0) k_out[b] = static_cast<int32_t>(k);
}

}  // namespace ng
}  // namespace sv

using namespace sv;

extern "C" sv_status spec_ngram_draft(const int32_t *tokens, const int32_t *ctx_offsets, int B, int K, int n_min,
                                      int n_max, int32_t *draft_out, int32_t *k_out, void *stream) {
    if (B < 0 || K < 0 || K > SV_MAX_K || n_min < 1 || n_max < n_min || n_max > ng::kMaxN) return SV_ERR_INVALID;
    if (B == 0) {
        set_launches(0);
        return SV_OK;
    }
    if (!tokens || !ctx_offsets || !k_out || (K > 0 && !draft_out)) return SV_ERR_INVALID;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B);
    cfg.blockDim = dim3(ng::kThreads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e =
        cudaLaunchKernelEx(&cfg, ng::ngram_kernel, tokens, ctx_offsets, K, n_min, n_max, draft_out, k_out);
    set_launches(1);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
