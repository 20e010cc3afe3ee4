// Model-free n-gram (prompt lookup) drafter: proposes the tokens that
// followed the latest earlier occurrence of the context's longest matching
// suffix.  "Co-Designing AI Models Using Speculative Decoding for Faster LLM
// Inference", Table 1 (suffix / n-gram: string matching over the token
// stream, no model, one lookup), and the model-free passage of "Speculative
// Decoding" (glossary), section "Variants: Draft Models, EAGLE, Medusa, and
// Model-Free Methods" (prompt lookup matches strings already in the context).
//
// One cluster of kSplit CTAs per request: CTA s of the cluster takes the
// s-th quarter of the candidate end positions e <= L - 2 and measures, for
// each, m(e), the length of the common suffix of ctx[..e] and ctx[..L-1] (at
// most min(n_max, e + 1)); its range of the context (with the kMaxN tokens
// before it) passes through shared memory in tiles of kTile tokens, copied
// asynchronously.  The winner maximises (m, e) with m >= n_min: the longest
// suffix first, then its latest occurrence -- the order in which the method
// tries n = n_max .. n_min and scans back from the end.  Each CTA's best
// (m, e) goes to the first CTA of the cluster through distributed shared
// memory; that CTA writes the proposal.  Splitting a context over four CTAs
// divides its copy latency and its compares by four; the compares read four
// candidate ends at a time and test them against the context's last token
// first, so that only the few that match it are extended.
#include <cstdint>

#include "../../include/specverify.h"
#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {
namespace ng {

constexpr int kSplit = 4;       // CTAs per request (one cluster)
constexpr int kThreads = 256;
constexpr int kMaxN = 32;
constexpr int kTile = 4096;     // candidate ends (and context tokens) staged in shared memory at a time

__device__ __forceinline__ void cp_async_4(int32_t *dst, const int32_t *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

__global__ void __launch_bounds__(kThreads) ngram_kernel(const int32_t *tokens, const int32_t *ctx_offsets, int K,
                                                         int n_min, int n_max, int32_t *draft_out, int32_t *k_out) {
    cluster_arrive_relaxed();  // matched by the wait before the first remote store
    pdl_wait_prior_grid();
    pdl_launch_dependents();
    // buf[kMaxN + i] = ctx[t0 + i]; buf[0 .. kMaxN) = the kMaxN tokens before the tile (zero before ctx[0])
    __shared__ __align__(16) int32_t buf[kMaxN + kTile + 4];
    __shared__ int32_t suf[kMaxN];
    __shared__ unsigned long long s_best[kThreads / 32];
    __shared__ unsigned long long s_keys[kSplit];  // the first CTA: every CTA's best key
    const int b = blockIdx.x, part = static_cast<int>(cluster_ctarank());
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long s0 = ctx_offsets[b];
    long long L = static_cast<long long>(ctx_offsets[b + 1]) - s0;
    if (L < 0) L = 0;  // decreasing offsets: an empty context, nothing proposed
    const int32_t *ctx = tokens + s0;
    if (tid < n_max && tid < L) suf[tid] = ctx[L - 1 - tid];
    const long long n_cand = L >= 2 ? L - 1 : 0;  // candidate ends 0 .. L - 2
    const long long chunk = (n_cand + kSplit - 1) / kSplit;
    const long long c0 = part * chunk, c1 = (c0 + chunk < n_cand) ? c0 + chunk : n_cand;
    // key = m << 32 | e, 0 = no candidate (m >= n_min >= 1 makes every real key nonzero)
    unsigned long long best = 0ull;
    for (long long t0 = c0; t0 < c1; t0 += kTile) {
        const int n_here = static_cast<int>((c1 - t0) < kTile ? (c1 - t0) : kTile);
        __syncthreads();  // the previous tile's compares are done (and suf is written)
        for (int i = tid; i < kMaxN + n_here; i += kThreads) {
            const long long src = t0 - kMaxN + i;
            if (src >= 0) cp_async_4(buf + i, ctx + src);
            else buf[i] = 0;
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        // four candidate ends per 16-byte read, each first tested against the context's last token;
        // only those that match it (rare) are extended backwards
        const int32_t last = suf[0];
        for (int i4 = tid * 4; i4 < n_here; i4 += kThreads * 4) {
            const int4 w = *reinterpret_cast<const int4 *>(buf + kMaxN + i4);
            const int32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = i4 + q;
                if (i < n_here && v[q] == last) {
                    const long long e = t0 + i;
                    const int lim = static_cast<int>(e + 1 < n_max ? e + 1 : n_max);
                    int m = 1;
                    while (m < lim && buf[kMaxN + i - m] == suf[m]) ++m;
                    if (m >= n_min) {
                        const unsigned long long key =
                            (static_cast<unsigned long long>(m) << 32) | static_cast<unsigned long long>(e);
                        best = key > best ? key : best;
                    }
                }
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
    }
    cluster_wait();  // every CTA of the cluster runs: the first one's shared memory is valid
    if (tid == 0)
        st_dsmem_f32x2(reinterpret_cast<float2 *>(&s_keys[part]), __uint_as_float(static_cast<uint32_t>(best)),
                       __uint_as_float(static_cast<uint32_t>(best >> 32)), 0);
    cluster_sync();  // the keys are in; no CTA touches another's shared memory after this
    if (part != 0) return;
    best = 0ull;
#pragma unroll
    for (int i = 0; i < kSplit; ++i) best = s_keys[i] > best ? s_keys[i] : best;
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
    cfg.gridDim = dim3(B, ng::kSplit);
    cfg.blockDim = dim3(ng::kThreads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;  // the kSplit CTAs of a request form one cluster
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = ng::kSplit;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t e =
        cudaLaunchKernelEx(&cfg, ng::ngram_kernel, tokens, ctx_offsets, K, n_min, n_max, draft_out, k_out);
    set_launches(1);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
