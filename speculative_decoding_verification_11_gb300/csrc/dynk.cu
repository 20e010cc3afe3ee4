// Dynamic draft length (K) after verification, on the device: the accept
// lengths never leave the GPU between a verification and the next step's
// drafting.  "Hardware Aware Dynamic Speculative Decoding", section "Dynamic
// speculative decoding" (K adapted to
// the hardware and the acceptance; goodput = AL / ITL, an offline table that
// can take live AL and ITL statistics) and "Speculative Decoding in
// Production: Accelerating LLM Inference via Custom Draft Models",
// "Production Failure Modes and Mitigation Strategies", item 1 (dynamic window
// sizing: K from 5 down to 1 or 2 when the running average of accepted tokens
// over the last 10 falls below 1.5).
//
// Per request: a ring of its last W results (AL, K used).  Window rule: the
// mean AL over the ring against a threshold.  Goodput rule: alpha = S / (S +
// F) over the ring (S accepted drafts, F rejections), E(K) = 1 + alpha + ...
// + alpha^K, K_next = argmax E(K) / itl[K].  All decisions in fp32 with
// explicit round-to-nearest operations, in a fixed order.  One CTA: one
// thread per request in tiles of 1024, then a block-wide scan for the row
// offsets of the next ragged verification.
#include <cmath>
#include <cstdint>

#include "../../include/specverify.h"
#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {
namespace dk {

constexpr int kThreads = 1024;

__device__ __forceinline__ long long block_exclusive_scan(long long v, long long *total) {
    __shared__ long long warp_sum[kThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        long long w = warp_sum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sum[lane] = w;
    }
    __syncthreads();
    const long long pre = (warp > 0 ? warp_sum[warp - 1] : 0ll) + incl - v;
    *total = warp_sum[kThreads / 32 - 1];
    __syncthreads();
    return pre;
}

__global__ void __launch_bounds__(kThreads) dynk_kernel(const int32_t *accept_len, const int32_t *k_used,
                                                        int32_t *hist, int32_t *count, int B, int W, int policy,
                                                        float threshold, int k_low, int k_high, const float *itl,
                                                        float alpha_prior, int32_t *k_next, int32_t *row_offsets) {
    pdl_wait_prior_grid();  // accept_len comes from the verification before it
    pdl_launch_dependents();
    const int tid = threadIdx.x;
    long long carry = 0;
    for (int b0 = 0; b0 < B; b0 += kThreads) {
        const int b = b0 + tid;
        int kn = 0;
        if (b < B) {
            const int al = accept_len[b], k = k_used[b];
            int c = count[b];
            int32_t *ring = hist + static_cast<size_t>(b) * W * 2;
            if (al > 0) {  // an invalid request (AL = 0) leaves no result
                const int slot = c % W;
                ring[2 * slot] = al;
                ring[2 * slot + 1] = k;
                ++c;
                count[b] = c;
            }
            const int n = c < W ? c : W;
            if (policy == SV_DYNK_WINDOW) {
                if (n == 0) {
                    kn = k_high;
                } else {
                    long long tot = 0;
                    for (int i = 0; i < n; ++i) tot += ring[2 * i];
                    const float mean = __fdiv_rn(__ll2float_rn(tot), __int2float_rn(n));
                    kn = mean < threshold ? k_low : k_high;
                }
            } else {
                long long S = 0, F = 0;
                for (int i = 0; i < n; ++i) {
                    const int a = ring[2 * i], kk = ring[2 * i + 1];
                    S += a - 1;
                    F += (a - 1 < kk) ? 1 : 0;
                }
                const float alpha = (S + F == 0) ? alpha_prior : __fdiv_rn(__ll2float_rn(S), __ll2float_rn(S + F));
                float e = 1.f, p = 1.f, best_g = 0.f;
                kn = k_low;
                bool have = false;
                for (int K = 0; K <= k_high; ++K) {
                    if (K > 0) {
                        p = __fmul_rn(p, alpha);
                        e = __fadd_rn(e, p);
                    }
                    if (K < k_low) continue;
                    const float g = __fdiv_rn(e, itl[K]);
                    if (!have || g > best_g) {
                        kn = K;
                        best_g = g;
                        have = true;
                    }
                }
            }
            k_next[b] = kn;
        }
        if (row_offsets) {
            long long tile;
            const long long pre = block_exclusive_scan(b < B ? kn + 1 : 0, &tile);
            if (b < B) row_offsets[b] = static_cast<int32_t>(carry + pre);
            carry += tile;
        }
    }
    if (row_offsets && tid == 0) row_offsets[B] = static_cast<int32_t>(carry);
}

}  // namespace dk
}  // namespace sv

using namespace sv;

extern "C" sv_status spec_dynk_update(const int32_t *accept_len, const int32_t *k_used, int32_t *hist,
                                      int32_t *count, int B, int W, int policy, float threshold, int k_low,
                                      int k_high, const float *itl, float alpha_prior, int32_t *k_next,
                                      int32_t *row_offsets, void *stream) {
    if (B < 0 || W < 1 || k_low < 0 || k_high < k_low || k_high > SV_MAX_K ||
        (policy != SV_DYNK_WINDOW && policy != SV_DYNK_GOODPUT))
        return SV_ERR_INVALID;
    if (policy == SV_DYNK_WINDOW && !std::isfinite(threshold)) return SV_ERR_INVALID;
    if (policy == SV_DYNK_GOODPUT && (!itl || !(alpha_prior >= 0.f && alpha_prior <= 1.f))) return SV_ERR_INVALID;
    if (B == 0) {
        set_launches(0);
        return SV_OK;
    }
    if (!accept_len || !k_used || !hist || !count || !k_next) return SV_ERR_INVALID;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(dk::kThreads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, dk::dynk_kernel, accept_len, k_used, hist, count, B, W, policy,
                                             threshold, k_low, k_high, itl, alpha_prior, k_next, row_offsets);
    set_launches(1);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
