// Paged KV-cache bookkeeping around the verification step: reserve the blocks
// of the speculative slots before the draft and target passes, and give back
// the blocks of the rejected slots after verification.
//
// "Speculative Decoding in Large Language Models: Architecture, Mathematical
// Foundations, and Production Engineering", section 4, "Segmented Block
// Allocation (PagedAttention)": fixed-size blocks, block pointers handed out
// for the speculative tokens, and a rejection returns the pointers of the
// evicted positions to the global free list with no copy.  "Speculative
// Decoding in Production: Accelerating LLM Inference via Custom Draft Models",
// "Serving Architecture and KV Cache Syncing": with M of K drafts accepted,
// K - M speculative slots are evicted, in the draft's cache and the target's.
//
// Only block ids move: O(blocks touched) integer work per request and no KV
// data.  One CTA does the whole batch in two passes (validate and count,
// then assign stack slots by a block-wide prefix sum in request order), so a
// call is deterministic and a rejected call changes nothing.
#include <cstdint>

#include "../../include/specverify.h"
#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {
namespace kvb {

constexpr int kThreads = 1024;

__device__ __forceinline__ long long blocks_for(long long n, int bs) { return (n + bs - 1) / bs; }

// Exclusive prefix of v over the CTA's threads in thread order; *total = the sum.
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
    __syncthreads();  // warp_sum is reused by the next call
    return pre;
}

__global__ void __launch_bounds__(kThreads) reserve_kernel(int32_t *block_table, const int32_t *seq_len,
                                                           const int32_t *free_ids, int32_t *free_count,
                                                           const int32_t *n_new, int B, int max_blocks, int bs,
                                                           uint32_t *status) {
    pdl_wait_prior_grid();
    pdl_launch_dependents();
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    if (tid == 0) s_bad = 0;
    __syncthreads();
    // pass 1: validate every request and count the blocks to take
    long long cnt = 0;
    bool bad = false;
    for (int b = tid; b < B; b += kThreads) {
        const long long len = seq_len[b], n = n_new[b];
        if (len < 0 || n < 0 || blocks_for(len + n, bs) > max_blocks) {
            bad = true;
            continue;
        }
        const long long have = blocks_for(len, bs), want = blocks_for(len + n, bs);
        const int32_t *row = block_table + static_cast<size_t>(b) * max_blocks;
        for (long long i = have; i < want; ++i) bad |= (row[i] >= 0);  // would leak the block held there
        cnt += want - have;
    }
    if (bad) atomicOr(&s_bad, 1);
    long long total;
    block_exclusive_scan(cnt, &total);
    const int fc = *free_count;
    if (s_bad || total > fc) {
        if (tid == 0) atomicOr(status, s_bad ? SV_FLAG_KV_BAD_INPUT : SV_FLAG_KV_OUT_OF_BLOCKS);
        return;
    }
    // pass 2: request b takes stack slots base + (blocks of the requests before it) + i
    const long long base = fc - total;
    long long carry = 0;
    for (int b0 = 0; b0 < B; b0 += kThreads) {
        const int b = b0 + tid;
        long long have = 0, need = 0;
        if (b < B) {
            const long long len = seq_len[b];
            have = blocks_for(len, bs);
            need = blocks_for(len + n_new[b], bs) - have;
        }
        long long tile;
        const long long pre = block_exclusive_scan(need, &tile);
        if (b < B) {
            int32_t *row = block_table + static_cast<size_t>(b) * max_blocks;
            for (long long i = 0; i < need; ++i) row[have + i] = free_ids[base + carry + pre + i];
        }
        carry += tile;
    }
    if (tid == 0) *free_count = static_cast<int32_t>(base);
}

__global__ void __launch_bounds__(kThreads) rollback_kernel(int32_t *block_table, int32_t *seq_len,
                                                            int32_t *free_ids, int32_t *free_count,
                                                            const int32_t *n_spec, const int32_t *accept_len,
                                                            int B, int max_blocks, int bs, int capacity,
                                                            uint32_t *status) {
    pdl_wait_prior_grid();  // accept_len comes from the verification kernel before it
    pdl_launch_dependents();
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    if (tid == 0) s_bad = 0;
    __syncthreads();
    // pass 1: validate every request and count the blocks to give back
    long long cnt = 0;
    bool bad = false;
    for (int b = tid; b < B; b += kThreads) {
        const long long len = seq_len[b], n = n_spec[b], al = accept_len[b];
        if (len < 0 || n < 0 || al < 0 || al > n + 1 || blocks_for(len + n, bs) > max_blocks) {
            bad = true;
            continue;
        }
        const long long new_len = len + (al > 0 ? al - 1 : 0);
        const long long lo = blocks_for(new_len, bs), hi = blocks_for(len + n, bs);
        const int32_t *row = block_table + static_cast<size_t>(b) * max_blocks;
        for (long long i = lo; i < hi; ++i) bad |= (row[i] < 0);  // a block to give back is missing
        cnt += hi - lo;
    }
    if (bad) atomicOr(&s_bad, 1);
    long long total;
    block_exclusive_scan(cnt, &total);
    const int fc = *free_count;
    if (s_bad || fc + total > capacity) {
        if (tid == 0) atomicOr(status, SV_FLAG_KV_BAD_INPUT);
        return;
    }
    // pass 2: request b's blocks go to stack slots fc + (blocks of the requests before it) + i
    long long carry = 0;
    for (int b0 = 0; b0 < B; b0 += kThreads) {
        const int b = b0 + tid;
        long long lo = 0, cntb = 0, new_len = 0;
        if (b < B) {
            const long long len = seq_len[b], al = accept_len[b];
            new_len = len + (al > 0 ? al - 1 : 0);
            lo = blocks_for(new_len, bs);
            cntb = blocks_for(len + n_spec[b], bs) - lo;
        }
        long long tile;
        const long long pre = block_exclusive_scan(cntb, &tile);
        if (b < B) {
            int32_t *row = block_table + static_cast<size_t>(b) * max_blocks;
            for (long long i = 0; i < cntb; ++i) {
                free_ids[fc + carry + pre + i] = row[lo + i];
                row[lo + i] = -1;
            }
            seq_len[b] = static_cast<int32_t>(new_len);
        }
        carry += tile;
    }
    if (tid == 0) *free_count = static_cast<int32_t>(fc + total);
}

template <typename KernelT, typename... Args>
static cudaError_t launch_one_cta(KernelT kernel, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace kvb
}  // namespace sv

using namespace sv;

extern "C" sv_status spec_kv_reserve(int32_t *block_table, const int32_t *seq_len, const int32_t *free_ids,
                                     int32_t *free_count, const int32_t *n_new, int B, int max_blocks,
                                     int block_size, uint32_t *status, void *stream) {
    if (B < 0 || max_blocks <= 0 || block_size <= 0) return SV_ERR_INVALID;
    if (B == 0) {
        set_launches(0);
        return SV_OK;
    }
    if (!block_table || !seq_len || !free_ids || !free_count || !n_new || !status) return SV_ERR_INVALID;
    const cudaError_t e = kvb::launch_one_cta(kvb::reserve_kernel, static_cast<cudaStream_t>(stream), block_table,
                                              seq_len, free_ids, free_count, n_new, B, max_blocks, block_size, status);
    set_launches(1);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" sv_status spec_kv_rollback(int32_t *block_table, int32_t *seq_len, int32_t *free_ids,
                                      int32_t *free_count, const int32_t *n_spec, const int32_t *accept_len, int B,
                                      int max_blocks, int block_size, int capacity, uint32_t *status,
                                      void *stream) {
    if (B < 0 || max_blocks <= 0 || block_size <= 0 || capacity < 0) return SV_ERR_INVALID;
    if (B == 0) {
        set_launches(0);
        return SV_OK;
    }
    if (!block_table || !seq_len || !free_ids || !free_count || !n_spec || !accept_len || !status)
        return SV_ERR_INVALID;
    const cudaError_t e =
        kvb::launch_one_cta(kvb::rollback_kernel, static_cast<cudaStream_t>(stream), block_table, seq_len, free_ids,
                            free_count, n_spec, accept_len, B, max_blocks, block_size, capacity, status);
    set_launches(1);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
