// Verification kernels and the C ABI of libspecverify.so (sm_103a).
//
// Pass 1  stats_tma_kernel (rows 16-byte aligned) / stats_scalar_kernel (any)
//         streams every logit once and reduces each 32 KB chunk of a row to
//         (M, s) = (max z c, sum 2^(z c - M)) with c = log2(e)/T (sampling) or
//         to (max z, first argmax) (greedy).  The TMA variant is persistent:
//         one CTA per SM, a producer warp feeding a 6-stage shared ring with
//         bulk async copies, 8 consumer warps that need no block barrier.
//         The arrival that completes a request's count (release atomic) runs
//         the decide step in one warp: accept tests u q(x) <= p(x), ballot
//         for the first rejection, emitted drafts, AL, and the record of the
//         row the final token comes from.
// Pass 2  residual_kernel (sampling only) one cluster of 1-8 CTAs per request over
//         the selected row, one warp per 1024-token tile: r = max(0, p - q)
//         at a rejection or r = p for the bonus, tile masses in shared
//         memory; rank 0 takes the prefix over tiles in fp64 through
//         distributed shared memory, finds the tile holding u R, and resolves
//         the token inside it with the same warp scan that produced the
//         tile's mass.
//
// The operation is the one stated on "Speculative Decoding in Large Language
// Models", section 2 "Modified Rejection Sampling" (accept test, residual
// p'(x)), with the stop at the first mismatch and the extra target token of
// "Co-Designing AI Models Using Speculative Decoding", "What is speculative
// decoding?".  See include/specverify.h for the full contract.
#include <cmath>
#include <cstdio>
#include <cstring>

#include "../../include/specverify.h"
#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

// ---------------------------------------------------------------------------
// Shared state between the passes (lives in the caller's workspace)
// ---------------------------------------------------------------------------
struct Decision {
    int row;     // logits row the final token is drawn from
    int qrow;    // q row to subtract (rejection), -1 for the bonus draw
    int slot;    // out_tokens index of the final token
    int valid;   // 0 for an invalid request (nothing to draw)
    float M;     // row max of z c (log2 units)
    float invS;  // 1 / sum 2^(z c - M)
    float u;     // final uniform u_K
    int pad;
};

struct Args {
    const void *logits;
    const float *q;
    const int32_t *row_offsets;  // nullptr for fixed K
    const int32_t *draft;
    const float *uniforms;
    int32_t *out_tokens;
    int32_t *accept_len;
    float *diag;
    int B, K, V, rows, n_chunks, n_tiles, n_draft;
    float c;  // log2(e) / T
    // workspace
    uint32_t *status;
    const int *csr_ok;
    uint32_t *tickets1;
    Decision *dec;
    float2 *partials;
    float *tile_mass;
};

constexpr long long kWaitBudget = 4000000000ll;  // SM cycles (~2 s) before a wait gives up

__device__ __forceinline__ void request_rows(const Args &a, int b, int &r0, int &nr) {
    if (a.row_offsets) {
        r0 = __ldg(a.row_offsets + b);
        nr = __ldg(a.row_offsets + b + 1) - r0;
    } else {
        r0 = b * (a.K + 1);
        nr = a.K + 1;
    }
}

// Request that owns logits row r (offsets already validated in ragged mode).
__device__ __forceinline__ int request_of_row(const Args &a, int r) {
    if (!a.row_offsets) return r / (a.K + 1);
    int lo = 0, hi = a.B;  // invariant: ro[lo] <= r < ro[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(a.row_offsets + mid) <= r) lo = mid; else hi = mid;
    }
    return lo;
}

template <typename T>
__device__ __forceinline__ float logit_at(const Args &a, size_t i) {
    return Elem<T>::at(reinterpret_cast<const T *>(a.logits), i);
}

template <bool kSample>
__device__ __forceinline__ void warp_partial_reduce(float &ra, int &rb) {
    if (kSample) {
        float s = __int_as_float(rb);
        warp_ms_reduce(ra, s);
        rb = __float_as_int(s);
    } else {
        warp_am_reduce(ra, rb);
    }
}

template <bool kSample>
__device__ __forceinline__ void merge_pair(float &ra, int &rb, float2 w) {
    if (kSample) {
        float s = __int_as_float(rb);
        ms_merge(ra, s, w.x, w.y);
        rb = __float_as_int(s);
    } else {
        am_merge(ra, rb, w.x, __float_as_int(w.y));
    }
}

// ---------------------------------------------------------------------------
// Decide step of request b, run by one warp once every chunk partial of the
// request's rows is visible.  Lane j owns row jb + j: it merges the row's
// chunk partials in chunk order, evaluates the accept test of its draft, and
// a ballot finds the first rejection.
// ---------------------------------------------------------------------------
template <typename T, bool kSample>
__device__ void decide_warp(const Args &a, int b, int lane) {
    int r0, nr;
    request_rows(a, b, r0, nr);
    const int Kb = nr - 1;
    const int d0 = r0 - b;
    if (lane == 0) a.tickets1[b] = 0u;  // every arrival of this call is in: leave the counter clean
    bool bad = false;
    for (int j = lane; j < Kb; j += 32) {
        const int x = __ldg(a.draft + d0 + j);
        bad |= (x < 0 || x >= a.V);
    }
    if (__any_sync(0xffffffffu, bad)) {
        for (int j = lane; j < nr; j += 32) a.out_tokens[r0 + j] = -1;
        if (lane == 0) {
            a.accept_len[b] = 0;
            if (kSample) {
                Decision d{};
                a.dec[b] = d;
            }
            atomicOr(a.status, SV_FLAG_BAD_TOKEN);
        }
        return;
    }
    int ks = Kb;
    float Msel = 0.f, Ssel = 1.f;
    int argsel = 0;
    for (int jb = 0; jb < nr; jb += 32) {
        const int j = jb + lane;
        // gathers of this block's drafts first: their latency overlaps the merges
        int x = 0;
        float z = 0.f, qv = 0.f, u = 0.f;
        if (j < Kb) {
            x = __ldg(a.draft + d0 + j);
            if (kSample) {
                z = logit_at<T>(a, static_cast<size_t>(r0 + j) * a.V + x);
                qv = __ldg(a.q + static_cast<size_t>(d0 + j) * a.V + x);
                u = __ldg(a.uniforms + r0 + j);
            }
        }
        // merge the chunk partials of rows jb .. jb+31: lanes over chunks, all
        // loads of a row issued together, butterfly across lanes
        float M = -INFINITY, S = 0.f, bv = -INFINITY;
        int bi = 0x7fffffff;
        const int rows_here = min(32, nr - jb);
        for (int rg = 0; rg < rows_here; rg += 8) {
            float ma[8];
            int mb[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                ma[i] = -INFINITY;
                mb[i] = kSample ? __float_as_int(0.f) : 0x7fffffff;
            }
            for (int c = lane; c < a.n_chunks; c += 32) {
                float2 w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)  // 8 rows' loads in flight together
                    w[i] = (rg + i < rows_here)
                               ? __ldcg(a.partials + static_cast<size_t>(r0 + jb + rg + i) * a.n_chunks + c)
                               : make_float2(-INFINITY, kSample ? 0.f : __int_as_float(0x7fffffff));
#pragma unroll
                for (int i = 0; i < 8; ++i) merge_pair<kSample>(ma[i], mb[i], w[i]);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                warp_partial_reduce<kSample>(ma[i], mb[i]);
                if (lane == rg + i) {
                    if (kSample) {
                        M = ma[i];
                        S = __int_as_float(mb[i]);
                    } else {
                        bv = ma[i];
                        bi = mb[i];
                    }
                }
            }
        }
        bool rej = false;
        if (j < Kb) {
            if (kSample) {
                const float p = exp2f(fmaf(z, a.c, -M)) / S;
                rej = !(u * qv <= p);
                if (a.diag) a.diag[d0 + j] = p;
            } else {
                rej = (x != bi);
            }
        }
        const unsigned m = __ballot_sync(0xffffffffu, rej);
        if (m || jb + 32 >= nr) {
            const int src = m ? (__ffs(m) - 1) : (Kb - jb);
            ks = jb + src;
            Msel = __shfl_sync(0xffffffffu, M, src);
            Ssel = __shfl_sync(0xffffffffu, S, src);
            argsel = __shfl_sync(0xffffffffu, bi, src);
            break;
        }
    }
    for (int j = lane; j < nr; j += 32) {
        int v = -1;
        if (j < ks) v = __ldg(a.draft + d0 + j);
        else if (j == ks && !kSample) v = argsel;
        a.out_tokens[r0 + j] = v;
    }
    if (lane == 0) {
        a.accept_len[b] = ks + 1;
        if (kSample) {
            Decision d;
            d.row = r0 + ks;
            d.qrow = (ks < Kb) ? d0 + ks : -1;
            d.slot = r0 + ks;
            d.valid = 1;
            d.M = Msel;
            d.invS = 1.f / Ssel;
            d.u = __ldg(a.uniforms + r0 + Kb);
            d.pad = 0;
            a.dec[b] = d;
        }
    }
}

// Reduce `vals` (this lane's elements, element (j, k) valid when idx(j,k) < n)
// to the lane's partial: sampling (M, s) or greedy (max, first index).
template <bool kSample, int VEC>
__device__ __forceinline__ void lane_partial(const float (&vals)[kLoadsPerThread][VEC], const int (&e0)[kLoadsPerThread],
                                             int n, int c0, float c, float &ra, int &rb) {
    if (kSample) {
        float bm = -INFINITY;
#pragma unroll
        for (int j = 0; j < kLoadsPerThread; ++j)
#pragma unroll
            for (int k = 0; k < VEC; ++k)
                if (e0[j] + k < n) bm = fmaxf(bm, vals[j][k]);
        const float M = bm * c;
        float s = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int j = 0; j < kLoadsPerThread; ++j)
#pragma unroll
                for (int k = 0; k < VEC; ++k)
                    if (e0[j] + k < n) s += ex2(fmaf(vals[j][k], c, -M));
        }
        ra = M;
        rb = __float_as_int(s);
    } else {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < kLoadsPerThread; ++j)
#pragma unroll
            for (int k = 0; k < VEC; ++k)
                if (e0[j] + k < n && (bi == 0x7fffffff || vals[j][k] > bv)) {
                    bv = vals[j][k];
                    bi = c0 + e0[j] + k;
                }
        ra = bv;
        rb = bi;
    }
}



// Publish the chunk partial of (row, chunk); the arrival that completes the
// request's count runs the decide step.  Called by one whole warp.
template <typename T, bool kSample>
__device__ __forceinline__ void publish_partial(const Args &a, int row, int chunk, float ra, int rb, int lane) {
    int islast = 0, b = 0;
    if (lane == 0) {
        a.partials[static_cast<size_t>(row) * a.n_chunks + chunk] = make_float2(ra, __int_as_float(rb));
        b = request_of_row(a, row);
        int r0, nr;
        request_rows(a, b, r0, nr);
        const uint32_t old = atom_add_release_gpu(a.tickets1 + b, 1u);
        islast = (old + 1u == static_cast<uint32_t>(nr) * static_cast<uint32_t>(a.n_chunks));
        if (islast) fence_acq_rel_gpu();
    }
    islast = __shfl_sync(0xffffffffu, islast, 0);
    b = __shfl_sync(0xffffffffu, b, 0);
    if (islast) decide_warp<T, kSample>(a, b, lane);
}

// ---------------------------------------------------------------------------
// Pass 1, aligned rows: persistent CTA per SM over a contiguous range of
// (row, chunk) items.
//   warp 16 (producer)  streams 32 KB chunks with bulk async copies into a
//                       kStages-deep shared ring (full/empty mbarriers);
//   warps 0-15 (consumers) each reduce a 2 KB slice of every chunk into a
//                       per-lane running partial of the current row segment;
//                       at a row boundary each posts its warp partial to a
//                       mailbox slot (mbarrier, 16 arrivals) and goes on;
//   warp 17 (publisher) merges the 16 posts in warp order, writes the
//                       segment's chunk partials, adds the segment's chunk
//                       count to the request's counter (release atomic) and,
//                       on the arrival that completes the count, runs the
//                       decide step.
// Consumers never wait on global memory or on each other.
// ---------------------------------------------------------------------------
constexpr int kStages = 6;
constexpr int kChunkBytes = 32768;
constexpr int kConsumerWarps = 16;
constexpr int kTmaVecs = kChunkBytes / 16 / (kConsumerWarps * 32);  // 16-byte vectors per lane per chunk
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kPublisherWarp = kConsumerWarps + 1;
constexpr int kTmaThreads = (kConsumerWarps + 2) * 32;
constexpr int kSegSlots = 4;

struct SegMsg {
    int row, first_chunk, n_chunk, pad;
};

struct TmaSmem {
    alignas(128) unsigned char ring[kStages][kChunkBytes];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t seg_full[kSegSlots];
    uint64_t seg_empty[kSegSlots];
    float2 segpart[kSegSlots][kConsumerWarps];
    SegMsg seg[kSegSlots];
    int abort;
};

// Fold one chunk slice into the lane's running partial.  Vector j (VEC
// consecutive tokens) is valid iff e0[j] < n (n is a multiple of VEC on this
// path).  Max and sum run as trees over independent per-vector values.
template <bool kSample, int NV, int VEC>
__device__ __forceinline__ void lane_accumulate(const float (&vals)[NV][VEC], const int (&e0)[NV], int n, int c0,
                                                float c, float &ra, int &rb) {
    if (kSample) {
        float vm[NV];
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            float m = vals[j][0];
#pragma unroll
            for (int k = 1; k < VEC; ++k) m = fmaxf(m, vals[j][k]);
            vm[j] = (e0[j] < n) ? m : -INFINITY;
        }
#pragma unroll
        for (int w = 1; w < NV; w <<= 1)
#pragma unroll
            for (int j = 0; j + w < NV; j += 2 * w) vm[j] = fmaxf(vm[j], vm[j + w]);
        const float bm = vm[0];
        if (bm != -INFINITY) {
            const float Mn = fmaxf(ra, bm * c);
            float acc[NV];
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                float e[VEC];
#pragma unroll
                for (int k = 0; k < VEC; ++k) e[k] = ex2(fmaf(vals[j][k], c, -Mn));
#pragma unroll
                for (int w = 1; w < VEC; w <<= 1)
#pragma unroll
                    for (int k = 0; k + w < VEC; k += 2 * w) e[k] += e[k + w];
                acc[j] = (e0[j] < n) ? e[0] : 0.f;
            }
#pragma unroll
            for (int w = 1; w < NV; w <<= 1)
#pragma unroll
                for (int j = 0; j + w < NV; j += 2 * w) acc[j] += acc[j + w];
            const float s_old = __int_as_float(rb) * ex2(ra - Mn);  // ra = -inf: 0
            ra = Mn;
            rb = __float_as_int(s_old + acc[0]);
        }
    } else {
        float vv[NV];
        int vi[NV];
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            float m = vals[j][0];
            int mi = 0;
#pragma unroll
            for (int k = 1; k < VEC; ++k)
                if (vals[j][k] > m) {
                    m = vals[j][k];
                    mi = k;
                }
            vv[j] = (e0[j] < n) ? m : -INFINITY;
            vi[j] = (e0[j] < n) ? c0 + e0[j] + mi : 0x7fffffff;
        }
#pragma unroll
        for (int w = 1; w < NV; w <<= 1)
#pragma unroll
            for (int j = 0; j + w < NV; j += 2 * w) am_merge(vv[j], vi[j], vv[j + w], vi[j + w]);
        if (vi[0] != 0x7fffffff) am_merge(ra, rb, vv[0], vi[0]);
    }
}

template <bool kSample>
__device__ __forceinline__ void partial_identity(float &ra, int &rb) {
    ra = -INFINITY;
    rb = kSample ? __float_as_int(0.f) : 0x7fffffff;
}

template <typename T, bool kSample>
__global__ void __launch_bounds__(kTmaThreads, 1) stats_tma_kernel(Args a) {
    constexpr int VEC = Elem<T>::kVec;
    constexpr int CHUNK = chunk_elems<T>();
    static_assert(CHUNK * sizeof(T) == kChunkBytes, "chunk must fill one ring stage");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    TmaSmem &sm = *reinterpret_cast<TmaSmem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_launch_dependents();  // pass 2 may be scheduled as this grid drains
    if (a.csr_ok && !__ldcg(a.csr_ok)) return;
    const long long total = static_cast<long long>(a.rows) * a.n_chunks;
    const int i0 = static_cast<int>(total * blockIdx.x / gridDim.x);
    const int i1 = static_cast<int>(total * (blockIdx.x + 1) / gridDim.x);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        for (int s = 0; s < kSegSlots; ++s) {
            mbar_init(&sm.seg_full[s], kConsumerWarps);
            mbar_init(&sm.seg_empty[s], 1);
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    volatile int *abort_flag = &sm.abort;
    auto timeout = [&]() {
        *abort_flag = 1;
        atomicOr(a.status, SV_FLAG_TIMEOUT);
    };

    if (warp == kProducerWarp) {
        if (lane == 0) {
            int k = 0;
            for (int item = i0; item < i1; ++item, ++k) {
                const int s = k % kStages;
                if (k >= kStages && !mbar_wait_bounded(&sm.empty[s], ((k / kStages) - 1) & 1, kWaitBudget))
                    timeout();
                if (*abort_flag) {
                    // let the copies already issued into the ring land before leaving
                    for (int kk = max(0, k - kStages); kk < k; ++kk)
                        mbar_wait_bounded(&sm.full[kk % kStages], (kk / kStages) & 1, kWaitBudget);
                    break;
                }
                const int row = item / a.n_chunks;
                const int chunk = item - row * a.n_chunks;
                const int c0 = chunk * CHUNK;
                const int n = min(CHUNK, a.V - c0);
                const T *src = reinterpret_cast<const T *>(a.logits) + static_cast<size_t>(row) * a.V + c0;
                const uint32_t bytes = static_cast<uint32_t>(n) * sizeof(T);
                mbar_arrive_expect_tx(&sm.full[s], bytes);
                bulk_g2s(sm.ring[s], src, bytes, &sm.full[s]);
            }
        }
        return;
    }

    if (warp == kPublisherWarp) {
        const int n_seg = (i1 - 1) / a.n_chunks - i0 / a.n_chunks + 1;
        for (int g = 0; g < n_seg; ++g) {
            const int slot = g % kSegSlots;
            if (!mbar_wait_bounded(&sm.seg_full[slot], (g / kSegSlots) & 1, kWaitBudget)) timeout();
            if (*abort_flag) break;
            const SegMsg msg = sm.seg[slot];
            float ra = -INFINITY;
            int rb = kSample ? __float_as_int(0.f) : 0x7fffffff;
            if (lane == 0)
                for (int w = 0; w < kConsumerWarps; ++w) merge_pair<kSample>(ra, rb, sm.segpart[slot][w]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.seg_empty[slot]);
            // the segment's chunk partials: the merged value in its first chunk,
            // the identity in the others
            float2 *P = a.partials + static_cast<size_t>(msg.row) * a.n_chunks + msg.first_chunk;
            for (int c = lane; c < msg.n_chunk; c += 32) {
                float ia;
                int ib;
                partial_identity<kSample>(ia, ib);
                P[c] = (c == 0) ? make_float2(ra, __int_as_float(rb)) : make_float2(ia, __int_as_float(ib));
            }
            __threadfence();
            __syncwarp();
            int islast = 0, b = 0;
            if (lane == 0) {
                b = request_of_row(a, msg.row);
                int r0, nr;
                request_rows(a, b, r0, nr);
                const uint32_t old = atom_add_release_gpu(a.tickets1 + b, static_cast<uint32_t>(msg.n_chunk));
                islast = (old + msg.n_chunk == static_cast<uint32_t>(nr) * static_cast<uint32_t>(a.n_chunks));
                if (islast) fence_acq_rel_gpu();
            }
            islast = __shfl_sync(0xffffffffu, islast, 0);
            b = __shfl_sync(0xffffffffu, b, 0);
            if (islast) decide_warp<T, kSample>(a, b, lane);
        }
        return;
    }

    // consumers
    int k = 0, g = 0;
    int seg_row = i0 / a.n_chunks;
    int seg_first = i0 - seg_row * a.n_chunks;
    int seg_n = 0;
    float ra;
    int rb;
    partial_identity<kSample>(ra, rb);
    auto post = [&]() -> bool {
        float wa = ra;
        int wb = rb;
        warp_partial_reduce<kSample>(wa, wb);
        const int slot = g % kSegSlots;
        if (g >= kSegSlots && !mbar_wait_bounded(&sm.seg_empty[slot], ((g / kSegSlots) - 1) & 1, kWaitBudget))
            timeout();
        if (*abort_flag) return false;
        if (lane == 0) {
            sm.segpart[slot][warp] = make_float2(wa, __int_as_float(wb));
            if (warp == 0) sm.seg[slot] = SegMsg{seg_row, seg_first, seg_n, 0};
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.seg_full[slot]);
        ++g;
        return true;
    };
    for (int item = i0; item < i1; ++item, ++k) {
        const int row = item / a.n_chunks;
        const int chunk = item - row * a.n_chunks;
        if (row != seg_row) {
            if (!post()) return;
            seg_row = row;
            seg_first = chunk;
            seg_n = 0;
            partial_identity<kSample>(ra, rb);
        }
        const int s = k % kStages;
        if (!mbar_wait_bounded(&sm.full[s], (k / kStages) & 1, kWaitBudget)) timeout();
        if (*abort_flag) return;
        const int c0 = chunk * CHUNK;
        const int n = min(CHUNK, a.V - c0);
        const uint4 *stage = reinterpret_cast<const uint4 *>(sm.ring[s]);
        float vals[kTmaVecs][VEC];
        int e0[kTmaVecs];
#pragma unroll
        for (int j = 0; j < kTmaVecs; ++j) {
            const int v = warp * (kTmaVecs * 32) + j * 32 + lane;
            e0[j] = v * VEC;
            uint4 raw = make_uint4(0u, 0u, 0u, 0u);
            if (e0[j] < n) raw = stage[v];
            unpack(raw, vals[j]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);  // slice consumed: the stage may be refilled
        lane_accumulate<kSample, kTmaVecs, VEC>(vals, e0, n, c0, a.c, ra, rb);
        ++seg_n;
    }
    post();
}

// ---------------------------------------------------------------------------
// Pass 1, any alignment: one CTA per (row, chunk), element loads.
// ---------------------------------------------------------------------------
template <typename T, bool kSample>
__global__ void __launch_bounds__(kThreads) stats_scalar_kernel(Args a) {
    constexpr int VEC = Elem<T>::kVec;
    constexpr int CHUNK = chunk_elems<T>();
    __shared__ float2 wp[kWarps];
    pdl_launch_dependents();
    if (a.csr_ok && !__ldcg(a.csr_ok)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = blockIdx.x / a.n_chunks;
    const int chunk = blockIdx.x - row * a.n_chunks;
    const int c0 = chunk * CHUNK;
    const int n = min(CHUNK, a.V - c0);
    const T *zrow = reinterpret_cast<const T *>(a.logits) + static_cast<size_t>(row) * a.V + c0;
    float vals[kLoadsPerThread][VEC];
    int e0[kLoadsPerThread];
#pragma unroll
    for (int j = 0; j < kLoadsPerThread; ++j) {
        e0[j] = (warp * (kLoadsPerThread * 32) + j * 32 + lane) * VEC;
#pragma unroll
        for (int k = 0; k < VEC; ++k) vals[j][k] = (e0[j] + k < n) ? Elem<T>::at(zrow, e0[j] + k) : 0.f;
    }
    float ra;
    int rb;
    lane_partial<kSample, VEC>(vals, e0, n, c0, a.c, ra, rb);
    warp_partial_reduce<kSample>(ra, rb);
    if (lane == 0) wp[warp] = make_float2(ra, __int_as_float(rb));
    __syncthreads();
    if (warp == 0) {
        if (lane == 0) {
            float ma = -INFINITY;
            int mb = kSample ? __float_as_int(0.f) : 0x7fffffff;
            for (int w = 0; w < kWarps; ++w) merge_pair<kSample>(ma, mb, wp[w]);
            ra = ma;
            rb = mb;
        }
        publish_partial<T, kSample>(a, row, chunk, ra, rb, lane);
    }
}

// ---------------------------------------------------------------------------
// Pass 2: residual masses per 1024-token tile and the inverse-CDF draw.
// One thread-block cluster of C CTAs per request splits the
// selected row's tiles; tile masses stay in each CTA's shared memory.  After a
// cluster barrier, warp 0 of rank 0 reads all masses through distributed
// shared memory, takes the prefix over tiles in fp64 and resolves the token.
//
// A tile is owned by one warp: lane l holds tokens tile*1024 + (j*32 + l)*4 + k,
// j < 8, k < 4.  The running sum in token order is
//   E(j, l, k) = (base_j + excl_j(l)) + pre_k(l),   base_{j+1} = base_j + seg_j
// (Hillis-Steele lane scan per 128-token segment), and the tile's mass is
// E at its last position.  The tile masses that feed the prefix are plain
// sums of the same r values (tree + butterfly); where rounding leaves the
// tile's running sums short of u R, the draw moves on to the next token with
// r > 0, which is what the exact inverse CDF gives up to that rounding.
// ---------------------------------------------------------------------------
constexpr int kMaxResCluster = 8;  // portable cluster size limit
constexpr int kResWarps = 16;
constexpr int kResThreads = kResWarps * 32;

template <typename T> struct TileRaw;
template <> struct TileRaw<float> {
    float4 z[8];
    float4 q[8];
};
template <> struct TileRaw<__nv_bfloat16> {
    uint2 z[8];
    float4 q[8];
};

// Loads of one tile (issued together so they overlap).
template <typename T, bool kVecPath>
__device__ __forceinline__ void warp_tile_load(const T *zrow, const float *qrow, int V, int tile, int lane,
                                               TileRaw<T> &raw) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e0 = tile * kTileElems + (j * 32 + lane) * 4;
        if (kVecPath && e0 + 4 <= V) {
            if constexpr (sizeof(T) == 4) raw.z[j] = __ldg(reinterpret_cast<const float4 *>(zrow + e0));
            else raw.z[j] = __ldg(reinterpret_cast<const uint2 *>(zrow + e0));
            raw.q[j] = qrow ? __ldg(reinterpret_cast<const float4 *>(qrow + e0)) : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            float zz[4], qq[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int e = e0 + k;
                zz[k] = (e < V) ? Elem<T>::at(zrow, e) : -INFINITY;
                qq[k] = (qrow && e < V) ? __ldg(qrow + e) : 0.f;
            }
            if constexpr (sizeof(T) == 4) {
                raw.z[j] = make_float4(zz[0], zz[1], zz[2], zz[3]);
            } else {
                // bf16 values are exact in fp32: keep their upper halves
                raw.z[j] = make_uint2((__float_as_uint(zz[0]) >> 16) | (__float_as_uint(zz[1]) & 0xffff0000u),
                                      (__float_as_uint(zz[2]) >> 16) | (__float_as_uint(zz[3]) & 0xffff0000u));
            }
            raw.q[j] = make_float4(qq[0], qq[1], qq[2], qq[3]);
        }
    }
}

// r(v) of the tile's tokens from its loaded data.  Same arithmetic (no
// contraction) wherever it is called.
template <typename T>
__device__ __forceinline__ void warp_tile_compute(const TileRaw<T> &raw, bool has_q, int V, int tile, float c,
                                                  float M, float invS, int lane, float (&r)[8][4]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e0 = tile * kTileElems + (j * 32 + lane) * 4;
        float z[4];
        if constexpr (sizeof(T) == 4) {
            z[0] = raw.z[j].x; z[1] = raw.z[j].y; z[2] = raw.z[j].z; z[3] = raw.z[j].w;
        } else {
            z[0] = __uint_as_float(raw.z[j].x << 16);
            z[1] = __uint_as_float(raw.z[j].x & 0xffff0000u);
            z[2] = __uint_as_float(raw.z[j].y << 16);
            z[3] = __uint_as_float(raw.z[j].y & 0xffff0000u);
        }
        const float qv[4] = {raw.q[j].x, raw.q[j].y, raw.q[j].z, raw.q[j].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (e0 + k < V) {
                const float p = __fmul_rn(ex2(__fmaf_rn(z[k], c, -M)), invS);
                r[j][k] = has_q ? fmaxf(__fsub_rn(p, qv[k]), 0.f) : p;
            } else {
                r[j][k] = 0.f;
            }
        }
    }
}

struct TileScan {
    int v;       // found token (kFind) or -1
    float rv;    // its r(v)
    float mass;  // tile mass
};

// kFind = false: tile mass (valid in every lane).
// kFind = true : the smallest token v < V of the tile with base + E(v) > t
//                (or -1) and its r(v).
template <bool kFind>
__device__ __forceinline__ TileScan warp_tile_scan(const float (&r)[8][4], int tile, int V, double base_p,
                                                   double t, int lane) {
    float base = 0.f;
    float last = 0.f;
    TileScan res{-1, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float pre[4];
        pre[0] = r[j][0];
        pre[1] = __fadd_rn(pre[0], r[j][1]);
        pre[2] = __fadd_rn(pre[1], r[j][2]);
        pre[3] = __fadd_rn(pre[2], r[j][3]);
        float incl = pre[3];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl = __fadd_rn(incl, y);
        }
        float lex = __shfl_up_sync(0xffffffffu, incl, 1);
        if (lane == 0) lex = 0.f;
        const float seg = __shfl_sync(0xffffffffu, incl, 31);
        const float head = __fadd_rn(base, lex);
        if (kFind) {
            int cand = -1;
            const int e0 = tile * kTileElems + (j * 32 + lane) * 4;
#pragma unroll
            for (int k = 3; k >= 0; --k)
                if (e0 + k < V && base_p + static_cast<double>(__fadd_rn(head, pre[k])) > t) cand = k;
            const unsigned m = __ballot_sync(0xffffffffu, cand >= 0);
            if (m && res.v < 0) {  // first segment holding a crossing (no early exit: keeps r in registers)
                const int src = __ffs(m) - 1;
                const int ck = __shfl_sync(0xffffffffu, cand, src);
                float rsel = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (k == ck) rsel = r[j][k];
                res.v = tile * kTileElems + (j * 32 + src) * 4 + ck;
                res.rv = __shfl_sync(0xffffffffu, rsel, src);
            }
        }
        if (j == 7) last = __shfl_sync(0xffffffffu, __fadd_rn(head, pre[3]), 31);
        base = __fadd_rn(base, seg);
    }
    res.mass = last;
    return res;
}

// Tile mass for the prefix: per-lane tree over its 32 values, butterfly
// across lanes (the running sums of the draw are taken separately, in token
// order, on the one tile the draw lands in).
__device__ __forceinline__ float warp_tile_sum(const float (&r)[8][4]) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (r[j][0] + r[j][1]) + (r[j][2] + r[j][3]);
#pragma unroll
    for (int w = 1; w < 8; w <<= 1)
#pragma unroll
        for (int j = 0; j + w < 8; j += 2 * w) v[j] += v[j + w];
    float x = v[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <typename T, bool kVecPath>
__device__ __forceinline__ float tile_mass_of(const T *zrow, const float *qrow, int V, int tile, const Decision &d,
                                              float c, int lane, float (&r)[8][4]) {
    TileRaw<T> raw;
    warp_tile_load<T, kVecPath>(zrow, qrow, V, tile, lane, raw);
    warp_tile_compute<T>(raw, qrow != nullptr, V, tile, c, d.M, d.invS, lane, r);
    return warp_tile_sum(r);
}

// The draw (warp 0 of the cluster's rank 0).  Tile i's mass lives in the
// shared memory of rank i / per at index i % per; the slow paths keep theirs
// in the workspace.
template <typename T, bool kVecPath>
__device__ __forceinline__ void draw_final(const Args &a, int b, const Decision d, int lane, const float *smass,
                                           int per) {
    const T *zrow = reinterpret_cast<const T *>(a.logits) + static_cast<size_t>(d.row) * a.V;
    const float *qrow = (d.qrow >= 0) ? a.q + static_cast<size_t>(d.qrow) * a.V : nullptr;
    float *gmass = a.tile_mass + static_cast<size_t>(b) * a.n_tiles;
    bool from_smem = true;
    auto mass_at = [&](int i) -> float {
        if (!from_smem) return __ldcg(gmass + i);
        const int owner = i / per;
        return owner == 0 ? smass[i] : ld_dsmem_f32(smass + (i - owner * per), static_cast<uint32_t>(owner));
    };
    double R = 0.0, t = 0.0, fbase = 0.0;
    int ftile = -1;
    for (int attempt = 0; attempt < 2; ++attempt) {
        // fp64 prefix over the tile masses; lane l owns a contiguous group
        const int G = (a.n_tiles + 31) / 32;
        const int i0 = min(lane * G, a.n_tiles), i1 = min(i0 + G, a.n_tiles);
        double sum = 0.0;
        for (int i = i0; i < i1; ++i) sum += static_cast<double>(mass_at(i));
        double incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        R = __shfl_sync(0xffffffffu, incl, 31);
        double P = __shfl_up_sync(0xffffffffu, incl, 1);
        if (lane == 0) P = 0.0;
        t = static_cast<double>(d.u) * R;
        int found = -1;
        double fb = 0.0;
        for (int i = i0; i < i1; ++i) {
            const double Pn = P + static_cast<double>(mass_at(i));
            if (found < 0 && Pn > t) {
                found = i;
                fb = P;
            }
            P = Pn;
        }
        const unsigned ball = __ballot_sync(0xffffffffu, found >= 0);
        const int src = ball ? (__ffs(ball) - 1) : 0;
        ftile = ball ? __shfl_sync(0xffffffffu, found, src) : -1;
        fbase = __shfl_sync(0xffffffffu, fb, src);
        if (R > 0.0 || attempt == 1) break;
        // empty residual after a rejection: draw from p instead (slow path)
        qrow = nullptr;
        from_smem = false;
        if (lane == 0) atomicOr(a.status, SV_FLAG_ZERO_RESIDUAL);
        for (int tile = 0; tile < a.n_tiles; ++tile) {
            float r[8][4];
            const float m = tile_mass_of<T, kVecPath>(zrow, qrow, a.V, tile, d, a.c, lane, r);
            if (lane == 0) gmass[tile] = m;
        }
        __threadfence_block();
        __syncwarp();
    }
    int vstar = -1;
    float rstar = 0.f;
    if (ftile >= 0) {
        TileRaw<T> raw;
        float r[8][4];
        warp_tile_load<T, kVecPath>(zrow, qrow, a.V, ftile, lane, raw);
        warp_tile_compute<T>(raw, qrow != nullptr, a.V, ftile, a.c, d.M, d.invS, lane, r);
        const TileScan ts = warp_tile_scan<true>(r, ftile, a.V, fbase, t, lane);
        vstar = ts.v;
        rstar = ts.rv;
        // the tile's running sums ended just short of u R (rounding between the
        // tile sum and the running sums): the next token with r > 0
        for (int tile = ftile + 1; tile < a.n_tiles && vstar < 0; ++tile) {
            if (!(mass_at(tile) > 0.f)) continue;
            TileRaw<T> raw2;
            float r2[8][4];
            warp_tile_load<T, kVecPath>(zrow, qrow, a.V, tile, lane, raw2);
            warp_tile_compute<T>(raw2, qrow != nullptr, a.V, tile, a.c, d.M, d.invS, lane, r2);
            int loc = 0x7fffffff;
            float rloc = 0.f;
#pragma unroll
            for (int j = 7; j >= 0; --j)
#pragma unroll
                for (int k = 3; k >= 0; --k) {
                    const int e = (j * 32 + lane) * 4 + k;
                    if (tile * kTileElems + e < a.V && r2[j][k] > 0.f) {
                        loc = e;
                        rloc = r2[j][k];
                    }
                }
            const int best = __reduce_min_sync(0xffffffffu, loc);
            if (best != 0x7fffffff) {
                const unsigned m = __ballot_sync(0xffffffffu, loc == best);
                rstar = __shfl_sync(0xffffffffu, rloc, __ffs(m) - 1);
                vstar = tile * kTileElems + best;
            }
        }
    }
    if (vstar < 0) {
        // rounding left u R above every boundary: the largest token with r > 0
        for (int tile = a.n_tiles - 1; tile >= 0 && vstar < 0; --tile) {
            if (!(mass_at(tile) > 0.f)) continue;
            TileRaw<T> raw;
            float r[8][4];
            warp_tile_load<T, kVecPath>(zrow, qrow, a.V, tile, lane, raw);
            warp_tile_compute<T>(raw, qrow != nullptr, a.V, tile, a.c, d.M, d.invS, lane, r);
            int loc = -1;
            float rloc = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int e = (j * 32 + lane) * 4 + k;
                    if (tile * kTileElems + e < a.V && r[j][k] > 0.f) {
                        loc = e;
                        rloc = r[j][k];
                    }
                }
            const int best = __reduce_max_sync(0xffffffffu, loc);
            if (best >= 0) {
                const unsigned m = __ballot_sync(0xffffffffu, loc == best);
                rstar = __shfl_sync(0xffffffffu, rloc, __ffs(m) - 1);
                vstar = tile * kTileElems + best;
            }
        }
    }
    if (lane == 0) {
        a.out_tokens[d.slot] = vstar;
        if (a.diag) {
            a.diag[a.n_draft + 2 * b] = static_cast<float>(R);
            a.diag[a.n_draft + 2 * b + 1] = static_cast<float>(static_cast<double>(rstar) / R);
        }
    }
}

template <typename T, bool kVecPath>
__global__ void __launch_bounds__(kResThreads, 1) residual_kernel(Args a) {
    extern __shared__ float smass[];  // ceil(n_tiles / cluster size) tile masses of this CTA
    pdl_wait_prior_grid();  // decisions come from pass 1
    if (a.csr_ok && !__ldcg(a.csr_ok)) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int csize = static_cast<int>(cluster_nctarank());
    const int b = blockIdx.x / csize;
    const Decision d = a.dec[b];
    if (!d.valid) return;  // same decision for every CTA of the cluster
    const T *zrow = reinterpret_cast<const T *>(a.logits) + static_cast<size_t>(d.row) * a.V;
    const float *qrow = (d.qrow >= 0) ? a.q + static_cast<size_t>(d.qrow) * a.V : nullptr;
    const int per = (a.n_tiles + csize - 1) / csize;
    const int t0 = static_cast<int>(rank) * per;
    const int t1 = min(t0 + per, a.n_tiles);
    for (int t = t0 + warp; t < t1; t += kResWarps) {
        float r[8][4];
        const float m = tile_mass_of<T, kVecPath>(zrow, qrow, a.V, t, d, a.c, lane, r);
        if (lane == 0) smass[t - t0] = m;
    }
    cluster_sync();
    if (rank == 0 && warp == 0) draw_final<T, kVecPath>(a, b, d, lane, smass, per);
    cluster_sync();  // every CTA's shared memory stays alive until rank 0 has read it
}

// ---------------------------------------------------------------------------
// Decide step over precomputed chunk partials (the fused LM-head path writes
// them from its GEMM epilogue): one warp per request.
// ---------------------------------------------------------------------------
template <bool kSample>
__global__ void __launch_bounds__(kThreads) decide_kernel(Args a) {
    pdl_wait_prior_grid();  // partials and logits come from the previous kernel
    pdl_launch_dependents();
    const int b = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (b < a.B) decide_warp<float, kSample>(a, b, threadIdx.x & 31);
}

// ---------------------------------------------------------------------------
// CSR check for ragged calls (one CTA): offsets must start at 0, increase by
// 1..SV_MAX_K+1 and end at `rows`.  A malformed CSR invalidates the call.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) csr_check_kernel(Args a, int *csr_ok) {
    __shared__ int bad;
    if (threadIdx.x == 0) bad = (a.row_offsets[0] != 0 || a.row_offsets[a.B] != a.rows) ? 1 : 0;
    __syncthreads();
    for (int b = threadIdx.x; b < a.B; b += kThreads) {
        const int k1 = a.row_offsets[b + 1] - a.row_offsets[b];
        if (k1 < 1 || k1 > kMaxRowsPerRequest) bad = 1;
    }
    __syncthreads();
    if (threadIdx.x == 0) *csr_ok = bad ? 0 : 1;
    if (bad) {
        for (int b = threadIdx.x; b < a.B; b += kThreads) a.accept_len[b] = 0;
        for (int r = threadIdx.x; r < a.rows; r += kThreads) a.out_tokens[r] = -1;
        if (threadIdx.x == 0) atomicOr(a.status, SV_FLAG_BAD_OFFSETS);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct WsLayout {
    size_t status, csr_ok, tickets1, dec, partials, tile_mass, total;
};

static inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Per-request counters live in a region of fixed capacity right after the
// status words, whatever the call's shape, and every completed call leaves
// the counters it used at zero.  A workspace therefore serves calls of any
// shape once it has been zero-filled; only a call with more than kTicketCap
// requests (whose counters reach into other regions) clears them first.
constexpr int kTicketCap = 16384;

static WsLayout ws_layout(int B, int rows, int V, bool with_partials = true) {
    WsLayout L;
    const size_t n_chunks = (static_cast<size_t>(V) + chunk_elems<float>() - 1) / chunk_elems<float>();
    const size_t n_tiles = (static_cast<size_t>(V) + kTileElems - 1) / kTileElems;
    size_t o = 0;
    L.status = o; o = align256(o + 16);
    L.csr_ok = o; o = align256(o + 16);
    L.tickets1 = o; o = align256(o + 4ull * static_cast<size_t>(B > kTicketCap ? B : kTicketCap));
    L.dec = o; o = align256(o + sizeof(Decision) * static_cast<size_t>(B));
    L.partials = o; o = align256(o + (with_partials ? sizeof(float2) * static_cast<size_t>(rows) * n_chunks : 0));
    L.tile_mass = o; o = align256(o + sizeof(float) * static_cast<size_t>(B) * n_tiles);
    L.total = o;
    return L;
}

// Byte range [offset, offset + bytes) of the per-request counters inside a
// workspace laid out for (B, rows, V).
void counter_region(int B, int rows, int V, size_t *offset, size_t *bytes) {
    const WsLayout L = ws_layout(B, rows, V);
    *offset = L.tickets1;
    *bytes = L.dec - L.tickets1;
}

static void *g_prof_begin = nullptr;
static void *g_prof_end = nullptr;
static thread_local int g_last_launches = 0;

void prof_begin(cudaStream_t s) {
    if (g_prof_begin) cudaEventRecord(static_cast<cudaEvent_t>(g_prof_begin), s);
}
void prof_end(cudaStream_t s) {
    if (g_prof_end) cudaEventRecord(static_cast<cudaEvent_t>(g_prof_end), s);
}
void set_launches(int n) { g_last_launches = n; }

// Number of SMs of the current device (queried once per device).
int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

template <typename T, bool kSample>
static void launch_tma_pass1(const Args &a, cudaStream_t s) {
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!configured[dev]) {
        cudaFuncSetAttribute(stats_tma_kernel<T, kSample>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(TmaSmem)));
        configured[dev] = true;
    }
    const long long items = static_cast<long long>(a.rows) * a.n_chunks;
    const unsigned grid = static_cast<unsigned>(items < sm_count() ? items : sm_count());
    stats_tma_kernel<T, kSample><<<grid, kTmaThreads, sizeof(TmaSmem), s>>>(a);
}

template <typename T, bool kSample>
static void launch_scalar_pass1(const Args &a, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>(a.rows) * static_cast<unsigned>(a.n_chunks);
    stats_scalar_kernel<T, kSample><<<grid, kThreads, 0, s>>>(a);
}

// Pass 2 runs one cluster of C CTAs per request, C the largest power of two
// <= 8 that keeps B C within one CTA per SM.  It is launched as a
// programmatic dependent of pass 1: its CTAs may be scheduled while pass 1
// drains and wait (griddepcontrol.wait) for pass 1's completion before
// reading the decisions.
template <typename T, bool kVecPath>
static void launch_pass2(const Args &a, cudaStream_t s) {
    int C = 1;
    while (C < kMaxResCluster && static_cast<long long>(a.B) * (2 * C) <= sm_count()) C *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.B) * static_cast<unsigned>(C));
    cfg.blockDim = dim3(kResThreads);
    cfg.dynamicSmemBytes = sizeof(float) * static_cast<size_t>((a.n_tiles + C - 1) / C);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(C);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaLaunchKernelEx(&cfg, residual_kernel<T, kVecPath>, a);
}

template <typename T>
static sv_status run_typed(Args &a, bool sample, bool vec, cudaStream_t s) {
    a.n_chunks = (a.V + chunk_elems<T>() - 1) / chunk_elems<T>();
    int launches = 0;
    if (a.B > kTicketCap &&
        cudaMemsetAsync(a.tickets1, 0, sizeof(uint32_t) * static_cast<size_t>(a.B), s) != cudaSuccess)
        return SV_ERR_CUDA;
    if (a.row_offsets) {
        csr_check_kernel<<<1, kThreads, 0, s>>>(a, const_cast<int *>(a.csr_ok));
        ++launches;
    }
    prof_begin(s);
    if (sample) {
        if (vec) launch_tma_pass1<T, true>(a, s); else launch_scalar_pass1<T, true>(a, s);
    } else {
        if (vec) launch_tma_pass1<T, false>(a, s); else launch_scalar_pass1<T, false>(a, s);
    }
    prof_end(s);
    ++launches;
    if (sample) {
        if (vec) launch_pass2<T, true>(a, s); else launch_pass2<T, false>(a, s);
        ++launches;
    }
    set_launches(launches);
    return (cudaGetLastError() == cudaSuccess) ? SV_OK : SV_ERR_CUDA;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Common host path of the three logits-in entry points.
static sv_status verify_common(const void *logits, sv_dtype dt, const float *q,
                               const int32_t *row_offsets, int B, int K, int rows, int V,
                               float temperature, bool sample, const int32_t *draft,
                               const float *uniforms, int32_t *out_tokens, int32_t *accept_len,
                               float *diag, void *ws, size_t ws_bytes, void *stream) {
    if (B < 0 || V <= 0 || rows < 0 || (dt != SV_F32 && dt != SV_BF16)) return SV_ERR_INVALID;
    if (!row_offsets && (K < 0 || K > SV_MAX_K)) return SV_ERR_INVALID;
    if (B == 0) {
        set_launches(0);
        return SV_OK;
    }
    if (rows < B || static_cast<long long>(rows) * V >= (1ll << 62)) return SV_ERR_INVALID;
    if (!logits || !out_tokens || !accept_len || !ws) return SV_ERR_INVALID;
    if (rows > B && !draft) return SV_ERR_INVALID;
    if (sample && (!(temperature > 0.f) || !std::isfinite(temperature) || !uniforms || (rows > B && !q)))
        return SV_ERR_INVALID;
    const WsLayout L = ws_layout(B, rows, V);
    if (ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return SV_ERR_WORKSPACE;

    char *w = static_cast<char *>(ws);
    Args a{};
    a.logits = logits;
    a.q = q;
    a.row_offsets = row_offsets;
    a.draft = draft;
    a.uniforms = uniforms;
    a.out_tokens = out_tokens;
    a.accept_len = accept_len;
    a.diag = sample ? diag : nullptr;
    a.B = B;
    a.K = K;
    a.V = V;
    a.rows = rows;
    a.n_tiles = (V + kTileElems - 1) / kTileElems;
    a.n_draft = rows - B;
    a.c = sample ? static_cast<float>(1.4426950408889634 / static_cast<double>(temperature)) : 1.f;
    a.status = reinterpret_cast<uint32_t *>(w + L.status);
    a.csr_ok = row_offsets ? reinterpret_cast<const int *>(w + L.csr_ok) : nullptr;
    a.tickets1 = reinterpret_cast<uint32_t *>(w + L.tickets1);
    a.dec = reinterpret_cast<Decision *>(w + L.dec);
    a.partials = reinterpret_cast<float2 *>(w + L.partials);
    a.tile_mass = reinterpret_cast<float *>(w + L.tile_mass);

    const size_t esize = (dt == SV_F32) ? 4 : 2;
    const bool vec = aligned16(logits) && ((static_cast<size_t>(V) * esize) % 16 == 0) &&
                     (!q || (aligned16(q) && V % 4 == 0));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dt == SV_F32) return run_typed<float>(a, sample, vec, s);
    return run_typed<__nv_bfloat16>(a, sample, vec, s);
}


// Workspace of finish_from_partials (the partials live elsewhere).
size_t finish_workspace_size(int B, int rows, int V) { return ws_layout(B, rows, V, false).total; }

template <typename KernelT>
static cudaError_t launch_pdl(KernelT kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, const Args &a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Decide + (sampling) residual draw over fp32 logits rows and per-(row, part)
// partials that a previous kernel on `s` produced.  Launches 1 or 2 kernels.
sv_status finish_from_partials(const float *logits, const float2 *partials, int n_parts, const float *q, int B,
                               int K, int V, float temperature, bool sample, const int32_t *draft,
                               const float *uniforms, int32_t *out_tokens, int32_t *accept_len, float *diag,
                               void *ws, size_t ws_bytes, cudaStream_t s, int *launches) {
    const int rows = B * (K + 1);
    const WsLayout L = ws_layout(B, rows, V, false);
    if (ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return SV_ERR_WORKSPACE;
    char *w = static_cast<char *>(ws);
    Args a{};
    a.logits = logits;
    a.q = q;
    a.row_offsets = nullptr;
    a.draft = draft;
    a.uniforms = uniforms;
    a.out_tokens = out_tokens;
    a.accept_len = accept_len;
    a.diag = sample ? diag : nullptr;
    a.B = B;
    a.K = K;
    a.V = V;
    a.rows = rows;
    a.n_chunks = n_parts;
    a.n_tiles = (V + kTileElems - 1) / kTileElems;
    a.n_draft = rows - B;
    a.c = sample ? static_cast<float>(1.4426950408889634 / static_cast<double>(temperature)) : 1.f;
    a.status = reinterpret_cast<uint32_t *>(w + L.status);
    a.csr_ok = nullptr;
    a.tickets1 = reinterpret_cast<uint32_t *>(w + L.tickets1);
    a.dec = reinterpret_cast<Decision *>(w + L.dec);
    a.partials = const_cast<float2 *>(partials);
    a.tile_mass = reinterpret_cast<float *>(w + L.tile_mass);
    const dim3 grid_d((B + kWarps - 1) / kWarps);
    cudaError_t e = sample ? launch_pdl(decide_kernel<true>, grid_d, dim3(kThreads), 0, s, a)
                           : launch_pdl(decide_kernel<false>, grid_d, dim3(kThreads), 0, s, a);
    if (e != cudaSuccess) return SV_ERR_CUDA;
    *launches = 1;
    if (sample) {
        const bool vec = aligned16(logits) && (V % 4 == 0) && (!q || aligned16(q));
        if (vec) launch_pass2<float, true>(a, s); else launch_pass2<float, false>(a, s);
        *launches = 2;
    }
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace sv

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
using namespace sv;

extern "C" size_t spec_verify_workspace_size(int B, int rows, int V) {
    if (B <= 0 || rows < B || V <= 0) return 256;
    return ws_layout(B, rows, V).total;
}

extern "C" sv_status spec_verify_greedy(const void *logits, sv_dtype dt, int B, int K, int V,
                                        const int32_t *draft, int32_t *out_tokens,
                                        int32_t *accept_len, void *ws, size_t ws_bytes,
                                        void *stream) {
    if (K < 0 || K > SV_MAX_K || B < 0) return SV_ERR_INVALID;
    return verify_common(logits, dt, nullptr, nullptr, B, K, B * (K + 1), V, 0.f, false, draft,
                         nullptr, out_tokens, accept_len, nullptr, ws, ws_bytes, stream);
}

extern "C" sv_status spec_verify_sample(const void *logits, sv_dtype dt, const float *q, int B,
                                        int K, int V, float temperature, const int32_t *draft,
                                        const float *uniforms, int32_t *out_tokens,
                                        int32_t *accept_len, float *diag, void *ws,
                                        size_t ws_bytes, void *stream) {
    if (K < 0 || K > SV_MAX_K || B < 0) return SV_ERR_INVALID;
    return verify_common(logits, dt, q, nullptr, B, K, B * (K + 1), V, temperature, true, draft,
                         uniforms, out_tokens, accept_len, diag, ws, ws_bytes, stream);
}

extern "C" sv_status spec_verify_ragged(const void *logits, sv_dtype dt, const float *q,
                                        const int32_t *row_offsets, int B, int rows, int V,
                                        float temperature, const int32_t *draft,
                                        const float *uniforms, int32_t *out_tokens,
                                        int32_t *accept_len, float *diag, void *ws,
                                        size_t ws_bytes, void *stream) {
    if (!row_offsets || B < 0 || !(temperature >= 0.f)) return SV_ERR_INVALID;
    const bool sample = temperature > 0.f;
    return verify_common(logits, dt, q, row_offsets, B, -1, rows, V, temperature, sample, draft,
                         uniforms, out_tokens, accept_len, diag, ws, ws_bytes, stream);
}

extern "C" sv_status spec_verify_last_device_status(void *ws, void *stream, uint32_t *flags) {
    if (!ws) return SV_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SV_ERR_CUDA;
    if (cudaMemsetAsync(ws, 0, sizeof(word), s) != cudaSuccess) return SV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SV_ERR_CUDA;
    if (flags) *flags = word;
    if (word & SV_FLAG_TIMEOUT) return SV_ERR_TIMEOUT;
    if (word & (SV_FLAG_BAD_TOKEN | SV_FLAG_BAD_OFFSETS)) return SV_ERR_DEVICE_INPUT;
    return SV_OK;
}

extern "C" const char *spec_status_string(sv_status s) {
    switch (s) {
        case SV_OK: return "ok";
        case SV_ERR_INVALID: return "invalid argument";
        case SV_ERR_CUDA: return "CUDA error";
        case SV_ERR_DEVICE_INPUT: return "device-detected input error";
        case SV_ERR_TIMEOUT: return "device wait timed out";
        case SV_ERR_WORKSPACE: return "workspace too small or misaligned";
    }
    return "unknown status";
}

extern "C" sv_status spec_profile_set_events(void *begin, void *end) {
    if ((begin == nullptr) != (end == nullptr)) return SV_ERR_INVALID;
    g_prof_begin = begin;
    g_prof_end = end;
    return SV_OK;
}

extern "C" int spec_last_launch_count(void) { return g_last_launches; }
