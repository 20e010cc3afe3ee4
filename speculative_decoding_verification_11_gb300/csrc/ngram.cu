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
// most min(n_max, e + 1)).  The winner maximises (m, e) with m >= n_min: the
// longest suffix first, then its latest occurrence -- the order in which the
// method tries n = n_max .. n_min and scans back from the end.  Each CTA's
// best (m, e) goes to the first CTA of the cluster through distributed shared
// memory; that CTA writes the proposal.
//
// Data movement: a CTA's range passes through a ring of kStages shared-memory
// stages of kSeg candidate ends each (with the kHalo tokens before them), all
// stages in flight from the start.  A stage's 16-byte-aligned interior comes
// with one bulk copy completing on the stage's mbarrier; the at most three
// tokens on either side of it come with plain loads.  A stage holds token x
// at index x - (t0 - kHalo) + off, where off puts every token at the same
// position modulo 16 bytes in shared memory as in global memory, so the bulk
// copy's two ends are aligned whatever the context's start.  A warp tests 256
// candidate ends per pass against the context's last token (two 16-byte
// shared-memory loads per lane, one vote); only a pass holding a match ballots
// its matches and extends them backwards, one per lane.
#include <cstdint>

#include "../../include/specverify.h"
#include "sv_args.cuh"
#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {
namespace ng {

constexpr int kSplit = 4;      // CTAs per request (one cluster)
constexpr int kThreads = 256;
constexpr int kMaxN = 32;
constexpr int kHalo = kMaxN;   // tokens staged before a stage's first candidate end (an extension reads 31)
constexpr int kSeg = 2048;     // candidate ends per stage
constexpr int kStages = 3;
// a stage: up to 3 tokens of alignment offset, the halo, kSeg ends, and the last 16-byte group the
// compares read past the final end
constexpr int kStageElems = kHalo + kSeg + 8;
static_assert(kStageElems % 4 == 0, "stages stay 16-byte aligned");
static_assert(kStages + 2 <= kThreads / 32, "one warp per stage for its ragged ends, one for the suffix");
constexpr unsigned long long kFailKey = ~0ull;  // a CTA whose copy never landed (no real key has m = 2^32 - 1)

struct Stage {
    int t0;        // first candidate end
    int n;         // candidate ends in the stage
    int off;       // shared-memory position of token t0 - kHalo
};

__device__ __forceinline__ Stage stage_of(int c0, int c1, int g, int phase) {
    Stage st;
    st.t0 = c0 + g * kSeg;
    st.n = (c1 - st.t0) < kSeg ? (c1 - st.t0) : kSeg;
    st.off = (phase + st.t0 - kHalo) & 3;
    return st;
}

// Stage st's tokens [max(0, t0 - kHalo), t0 + n) split into a 16-byte-aligned interior [a, b), copied
// in bulk, and at most six tokens on its two sides, loaded plainly.
struct Span {
    int x_lo, a, b, x_hi, shift;  // shared index of token x = x + shift
};

__device__ __forceinline__ Span span_of(const Stage &st, int phase) {
    Span p;
    const int base = st.t0 - kHalo;
    p.x_lo = base > 0 ? base : 0;
    p.x_hi = st.t0 + st.n;
    p.a = p.x_lo + ((4 - ((phase + p.x_lo) & 3)) & 3);  // first aligned token
    p.b = p.x_hi - ((phase + p.x_hi) & 3);              // end of the aligned interior
    if (p.a >= p.b) p.a = p.b = p.x_hi;                 // no interior: every token by plain loads
    p.shift = st.off - base;
    return p;
}

// One thread: the interior's bulk copy, completing the stage's mbarrier phase (an arrival alone when
// there is no interior).
__device__ __forceinline__ void issue_bulk(int32_t *buf, uint64_t *bar, const int32_t *ctx, const Span &p) {
    if (p.a < p.b) {
        const uint64_t policy = l2_evict_first_policy();  // each context token is read once
        const uint32_t bytes = static_cast<uint32_t>(p.b - p.a) * 4u;
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s_hint(buf + (p.a + p.shift), ctx + p.a, bytes, bar, policy);
    } else {
        mbar_arrive(bar);
    }
}

// One warp: the tokens on both sides of the interior (lanes 0-7 before it, 8-15 after it).
__device__ __forceinline__ void load_ends(int32_t *buf, const int32_t *ctx, const Span &p, int lane) {
    const int head = p.a - p.x_lo, tail = p.x_hi - p.b;
    if (lane < head) buf[p.x_lo + lane + p.shift] = ctx[p.x_lo + lane];
    else if (lane >= 8 && lane - 8 < tail) buf[p.b + (lane - 8) + p.shift] = ctx[p.b + (lane - 8)];
}

// Position of the n-th (from 0) set bit of m; n < popc(m).
__device__ __forceinline__ int nth_set_bit(unsigned m, int n) {
    int pos = 0;
#pragma unroll
    for (int w = 16; w > 0; w >>= 1) {
        const unsigned lo = m & ((1u << w) - 1u);
        const int c = __popc(lo);
        if (n >= c) {
            n -= c;
            m >>= w;
            pos += w;
        } else {
            m = lo;
        }
    }
    return pos;
}

// The candidate ends of the 32 groups from gw that equal the last token, extended backwards one per lane
// (slot-major, then lane order), their (m, e) keys folded into best.  Called by a whole warp.
__device__ __forceinline__ void extend_matches(const int32_t *buf, int gw, int g_end, const Stage &st,
                                               const int32_t *suf, int n_min, int n_max, int lane,
                                               unsigned long long &best) {
    const int gi = gw + lane;
    const int32_t last = suf[0];
    const int4 w = gi < g_end ? reinterpret_cast<const int4 *>(buf)[gi] : make_int4(~last, ~last, ~last, ~last);
    const int i0 = 4 * gi - kHalo - st.off;  // candidate index of slot 0
    const unsigned m0 = __ballot_sync(0xffffffffu, i0 >= 0 && i0 < st.n && w.x == last);
    const unsigned m1 = __ballot_sync(0xffffffffu, i0 + 1 >= 0 && i0 + 1 < st.n && w.y == last);
    const unsigned m2 = __ballot_sync(0xffffffffu, i0 + 2 >= 0 && i0 + 2 < st.n && w.z == last);
    const unsigned m3 = __ballot_sync(0xffffffffu, i0 + 3 >= 0 && i0 + 3 < st.n && w.w == last);
    const int p1 = __popc(m0), p2 = p1 + __popc(m1), p3 = p2 + __popc(m2), cnt = p3 + __popc(m3);
    for (int r = lane; r < cnt; r += 32) {
        // the r-th match in (slot, lane) order
        const int q = (r >= p1) + (r >= p2) + (r >= p3);
        const unsigned mq = q == 0 ? m0 : q == 1 ? m1 : q == 2 ? m2 : m3;
        const int rq = r - (q == 0 ? 0 : q == 1 ? p1 : q == 2 ? p2 : p3);
        const int pos = 4 * (gw + nth_set_bit(mq, rq)) + q;
        const int e = st.t0 + (pos - kHalo - st.off);
        const int lim = e + 1 < n_max ? e + 1 : n_max;
        int m = 1;
        while (m < lim && buf[pos - m] == suf[m]) ++m;
        if (m >= n_min) {
            const unsigned long long key = (static_cast<unsigned long long>(m) << 32) | static_cast<unsigned long long>(e);
            best = key > best ? key : best;
        }
    }
}

// One stage's compares by one warp: 64 groups (256 candidate ends) per pass, two 16-byte loads per lane
// and one vote; only a pass holding a value equal to the last token (rare) goes on to the per-slot
// ballots.
__device__ __forceinline__ unsigned long long compare_stage(const int32_t *buf, Stage st, const int32_t *suf,
                                                         int n_min, int n_max, int g_end, int warp, int lane,
                                                         unsigned long long best) {
    const int32_t last = suf[0];
    for (int gw = (kHalo >> 2) + warp * 64; gw < g_end; gw += 64 * (kThreads / 32)) {
        const int ga = gw + lane, gb = ga + 32;
        const int4 no = make_int4(~last, ~last, ~last, ~last);
        const int4 wa = ga < g_end ? reinterpret_cast<const int4 *>(buf)[ga] : no;
        const int4 wb = gb < g_end ? reinterpret_cast<const int4 *>(buf)[gb] : no;
        const bool hit = (wa.x == last) | (wa.y == last) | (wa.z == last) | (wa.w == last) | (wb.x == last) |
                         (wb.y == last) | (wb.z == last) | (wb.w == last);
        if (__any_sync(0xffffffffu, hit)) {
            extend_matches(buf, gw, g_end, st, suf, n_min, n_max, lane, best);
            extend_matches(buf, gw + 32, g_end, st, suf, n_min, n_max, lane, best);
        }
    }
    return best;
}

__global__ void __launch_bounds__(kThreads, 8) ngram_kernel(const int32_t *tokens, const int32_t *ctx_offsets, int K,
                                                         int n_min, int n_max, int32_t *draft_out, int32_t *k_out) {
    __shared__ __align__(16) int32_t ring[kStages][kStageElems];
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ int32_t suf[kMaxN];
    __shared__ unsigned long long s_best[kThreads / 32];
    __shared__ unsigned long long s_keys[kSplit];  // the first CTA: every CTA's best key
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    cluster_arrive_relaxed();  // matched by the wait before the first remote store
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait_prior_grid();
    pdl_launch_dependents();
    const int b = blockIdx.x, part = static_cast<int>(cluster_ctarank());
    const int s0 = ctx_offsets[b];
    const int e0 = ctx_offsets[b + 1];
    // a negative start or decreasing offsets: an empty context, nothing proposed (and nothing read)
    const int L = (s0 >= 0 && e0 > s0) ? e0 - s0 : 0;
    const int32_t *ctx = tokens + s0;
    // 4-byte units of ctx[0]'s address modulo 4 (the pointer is 4-byte aligned: checked on the host)
    const int phase = static_cast<int>(((reinterpret_cast<uintptr_t>(tokens) >> 2) + static_cast<uintptr_t>(s0)) & 3);
    const int n_cand = L >= 2 ? L - 1 : 0;  // candidate ends 0 .. L - 2
    const int chunk = n_cand / kSplit + (n_cand % kSplit != 0);
    const int c0 = part * chunk < n_cand ? part * chunk : n_cand;
    const int c1 = c0 + chunk < n_cand ? c0 + chunk : n_cand;
    const int n_seg = (c1 - c0) / kSeg + ((c1 - c0) % kSeg != 0);
    // fill the ring: thread 0 issues the bulk copies first; warps 1-3 load the stages' ragged ends and
    // warp 4 the context's suffix, in parallel
    if (tid == 0)
        for (int g = 0; g < n_seg && g < kStages; ++g)
            issue_bulk(ring[g], &full[g], ctx, span_of(stage_of(c0, c1, g, phase), phase));
    if (warp >= 1 && warp <= kStages && warp - 1 < n_seg)
        load_ends(ring[warp - 1], ctx, span_of(stage_of(c0, c1, warp - 1, phase), phase), lane);
    if (warp == kStages + 1 && lane < n_max && lane < L) suf[lane] = ctx[L - 1 - lane];
    // key = m << 32 | e, 0 = no candidate (m >= n_min >= 1 makes every real key nonzero)
    unsigned long long best = 0ull;
    int g = 0;
    bool ok = true;
    for (; g < n_seg; ++g) {
        const int s = g % kStages;
        // the stage's bulk copy (issued by this CTA) and, after the barrier, its plain loads; one thread
        // polls the mbarrier, the others wait at the barrier without taking issue slots from the SM's
        // other CTAs
        const bool landed = tid != 0 || mbar_wait_bounded(&full[s], (g / kStages) & 1, kDrainBudget);
        if (!__syncthreads_and(landed)) {
            ok = false;
            break;
        }
        const Stage st = stage_of(c0, c1, g, phase);
        const int32_t *buf = ring[s];
        const int g_end = (kHalo + st.off + st.n + 3) >> 2;  // 16-byte groups holding the stage's ends
        best = compare_stage(buf, st, suf, n_min, n_max, g_end, warp, lane, best);
        __syncthreads();  // every compare of stage s is done: it may be refilled
        if (g + kStages < n_seg) {
            const Span p = span_of(stage_of(c0, c1, g + kStages, phase), phase);
            if (tid == 0) issue_bulk(ring[s], &full[s], ctx, p);
            if (warp == 1) load_ends(ring[s], ctx, p, lane);
        }
    }
    if (!ok) {
        // a copy did not land within the drain limit: wait once more (bounded) for it and for this
        // CTA's later copies in flight, then report the request as failed to the first CTA (it
        // proposes nothing)
        const int issued = n_seg < g + kStages ? n_seg : g + kStages;
        if (tid == 0)
            for (int h = g; h < issued; ++h) mbar_wait_bounded(&full[h % kStages], (h / kStages) & 1, kDrainBudget);
        __syncthreads();
        best = kFailKey;
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
    int k = 0, e_w = -1;
    if (best != 0ull && best != kFailKey) {
        e_w = static_cast<int>(best & 0xffffffffull);
        k = L - 1 - e_w;
        if (k > K) k = K;
    }
    for (int j = tid; j < K; j += kThreads)
        draft_out[static_cast<size_t>(b) * K + j] = (j < k) ? ctx[e_w + 1 + j] : -1;
    if (tid == 0) k_out[b] = k;
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
    if (reinterpret_cast<uintptr_t>(tokens) & 3u) return SV_ERR_INVALID;  // int32 tokens, 4-byte aligned
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
