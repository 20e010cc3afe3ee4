// Verification kernels and the C ABI of libspecverify.so (sm_103a).
//
// Rows 16-byte aligned: fused_kernel runs the whole step in one persistent
//   kernel (see the section "Fused verification" below).
// Any alignment: two passes.
// Pass 1  stats_scalar_kernel: one CTA per (row, 32 KB chunk) reduces the chunk
//         to (M, s) = (max z c, sum 2^(z c - M)) with c = log2(e)/T (sampling)
//         or to (max z, first argmax) (greedy); the arrival that completes a
//         request's count (release atomic) runs the decide step in one warp:
//         accept tests u q(x) <= p(x), ballot for the first rejection, emitted
//         drafts, AL, and the record of the row the final token comes from.
// Pass 2  residual_kernel (sampling only) one cluster of 1-8 CTAs per request over
//         the selected row, one warp per 1024-token tile: r = max(0, p - q)
//         at a rejection or r = p for the bonus, tile masses in shared
//         memory; rank 0 takes the prefix over tiles in fp64 through
//         distributed shared memory, finds the tile holding u R, and resolves
//         the token inside it with running sums in token order.
//
// The operation is the one stated on "Speculative Decoding in Large Language
// Models", section 2 "Modified Rejection Sampling" (accept test, residual
// p'(x)), with the stop at the first mismatch and the extra target token of
// "Co-Designing AI Models Using Speculative Decoding", "What is speculative
// decoding?".  See include/specverify.h for the full contract.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>

#include "../../include/specverify.h"
#include "sv_device.cuh"
#include "sv_draw.cuh"
#include "sv_args.cuh"
#include "sv_host.h"

namespace sv {


// A decision written by another CTA during the same kernel: read it from L2
// (an L1 line may still hold a neighbour's older bytes).
__device__ __forceinline__ Decision load_decision(const Decision *p) {
    static_assert(sizeof(Decision) == 32, "decision is two 16-byte words");
    const int4 w0 = __ldcg(reinterpret_cast<const int4 *>(p));
    const int4 w1 = __ldcg(reinterpret_cast<const int4 *>(p) + 1);
    Decision d;
    d.row = w0.x;
    d.qrow = w0.y;
    d.slot = w0.z;
    d.valid = w0.w;
    d.M = __int_as_float(w1.x);
    d.invS = __int_as_float(w1.y);
    d.u = __int_as_float(w1.z);
    d.pad = w1.w;
    return d;
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

// Fold one chunk slice into the lane's running partial.  Vector j (VEC
// consecutive tokens) is valid iff e0[j] < n (n is a multiple of VEC on this
// path; kFull: the whole chunk, no test).  Max and sum run as trees over
// independent values; the exponent arguments and sums use packed fp32x2.
template <bool kSample, bool kFull, int NV, int VEC>
__device__ __forceinline__ void lane_accumulate(const float (&vals)[NV][VEC], const int (&e0)[NV], int n, int c0,
                                                float c, float &ra, int &rb) {
    if (kSample) {
        float vm[NV];
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            float m = fmaxf(vals[j][0], vals[j][1]);
#pragma unroll
            for (int k = 2; k < VEC; ++k) m = fmaxf(m, vals[j][k]);
            vm[j] = (kFull || e0[j] < n) ? m : -INFINITY;
        }
#pragma unroll
        for (int w = 1; w < NV; w <<= 1)
#pragma unroll
            for (int j = 0; j + w < NV; j += 2 * w) vm[j] = fmaxf(vm[j], vm[j + w]);
        const float bm = vm[0];
        if (bm != -INFINITY) {
            const float Mn = fmaxf(ra, bm * c);
            const float2 cc = make_float2(c, c), nm = make_float2(-Mn, -Mn);
            float2 acc[NV];
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                float2 sj = make_float2(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < VEC; k += 2) {
                    const float2 y = __ffma2_rn(make_float2(vals[j][k], vals[j][k + 1]), cc, nm);
                    sj = __fadd2_rn(sj, make_float2(ex2(y.x), ex2(y.y)));
                }
                acc[j] = (kFull || e0[j] < n) ? sj : make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int w = 1; w < NV; w <<= 1)
#pragma unroll
                for (int j = 0; j + w < NV; j += 2 * w) acc[j] = __fadd2_rn(acc[j], acc[j + w]);
            const float s_old = __int_as_float(rb) * ex2(ra - Mn);  // ra = -inf: 0
            ra = Mn;
            rb = __float_as_int(s_old + (acc[0].x + acc[0].y));
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
            const bool ok = kFull || e0[j] < n;
            vv[j] = ok ? m : -INFINITY;
            vi[j] = ok ? c0 + e0[j] + mi : 0x7fffffff;
        }
#pragma unroll
        for (int w = 1; w < NV; w <<= 1)
#pragma unroll
            for (int j = 0; j + w < NV; j += 2 * w) am_merge(vv[j], vi[j], vv[j + w], vi[j + w]);
        if (vi[0] != 0x7fffffff) am_merge(ra, rb, vv[0], vi[0]);
    }
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
    const Decision d = load_decision(a.dec + b);
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
// Fused verification: one persistent kernel runs the whole step (rows 16-byte
// aligned).  One CTA per SM, three roles:
//   producer (one thread)  streams 32 KB stages into a 6-stage shared-memory
//                          ring with bulk copies: first stats blocks (4
//                          chunks of one row) from a grid-wide counter in row
//                          order, then residual blocks (4096 tokens of a
//                          request's selected row and its q row) from a second
//                          counter in request-major order, each once its
//                          request's decision is published.  Stats go first
//                          because every decision waits on them, and a
//                          residual stage queued ahead of them in a ring would
//                          delay the decisions still to come;
//   16 consumer warps      reduce each stats block to one partial per warp
//                          and each residual stage to one mass per 256-token
//                          segment, and store them to the workspace;
//   worker warp            owns requests b = CTA, CTA + G, ...: gathers the
//                          drafts' z(x), q(x) and uniforms, waits for the
//                          request's partials, runs the accept tests and the
//                          first-reject scan, publishes the decision, waits
//                          for the segment masses and draws the final token.
// Every record that crosses CTAs is one 32- or 64-bit word that reads zero
// until it is written (the stored encodings are never zero).  Readers poll
// with relaxed loads and zero what they consumed, so no fence lies on a
// request's path, and a completed call leaves the records zeroed for the
// next one.  The arithmetic of the final draw's prefix sums is double-single
// fp32, not fp64 (see DS below).
// ---------------------------------------------------------------------------
namespace fz {

constexpr int kStages = 6;
constexpr int kChunkBytes = 32768;
constexpr int kCons = 16;                                   // consumer warps
constexpr int kVecs = kChunkBytes / 16 / (kCons * 32);      // 16-byte vectors per lane per stats chunk
constexpr int kProducer = kCons, kWorker = kCons + 1;
constexpr int kThreads = (kCons + 2) * 32;
constexpr int kBlockChunks = 4;                             // chunks per stats block
constexpr int kResElems = kResStageElems;                   // tokens per residual stage
constexpr int kResQOffset = 16384;                          // byte offset of the q part in a stage
constexpr unsigned kPollNs = 64;

enum { kStats = 0, kRes = 1, kEnd = 2 };

struct Tag {
    int kind;
    int row;    // stats: logits row        residual: request
    int chunk;  // stats: chunk index       residual: stage index within the row
    int n;      // tokens in the stage
    int has_q;  // residual: 1 if the q part is present
    int last;   // stats: 1 on the block's last chunk
    float M, invS;  // residual: the decision's normaliser
};

constexpr int kWorkerMassCap = 512;  // segment masses a draw keeps in registers and shared memory
struct Smem {
    alignas(128) unsigned char ring[kStages][kChunkBytes];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    Tag tag[kStages];
    int abort;
    float wmass[kWorkerMassCap];  // the worker's copy of one request's segment masses (draw)
};

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t *p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Residual claims, in request order: a request before tail_b0 takes n_rb
// claims of kResBlockStages stages; the last requests (decided last, since
// stats stream in row order) take one claim per stage, so that their
// residual spreads over many CTAs at the end of the step.
struct Claim {
    int b, st0, nst;
};
__device__ __forceinline__ uint32_t residual_claims(const Args &a) {
    return static_cast<uint32_t>(a.tail_b0) * a.n_rb + static_cast<uint32_t>(a.B - a.tail_b0) * a.n_st;
}
__device__ __forceinline__ Claim decode_claim(uint32_t p, const Args &a) {
    const uint32_t big = static_cast<uint32_t>(a.tail_b0) * a.n_rb;
    if (p < big) {
        const int b = static_cast<int>(p / static_cast<uint32_t>(a.n_rb));
        return Claim{b, static_cast<int>(p - static_cast<uint32_t>(b) * a.n_rb) * kResBlockStages, kResBlockStages};
    }
    const uint32_t q = p - big;
    const int i = static_cast<int>(q / static_cast<uint32_t>(a.n_st));
    return Claim{a.tail_b0 + i, static_cast<int>(q - static_cast<uint32_t>(i) * a.n_st), 1};
}

// A partial (a, b) as one word: low half a; high half b with its top bit
// flipped.  b is a sum of exponentials (>= +0) or a token index (>= 0), so
// the high half is never zero.
template <bool kSample>
__device__ __forceinline__ uint64_t enc_partial(float a, int b) {
    if (kSample) b = __float_as_int(__fadd_rn(__int_as_float(b), 0.f));  // -0 -> +0
    return (static_cast<uint64_t>(static_cast<uint32_t>(b) ^ 0x80000000u) << 32) | __float_as_uint(a);
}
__device__ __forceinline__ bool partial_written(uint64_t w) { return (w >> 32) != 0; }
__device__ __forceinline__ float2 dec_partial(uint64_t w) {
    return make_float2(__uint_as_float(static_cast<uint32_t>(w)),
                       __int_as_float(static_cast<int>(static_cast<uint32_t>(w >> 32) ^ 0x80000000u)));
}

// A residual mass (>= 0, or NaN on bad inputs) with its top bit flipped: never zero.
__device__ __forceinline__ uint32_t enc_mass(float m) { return __float_as_uint(__fadd_rn(m, 0.f)) ^ 0x80000000u; }
__device__ __forceinline__ float dec_mass(uint32_t w) { return __uint_as_float(w ^ 0x80000000u); }

// The decision of request b as two words: {M, 1/S} and {row, qrow + 2};
// row < 0 marks a request without a draw (an invalid draft).
__device__ __forceinline__ void publish_decision(uint64_t *rec, float M, float invS, int row, int qrow) {
    st_relaxed_u64(rec, (static_cast<uint64_t>(__float_as_uint(invS) ^ 0x80000000u) << 32) | __float_as_uint(M));
    st_relaxed_u64(rec + 1, (static_cast<uint64_t>(static_cast<uint32_t>(qrow + 2)) << 32) |
                                static_cast<uint32_t>(row));
}

// r(v) of 8 tokens of a residual chunk held by one lane: token
// base + (j * 32 + lane) * 4 + k of the chunk, j < 2, k < 4.
template <typename T>
__device__ __forceinline__ float res_lane_sum(const unsigned char *stage, int warp, int lane, int n, bool has_q,
                                              float c, float M, float invS) {
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int v = warp * 64 + j * 32 + lane;  // index of this lane's 4-token group
        const int e0 = v * 4;
        if (e0 >= n) continue;
        float z[4], qv[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (sizeof(T) == 4) {
            const float4 w = reinterpret_cast<const float4 *>(stage)[v];
            z[0] = w.x; z[1] = w.y; z[2] = w.z; z[3] = w.w;
        } else {
            const uint2 w = reinterpret_cast<const uint2 *>(stage)[v];
            z[0] = __uint_as_float(w.x << 16);
            z[1] = __uint_as_float(w.x & 0xffff0000u);
            z[2] = __uint_as_float(w.y << 16);
            z[3] = __uint_as_float(w.y & 0xffff0000u);
        }
        if (has_q) {
            const float4 w = reinterpret_cast<const float4 *>(stage + kResQOffset)[v];
            qv[0] = w.x; qv[1] = w.y; qv[2] = w.z; qv[3] = w.w;
        }
        float r[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float p = __fmul_rn(ex2(__fmaf_rn(z[k], c, -M)), invS);
            r[k] = has_q ? fmaxf(__fsub_rn(p, qv[k]), 0.f) : p;
        }
        acc += (r[0] + r[1]) + (r[2] + r[3]);  // n is a multiple of 4 on this path
    }
    return acc;
}


struct Sel {
    int valid;   // 0: an invalid draft id (nothing to draw)
    int ks;      // accepted drafts: row r0 + ks carries the final token
    int row, qrow;
    float M, S;  // normaliser of row ks (sampling)
};

// Lane 0's verdict, the same in every lane: stop waiting (abort or time budget spent).
__device__ __forceinline__ bool give_up(const Args &a, volatile int *abort_flag, long long t_start, int lane) {
    int stop = 0;
    if (lane == 0) {
        stop = *abort_flag;
        if (!stop && clock64() - t_start > a.wait_budget) {
            *abort_flag = 1;
            atomicOr(a.status, SV_FLAG_TIMEOUT);
            stop = 1;
        }
    }
    return __shfl_sync(0xffffffffu, stop, 0) != 0;
}

// Decide step of request b by its owning worker warp.  Lane j holds row
// jb + j: its draft's gathers go out first, then the warp waits for the rows'
// partials (8 rows at a time, lanes over a row's partials, so every load of a
// poll is in flight at once), merges them in index order and zeroes them.
// Every row is consumed even after a rejection, so the records are left
// zeroed.  Returns false when it gave up waiting.
template <typename T, bool kSample>
__device__ bool fused_decide(const Args &a, int b, int lane, volatile int *abort_flag, long long t_start, Sel &sel) {
    int r0, nr;
    request_rows(a, b, r0, nr);
    const int Kb = nr - 1;
    const int d0 = r0 - b;
    const int E = a.n_pe;
    bool bad = false;
    for (int j = lane; j < Kb; j += 32) {
        const int x = __ldg(a.draft + d0 + j);
        bad |= (x < 0 || x >= a.V);
    }
    bad = __any_sync(0xffffffffu, bad);
    int ks = -1;
    float Msel = 0.f, Ssel = 1.f;
    int argsel = 0;
    for (int jb = 0; jb < nr; jb += 32) {
        const int j = jb + lane;
        int x = 0;
        float z = 0.f, qv = 0.f, u = 0.f;
        if (j < Kb && !bad) {
            x = __ldg(a.draft + d0 + j);
            if (kSample) {
                z = logit_at<T>(a, static_cast<size_t>(r0 + j) * a.V + x);
                qv = __ldg(a.q + static_cast<size_t>(d0 + j) * a.V + x);
                u = __ldg(a.uniforms + r0 + j);
            }
        }
        float M = -INFINITY, S = 0.f, bv = -INFINITY;
        int bi = 0x7fffffff;
        const int rows_here = min(32, nr - jb);
        for (int rg = 0; rg < rows_here; rg += 8) {
            uint64_t *base = a.fpart + static_cast<size_t>(r0 + jb + rg) * E;
            float ma[8];
            int mb[8];
            for (;;) {
#pragma unroll
                for (int i = 0; i < 8; ++i) partial_identity<kSample>(ma[i], mb[i]);
                bool all = true;
                for (int e = lane; e < E; e += 32) {
                    uint64_t w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        w[i] = (rg + i < rows_here) ? ld_relaxed_u64(base + static_cast<size_t>(i) * E + e) : 0ull;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (rg + i < rows_here) {
                            all &= partial_written(w[i]);
                            merge_pair<kSample>(ma[i], mb[i], dec_partial(w[i]));
                        }
                }
                if (__all_sync(0xffffffffu, all)) break;
                if (give_up(a, abort_flag, t_start, lane)) return false;
                __nanosleep(kPollNs);
            }
            for (int e = lane; e < E; e += 32)
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (rg + i < rows_here) st_relaxed_u64(base + static_cast<size_t>(i) * E + e, 0ull);
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
        if (j < Kb && !bad) {
            if (kSample) {
                const float p = exp2f(fmaf(z, a.c, -M)) / S;
                rej = !(u * qv <= p);
                if (a.diag) a.diag[d0 + j] = p;
            } else {
                rej = (x != bi);
            }
        }
        const unsigned m = __ballot_sync(0xffffffffu, rej);
        if (ks < 0 && !bad && (m || jb + 32 >= nr)) {
            const int src = m ? (__ffs(m) - 1) : (Kb - jb);
            ks = jb + src;
            Msel = __shfl_sync(0xffffffffu, M, src);
            Ssel = __shfl_sync(0xffffffffu, S, src);
            argsel = __shfl_sync(0xffffffffu, bi, src);
        }
        (void)bv;
    }
    if (bad) {
        for (int j = lane; j < nr; j += 32) a.out_tokens[r0 + j] = -1;
        if (lane == 0) {
            a.accept_len[b] = 0;
            atomicOr(a.status, SV_FLAG_BAD_TOKEN);
        }
        sel.valid = 0;
        sel.ks = -1;
        sel.row = -1;
        sel.qrow = -1;
        return true;
    }
    for (int j = lane; j < nr; j += 32) {
        int v = -1;
        if (j < ks) v = __ldg(a.draft + d0 + j);
        else if (j == ks && !kSample) v = argsel;
        a.out_tokens[r0 + j] = v;
    }
    if (lane == 0) a.accept_len[b] = ks + 1;
    sel.valid = 1;
    sel.ks = ks;
    sel.row = r0 + ks;
    sel.qrow = (ks < Kb) ? d0 + ks : -1;
    sel.M = Msel;
    sel.S = Ssel;
    return true;
}


// Final draw of request b by its owning worker warp, once every segment mass
// of the selected row is in: an fp64 prefix over the segments, then running
// sums in token order inside the segment that holds u R.  Rounding
// fallbacks: sums that end short of u R take the next token with r > 0; u R
// at or above every boundary takes the last token with r > 0.  An empty
// residual after a rejection draws from p instead.  Returns false when it
// gave up waiting.
template <typename T>
__device__ bool fused_draw(const Args &a, int b, const Sel &sel, float invS, int lane, volatile int *abort_flag,
                           long long t_start, float *wmass) {
    int r0, nr;
    request_rows(a, b, r0, nr);
    const T *zrow = reinterpret_cast<const T *>(a.logits) + static_cast<size_t>(sel.row) * a.V;
    const float *qrow = (sel.qrow >= 0) ? a.q + static_cast<size_t>(sel.qrow) * a.V : nullptr;
    const float M = sel.M;
    const float u = __ldg(a.uniforms + r0 + nr - 1);
    uint32_t *mw = a.fmass + static_cast<size_t>(b) * a.n_seg;
    const int ns = a.n_seg;
    const int G = (ns + 31) / 32;
    const int i0 = min(lane * G, ns), i1 = min(i0 + G, ns);
    // this lane's masses stay in registers (and in wmass) when they fit (V up to 131072)
    constexpr int kRegSeg = kWorkerMassCap / 32;
    const bool in_regs = G <= kRegSeg;
    float mv[kRegSeg];
    for (;;) {
        bool all = true;
        if (in_regs) {
#pragma unroll
            for (int i = 0; i < kRegSeg; ++i) {
                const uint32_t w = (i0 + i < i1) ? ld_relaxed_u32(mw + i0 + i) : enc_mass(0.f);
                all &= (w != 0u);
                mv[i] = dec_mass(w);
            }
        } else {
            for (int i = i0; i < i1; ++i) all &= (ld_relaxed_u32(mw + i) != 0u);
        }
        if (__all_sync(0xffffffffu, all)) break;
        if (give_up(a, abort_flag, t_start, lane)) return false;
        __nanosleep(kPollNs);
    }
    DS sum{0.f, 0.f};
    if (in_regs) {
        // the lane's masses summed pairwise: four levels of independent double-single adds rather
        // than a chain of sixteen (the draw waits on this sum)
        static_assert(kRegSeg == 16, "pairwise sum of 16 masses");
        DS s8[8];
#pragma unroll
        for (int i = 0; i < kRegSeg; ++i)
            if (i0 + i < i1) wmass[i0 + i] = mv[i];
#pragma unroll
        for (int i = 0; i < 8; ++i) s8[i] = ds_two_sum(mv[2 * i], mv[2 * i + 1]);
#pragma unroll
        for (int i = 0; i < 4; ++i) s8[i] = ds_add(s8[2 * i], s8[2 * i + 1]);
#pragma unroll
        for (int i = 0; i < 2; ++i) s8[i] = ds_add(s8[2 * i], s8[2 * i + 1]);
        sum = ds_add(s8[0], s8[1]);
        __syncwarp();
    } else {
        for (int i = i0; i < i1; ++i) sum = ds_add_f(sum, dec_mass(ld_relaxed_u32(mw + i)));
    }
    DS incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const DS y = ds_shfl_up(incl, o);
        if (lane >= o) incl = ds_add(incl, y);
    }
    DS R = ds_shfl(incl, 31);
    DS P = ds_shfl_up(incl, 1);
    if (lane == 0) P = DS{0.f, 0.f};
    DS t = ds_mul_f(R, u);
    int found = -1;
    DS fb{0.f, 0.f};
    int fseg = -1;
    DS fbase{0.f, 0.f};
    if (in_regs) {
        // The first lane whose running total passes t, then the first of its segments: its masses
        // spread over lanes 0..G-1 (read back from shared memory) and one double-single scan.  (If none of them passes t, a rounding
        // difference between the two sums: its last segment, whose in-segment scan then moves on.)
        const unsigned lb = __ballot_sync(0xffffffffu, ds_gt(incl, t));
        if (lb) {
            const int L = __ffs(lb) - 1;
            const int iL0 = min(L * G, ns), cnt = min(iL0 + G, ns) - iL0;
            const float mine = lane < cnt ? wmass[iL0 + lane] : 0.f;
            DS e{mine, 0.f};
#pragma unroll
            for (int o = 1; o < kRegSeg; o <<= 1) {
                const DS y = ds_shfl_up(e, o);
                if (lane >= o) e = ds_add(e, y);
            }
            DS ex = ds_shfl_up(e, 1);
            if (lane == 0) ex = DS{0.f, 0.f};
            const DS PL = ds_shfl(P, L);
            const unsigned fl = __ballot_sync(0xffffffffu, lane < cnt && ds_gt(ds_add(PL, e), t));
            const int j = fl ? __ffs(fl) - 1 : cnt - 1;
            fseg = iL0 + j;
            fbase = ds_add(PL, ds_shfl(ex, j));
        }
    } else {
        for (int i = i0; i < i1; ++i) {
            const DS Pn = ds_add_f(P, dec_mass(ld_relaxed_u32(mw + i)));
            if (found < 0 && ds_gt(Pn, t)) {
                found = i;
                fb = P;
            }
            P = Pn;
        }
    }
    for (int i = i0; i < i1; ++i) st_relaxed_u32(mw + i, 0u);  // consumed: leave the records zeroed
    if (!in_regs) {
        const unsigned ball = __ballot_sync(0xffffffffu, found >= 0);
        const int src = ball ? (__ffs(ball) - 1) : 0;
        fseg = ball ? __shfl_sync(0xffffffffu, found, src) : -1;
        fbase = ds_shfl(fb, src);
    }
    if (!(R.hi > 0.f)) {
        // empty residual after a rejection: draw from p instead (slow path, one segment at a time)
        qrow = nullptr;
        if (lane == 0) atomicOr(a.status, SV_FLAG_ZERO_RESIDUAL);
        DS acc{0.f, 0.f};
        for (int g = 0; g < ns; ++g) {
            float r[2][4];
            seg_load_r<T>(zrow, nullptr, a.V, g, a.c, M, invS, lane, r);
            acc = ds_add_f(acc, seg_sum(r));
        }
        R = acc;
        t = ds_mul_f(R, u);
        fseg = -1;
        fbase = DS{0.f, 0.f};
        DS Pp{0.f, 0.f};
        for (int g = 0; g < ns && fseg < 0; ++g) {
            float r[2][4];
            seg_load_r<T>(zrow, nullptr, a.V, g, a.c, M, invS, lane, r);
            const DS Pn = ds_add_f(Pp, seg_sum(r));
            if (ds_gt(Pn, t)) {
                fseg = g;
                fbase = Pp;
            }
            Pp = Pn;
        }
    }
    int vstar = -1;
    float rstar = 0.f;
    if (fseg >= 0) {
        float r[2][4];
        seg_load_r<T>(zrow, qrow, a.V, fseg, a.c, M, invS, lane, r);
        const TileScan ts = warp_seg_scan(r, fseg, a.V, fbase, t, lane);
        vstar = ts.v;
        rstar = ts.rv;
        for (int g = fseg + 1; g < ns && vstar < 0; ++g) {
            seg_load_r<T>(zrow, qrow, a.V, g, a.c, M, invS, lane, r);
            int loc = 0x7fffffff;
            float rloc = 0.f;
#pragma unroll
            for (int j = 1; j >= 0; --j)
#pragma unroll
                for (int k = 3; k >= 0; --k)
                    if (r[j][k] > 0.f) {
                        loc = (j * 32 + lane) * 4 + k;
                        rloc = r[j][k];
                    }
            const int best = __reduce_min_sync(0xffffffffu, loc);
            if (best != 0x7fffffff) {
                const unsigned m = __ballot_sync(0xffffffffu, loc == best);
                rstar = __shfl_sync(0xffffffffu, rloc, __ffs(m) - 1);
                vstar = g * kSegElems + best;
            }
        }
    }
    for (int g = ns - 1; g >= 0 && vstar < 0; --g) {
        float r[2][4];
        seg_load_r<T>(zrow, qrow, a.V, g, a.c, M, invS, lane, r);
        int loc = -1;
        float rloc = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (r[j][k] > 0.f) {
                    loc = (j * 32 + lane) * 4 + k;
                    rloc = r[j][k];
                }
        const int best = __reduce_max_sync(0xffffffffu, loc);
        if (best >= 0) {
            const unsigned m = __ballot_sync(0xffffffffu, loc == best);
            rstar = __shfl_sync(0xffffffffu, rloc, __ffs(m) - 1);
            vstar = g * kSegElems + best;
        }
    }
    if (lane == 0) {
        a.out_tokens[sel.row] = vstar;
        if (a.diag) {
            const float Rf = __fadd_rn(R.hi, R.lo);
            a.diag[a.n_draft + 2 * b] = Rf;
            a.diag[a.n_draft + 2 * b + 1] = __fdiv_rn(rstar, Rf);
        }
    }
    return true;
}

template <typename T, bool kSample>
__global__ void __launch_bounds__(kThreads, 1) fused_kernel(Args a) {
    constexpr int VEC = Elem<T>::kVec;
    constexpr int CHUNK = chunk_elems<T>();
    static_assert(CHUNK * sizeof(T) == kChunkBytes, "stats chunk must fill one ring stage");
    static_assert(kResElems * 4 <= kResQOffset && kResQOffset + kResElems * 4 <= kChunkBytes, "residual stage");
    static_assert(kResElems % kSegElems == 0 && kResElems / kSegElems == kCons, "one segment per consumer warp");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nb = (a.n_chunks + kBlockChunks - 1) / kBlockChunks;  // stats blocks per row
    const int total_blocks = a.rows * nb;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kCons);
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // Launched with programmatic stream serialization: the set-up above may
    // overlap the previous kernel on the stream, whose results (the logits,
    // this workspace) are visible only after this wait.
    pdl_wait_prior_grid();
    pdl_launch_dependents();
    if (a.row_offsets) {
        // the CSR offsets are checked here, by every CTA (the same verdict in each), instead of by a
        // kernel of their own ahead of this one: offsets[0] = 0, offsets[B] = rows, 1..256 rows each
        bool bad = tid == 0 && (__ldg(a.row_offsets) != 0 || __ldg(a.row_offsets + a.B) != a.rows);
        for (int b = tid; b < a.B; b += kThreads) {
            const int k1 = __ldg(a.row_offsets + b + 1) - __ldg(a.row_offsets + b);
            bad |= (k1 < 1 || k1 > kMaxRowsPerRequest);
        }
        if (__syncthreads_or(bad)) {
            if (blockIdx.x == 0) {
                for (int b = tid; b < a.B; b += kThreads) a.accept_len[b] = 0;
                for (int r = tid; r < a.rows; r += kThreads) a.out_tokens[r] = -1;
                if (tid == 0) atomicOr(a.status, SV_FLAG_BAD_OFFSETS);
            }
            return;
        }
    }
    volatile int *abort_flag = &sm.abort;
    const long long t_start = clock64();
    auto timeout = [&]() {
        *abort_flag = 1;
        atomicOr(a.status, SV_FLAG_TIMEOUT);
    };

    if (warp == kProducer) {
        if (lane == 0) {
            int k = 0;  // ring stage counter
            // next ring stage: wait until the consumers released it
            auto claim = [&](int &s) -> bool {
                s = k % kStages;
                if (k >= kStages && !mbar_wait_bounded(&sm.empty[s], ((k / kStages) - 1) & 1, a.wait_budget)) {
                    timeout();
                    return false;
                }
                return !*abort_flag;
            };
            bool ok = true;
            const uint32_t total_rb = kSample ? residual_claims(a) : 0u;
            // L2 priorities: a request's first rows are the ones its residual pass most often re-reads
            // (acceptance decays with position, so the earliest drafts are the likeliest to be rejected):
            // its first keep_rows rows are loaded at normal priority (keep_rows sized on the host to a
            // quarter of L2), every other stats row and every residual read as evict_first, so the kept
            // rows outlive the stream without outliving the step's successors.  With early residual
            // claims (no row kept) every stats row loads at normal priority: its request's residual
            // claim comes a few microseconds later, and evict_first lines would be gone by then.
            const uint64_t keep = l2_evict_normal_policy(), stream_through = l2_evict_first_policy();
            int jn = static_cast<int>(atomicAdd(a.sched + 0, 1u));
            uint32_t pn = 0xffffffffu;     // next residual claim (in flight)
            int nb_req = -1;               // request of the next claim whose decision words were read ahead
            uint64_t nw0 = 0ull, nw1 = 0ull;
            int cb = -1, crow = -1, cqrow = -1;  // the last decision read
            float cM = 0.f, cinvS = 0.f;
            // the stages of one residual claim (b's selected row and, after a rejection, its q row)
            auto issue_claim = [&](const Claim &cl, int row, int qrow, float M, float invS) -> bool {
                const bool has_q = qrow >= 0;
                for (int st = 0; st < cl.nst; ++st) {
                    const int c0 = (cl.st0 + st) * kResElems;
                    if (c0 >= a.V) break;
                    const int n = min(kResElems, a.V - c0);
                    int s;
                    if (!claim(s)) return false;
                    sm.tag[s] = Tag{kRes, cl.b, c0 / kResElems, n, has_q ? 1 : 0, 0, M, invS};
                    const uint32_t zb = static_cast<uint32_t>(n) * sizeof(T);
                    const uint32_t qb = has_q ? static_cast<uint32_t>(n) * 4u : 0u;
                    mbar_arrive_expect_tx(&sm.full[s], zb + qb);
                    bulk_g2s_hint(sm.ring[s], reinterpret_cast<const T *>(a.logits) + static_cast<size_t>(row) * a.V + c0,
                                  zb, &sm.full[s], stream_through);
                    if (has_q)
                        bulk_g2s_hint(sm.ring[s] + kResQOffset, a.q + static_cast<size_t>(qrow) * a.V + c0, qb,
                                      &sm.full[s], stream_through);
                    ++k;
                }
                return true;
            };
            // With early_res, a producer holds at most one residual claim during the stats stream.
            // Its request's decision words are loaded one stats block ahead; once they are out, the
            // claim's stages go ahead of the next stats block, while the request's rows are still in
            // L2.  Chosen on the host when no logits row can be kept in L2 through the whole stream:
            // then the residual pass after the stream would re-read every selected row from DRAM.
            uint32_t held = 0xffffffffu;
            bool claims_left = kSample && a.early_res != 0;
            uint64_t hw0 = 0ull, hw1 = 0ull;
            while (ok) {
                // 1. stats blocks first (row order, grid-wide counter): the decisions wait on them
                if (jn < total_blocks) {
                    if (kSample && (claims_left || held != 0xffffffffu)) {
                        if (held != 0xffffffffu && (hw0 >> 32) != 0 && (hw1 >> 32) != 0) {
                            const int hrow = static_cast<int>(static_cast<uint32_t>(hw1));
                            if (hrow >= 0 &&
                                !issue_claim(decode_claim(held, a), hrow,
                                             static_cast<int>(static_cast<uint32_t>(hw1 >> 32)) - 2,
                                             __uint_as_float(static_cast<uint32_t>(hw0)),
                                             __uint_as_float(static_cast<uint32_t>(hw0 >> 32) ^ 0x80000000u))) {
                                ok = false;
                                break;
                            }
                            held = 0xffffffffu;
                        }
                        if (held == 0xffffffffu && claims_left) {
                            held = atomicAdd(a.sched + 2, 1u);
                            if (held >= total_rb) {
                                held = 0xffffffffu;
                                claims_left = false;
                            }
                        }
                        if (held != 0xffffffffu) {  // checked before the next stats block
                            const int hb = decode_claim(held, a).b;
                            hw0 = ld_relaxed_u64(a.fdec + 2 * hb);
                            hw1 = ld_relaxed_u64(a.fdec + 2 * hb + 1);
                        }
                    }
                    const int j = jn;
                    jn = static_cast<int>(atomicAdd(a.sched + 0, 1u));  // in flight while this block is issued
                    const int row = j / nb;
                    const bool first_row = kSample && (a.row_offsets ? row - __ldg(a.row_offsets + request_of_row(a, row)) < a.keep_rows
                                                                     : row % (a.K + 1) < a.keep_rows);
                    const int first = (j - row * nb) * kBlockChunks;
                    const int cnt = min(kBlockChunks, a.n_chunks - first);
                    for (int cc = 0; cc < cnt; ++cc) {
                        int s;
                        if (!claim(s)) {
                            ok = false;
                            break;
                        }
                        const int chunk = first + cc;
                        const int c0 = chunk * CHUNK;
                        const int n = min(CHUNK, a.V - c0);
                        sm.tag[s] = Tag{kStats, row, chunk, n, 0, cc == cnt - 1 ? 1 : 0, 0.f, 0.f};
                        const uint32_t bytes = static_cast<uint32_t>(n) * sizeof(T);
                        mbar_arrive_expect_tx(&sm.full[s], bytes);
                        bulk_g2s_hint(sm.ring[s],
                                      reinterpret_cast<const T *>(a.logits) + static_cast<size_t>(row) * a.V + c0, bytes,
                                      &sm.full[s], (first_row || a.early_res) ? keep : stream_through);
                        ++k;
                    }
                    continue;
                }
                if (!kSample) break;
                // 2. residual claims (consecutive stages of one request's selected row), grid-wide
                // in request order.  One claim is kept in flight and its decision words are loaded
                // while the current claim's stages are issued.
                if (held != 0xffffffffu) {  // the claim held through the stats stream comes first
                    pn = held;
                    nb_req = decode_claim(held, a).b;
                    nw0 = hw0;
                    nw1 = hw1;
                    held = 0xffffffffu;
                }
                if (pn == 0xffffffffu) pn = atomicAdd(a.sched + 2, 1u);
                const uint32_t p = pn;
                if (p >= total_rb) break;
                const Claim cl = decode_claim(p, a);
                const int b = cl.b;
                if (b != cb) {
                    uint64_t w0 = (b == nb_req) ? nw0 : ld_relaxed_u64(a.fdec + 2 * b);
                    uint64_t w1 = (b == nb_req) ? nw1 : ld_relaxed_u64(a.fdec + 2 * b + 1);
                    while ((w0 >> 32) == 0 || (w1 >> 32) == 0) {  // not published yet
                        if (*abort_flag) {
                            ok = false;
                            break;
                        }
                        if (clock64() - t_start > a.wait_budget) {
                            timeout();
                            ok = false;
                            break;
                        }
                        __nanosleep(kPollNs);
                        w0 = ld_relaxed_u64(a.fdec + 2 * b);
                        w1 = ld_relaxed_u64(a.fdec + 2 * b + 1);
                    }
                    if (!ok) break;
                    cb = b;
                    crow = static_cast<int>(static_cast<uint32_t>(w1));
                    cqrow = static_cast<int>(static_cast<uint32_t>(w1 >> 32)) - 2;
                    cM = __uint_as_float(static_cast<uint32_t>(w0));
                    cinvS = __uint_as_float(static_cast<uint32_t>(w0 >> 32) ^ 0x80000000u);
                }
                pn = atomicAdd(a.sched + 2, 1u);  // the next claim
                if (pn < total_rb) {               // its decision, read ahead
                    nb_req = decode_claim(pn, a).b;
                    if (nb_req != cb) {
                        nw0 = ld_relaxed_u64(a.fdec + 2 * nb_req);
                        nw1 = ld_relaxed_u64(a.fdec + 2 * nb_req + 1);
                    } else {
                        nb_req = -1;
                    }
                }
                if (crow < 0) continue;  // invalid request: nothing to draw
                if (!issue_claim(cl, crow, cqrow, cM, cinvS)) ok = false;
            }
            // end of stream (a phase without data), or wait for issued copies on abort
            int s;
            if (ok && claim(s)) {
                sm.tag[s] = Tag{kEnd, 0, 0, 0, 0, 0, 0.f, 0.f};
                mbar_arrive(&sm.full[s]);
            } else {
                for (int kk = max(0, k - kStages); kk < k; ++kk)
                    mbar_wait_bounded(&sm.full[kk % kStages], (kk / kStages) & 1, kDrainBudget);  // own copies
            }
        }
        // This CTA streams nothing more.  The last producer out resets the scheduling counters
        // and zeroes the decision records for the next call: every producer has read them by then
        // (each request's decision is read before any of its residual blocks streams), and the
        // counters are used by producers only.  Off the path of the final draws.
        int last = 0;
        if (lane == 0) {
            __threadfence();
            last = (atomicAdd(a.sched + 1, 1u) + 1u == gridDim.x) ? 1 : 0;
            if (last) __threadfence();
        }
        if (__shfl_sync(0xffffffffu, last, 0)) {
            if (kSample)
                for (int i = lane; i < 2 * a.B; i += 32) a.fdec[i] = 0ull;
            if (lane == 0) {
                a.sched[0] = 0u;
                a.sched[2] = 0u;
                a.sched[1] = 0u;
            }
        }
    } else if (warp == kWorker) {
        for (int b = blockIdx.x; b < a.B; b += gridDim.x) {
            Sel sel;
            if (!fused_decide<T, kSample>(a, b, lane, abort_flag, t_start, sel)) break;
            if (!kSample) continue;
            const float invS = 1.f / sel.S;
            if (lane == 0) {
                if (sel.valid) publish_decision(a.fdec + 2 * b, sel.M, invS, sel.row, sel.qrow);
                else publish_decision(a.fdec + 2 * b, 0.f, 1.f, -1, -1);
            }
            if (sel.valid && !fused_draw<T>(a, b, sel, invS, lane, abort_flag, t_start, sm.wmass)) break;
        }
    } else {
        // consumers
        int open = 0, seg_row = 0, seg_first = 0;
        float ra;
        int rb;
        partial_identity<kSample>(ra, rb);
        for (int k = 0;; ++k) {
            const int s = k % kStages;
            if (!mbar_wait_bounded(&sm.full[s], (k / kStages) & 1, a.wait_budget)) timeout();
            if (*abort_flag) break;
            const Tag tg = sm.tag[s];
            if (tg.kind == kEnd) break;
            if (tg.kind == kRes) {
                float m = res_lane_sum<T>(sm.ring[s], warp, lane, tg.n, tg.has_q != 0, a.c, tg.M, tg.invS);
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.empty[s]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m += __shfl_xor_sync(0xffffffffu, m, o);
                const int seg = tg.chunk * (kResElems / kSegElems) + warp;  // this warp's 256 tokens
                if (lane == 0 && seg < a.n_seg)
                    st_relaxed_u32(a.fmass + static_cast<size_t>(tg.row) * a.n_seg + seg, enc_mass(m));
                continue;
            }
            if (!open) {  // first chunk of a stats block
                open = 1;
                seg_row = tg.row;
                seg_first = tg.chunk;
                partial_identity<kSample>(ra, rb);
            }
            const int c0 = tg.chunk * CHUNK;
            const uint4 *stage = reinterpret_cast<const uint4 *>(sm.ring[s]);
            float vals[kVecs][VEC];
            int e0[kVecs];
            if (tg.n == CHUNK) {
#pragma unroll
                for (int j = 0; j < kVecs; ++j) {
                    const int v = warp * (kVecs * 32) + j * 32 + lane;
                    e0[j] = v * VEC;
                    unpack(stage[v], vals[j]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.empty[s]);
                lane_accumulate<kSample, true, kVecs, VEC>(vals, e0, CHUNK, c0, a.c, ra, rb);
            } else {
#pragma unroll
                for (int j = 0; j < kVecs; ++j) {
                    const int v = warp * (kVecs * 32) + j * 32 + lane;
                    e0[j] = v * VEC;
                    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
                    if (e0[j] < tg.n) raw = stage[v];
                    unpack(raw, vals[j]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.empty[s]);
                lane_accumulate<kSample, false, kVecs, VEC>(vals, e0, tg.n, c0, a.c, ra, rb);
            }
            if (tg.last) {  // the block is complete: store this warp's partial of it
                float wa = ra;
                int wb = rb;
                warp_partial_reduce<kSample>(wa, wb);
                if (lane == 0)
                    st_relaxed_u64(a.fpart + static_cast<size_t>(seg_row) * a.n_pe + (seg_first / kBlockChunks) * kCons +
                                       warp,
                                   enc_partial<kSample>(wa, wb));
                open = 0;
            }
        }
    }
}

}  // namespace fz



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
    size_t status, csr_ok, tickets1, fpart, fmass, fdec, dec, partials, tile_mass, cv_segs, total;
    bool rec_overflow;  // the fused records exceed the fixed region: they follow the rest, cleared per call
};

static inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Per-request counters and the fused kernel's records live in a region of
// fixed capacity right after the status words, whatever the call's shape,
// and every completed call leaves what it used there at zero.  A workspace
// therefore serves calls of any shape once it has been zero-filled; only a
// call whose counters or records exceed the capacities clears them first.
constexpr int kTicketCap = 16384;
constexpr int kSchedWords = 8;
constexpr size_t kL2KeepBytes = 32ull << 20;  // fused kernel: logits rows kept in L2 (a quarter of it)
constexpr size_t kRecPartCap = 32768;  // fused partial records (rows x n_pe)
constexpr size_t kRecMassCap = 65536;  // fused segment masses (B x n_seg)
constexpr size_t kRecDecCap = 8192;    // fused decision words (2 B)

static WsLayout ws_layout(int B, int rows, int V, bool with_partials = true) {
    WsLayout L;
    const size_t n_chunks = (static_cast<size_t>(V) + chunk_elems<float>() - 1) / chunk_elems<float>();
    const size_t n_tiles = (static_cast<size_t>(V) + kTileElems - 1) / kTileElems;
    size_t o = 0;
    L.status = o; o = align256(o + 16);
    L.csr_ok = o; o = align256(o + 16);
    const size_t cap = static_cast<size_t>(B > kTicketCap ? B : kTicketCap);
    L.tickets1 = o; o = align256(o + 4ull * (cap + kSchedWords));  // tickets1 | sched
    // fused records, sized for fp32 chunks (the larger count)
    const size_t n_pe = ((n_chunks + fz::kBlockChunks - 1) / fz::kBlockChunks) * fz::kCons;
    const size_t n_seg = (static_cast<size_t>(V) + kSegElems - 1) / kSegElems;
    const size_t need_part = static_cast<size_t>(rows) * n_pe, need_mass = static_cast<size_t>(B) * n_seg,
                 need_dec = 2ull * static_cast<size_t>(B);
    L.rec_overflow = need_part > kRecPartCap || need_mass > kRecMassCap || need_dec > kRecDecCap;
    L.fpart = o; o = align256(o + 8 * kRecPartCap);
    L.fmass = o; o = align256(o + 4 * kRecMassCap);
    L.fdec = o; o = align256(o + 8 * kRecDecCap);
    L.dec = o; o = align256(o + sizeof(Decision) * static_cast<size_t>(B));
    L.partials = o; o = align256(o + (with_partials ? sizeof(float2) * static_cast<size_t>(rows) * n_chunks : 0));
    L.tile_mass = o; o = align256(o + sizeof(float) * static_cast<size_t>(B) * n_tiles);
    // segment sums of the cluster kernel, for the batches it may take
    const bool cv_fits = with_partials && B <= cv::kMaxB && cv::segs_per_cta(V) <= cv::kMaxSegs;
    L.cv_segs = o; o = align256(o + (cv_fits ? sizeof(float) * static_cast<size_t>(B) * n_seg : 0));
    if (L.rec_overflow) {
        L.fpart = o; o = align256(o + 8 * need_part);
        L.fmass = o; o = align256(o + 4 * need_mass);
        L.fdec = o; o = align256(o + 8 * need_dec);
    }
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

// Counters and fused records of a workspace laid out as L.
static void set_ws_records(Args &a, char *w, const WsLayout &L) {
    a.tickets1 = reinterpret_cast<uint32_t *>(w + L.tickets1);
    a.sched = a.tickets1 + (a.B > kTicketCap ? a.B : kTicketCap);
    a.fpart = reinterpret_cast<uint64_t *>(w + L.fpart);
    a.fmass = reinterpret_cast<uint32_t *>(w + L.fmass);
    a.fdec = reinterpret_cast<uint64_t *>(w + L.fdec);
    a.n_seg = (a.V + kSegElems - 1) / kSegElems;
    a.n_rb = (a.V + kResBlockElems - 1) / kResBlockElems;
}

static void *g_prof_begin = nullptr;
static void *g_prof_end = nullptr;
static thread_local int g_last_launches = 0;
static thread_local const char *g_last_kernel = "none";

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

template <typename T, bool kSample>
static void launch_fused(const Args &a, cudaStream_t s) {
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!configured[dev]) {
        cudaFuncSetAttribute(fz::fused_kernel<T, kSample>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(fz::Smem)));
        configured[dev] = true;
    }
    const int nb = (a.n_chunks + fz::kBlockChunks - 1) / fz::kBlockChunks;
    const long long blocks = static_cast<long long>(a.rows) * nb;
    const unsigned grid = static_cast<unsigned>(blocks < sm_count() ? blocks : sm_count());
    launch_pdl(fz::fused_kernel<T, kSample>, dim3(grid), dim3(fz::kThreads), sizeof(fz::Smem), s, a);
}

// small_nr > 0: the request-per-CTA kernel with room for small_nr rows per request;
// cluster_nr > 0: one cluster per request with room for cluster_nr rows per request.
template <typename T>
static sv_status run_typed(Args &a, bool sample, bool vec, int small_nr, int cluster_nr, cudaStream_t s) {
    a.n_chunks = (a.V + chunk_elems<T>() - 1) / chunk_elems<T>();
    int launches = 0;
    a.n_pe = ((a.n_chunks + fz::kBlockChunks - 1) / fz::kBlockChunks) * fz::kCons;
    a.n_st = (a.V + kResStageElems - 1) / kResStageElems;
    {
        const int tail = a.B / 8 > 0 ? a.B / 8 : 1;  // the last eighth of the requests
        a.tail_b0 = a.B - (tail < a.B ? tail : a.B);
    }
    {
        // positions per request whose logits rows fit in a quarter of L2 across the batch
        const size_t per_position = static_cast<size_t>(a.B) * a.V * sizeof(T);
        const size_t keep = per_position ? (kL2KeepBytes / per_position) : 0;
        a.keep_rows = static_cast<int>(keep < static_cast<size_t>(kMaxRowsPerRequest) ? keep : kMaxRowsPerRequest);
        // no row kept: start residual claims during the stats stream, while the selected rows are in L2
        a.early_res = (sample && a.keep_rows == 0) ? 1 : 0;
    }
    if (a.B > kTicketCap &&
        cudaMemsetAsync(a.tickets1, 0, sizeof(uint32_t) * (static_cast<size_t>(a.B) + kSchedWords), s) !=
            cudaSuccess)
        return SV_ERR_CUDA;
    const bool fused = small_nr == 0 && cluster_nr == 0 && vec;  // checks the offsets itself
    if (a.row_offsets && !fused) {
        csr_check_kernel<<<1, kThreads, 0, s>>>(a, const_cast<int *>(a.csr_ok));
        ++launches;
    }
    prof_begin(s);
    g_last_kernel = small_nr > 0 ? "small" : cluster_nr > 0 ? "cluster" : vec ? "stream" : "scalar";
    if (small_nr > 0) {
        // small vocabulary: one CTA per request, everything in shared memory
        const cudaError_t e = launch_small_kernel(a, small_nr, sample, sizeof(T) == 2, s);
        prof_end(s);
        ++launches;
        set_launches(launches);
        return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? SV_OK : SV_ERR_CUDA;
    }
    if (cluster_nr > 0) {
        // medium requests in small batches: one cluster of CTAs per request
        const cudaError_t e = launch_cluster_kernel(a, cluster_nr, sample, sizeof(T) == 2, s);
        prof_end(s);
        ++launches;
        set_launches(launches);
        return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? SV_OK : SV_ERR_CUDA;
    }
    if (vec) {
        // aligned rows: the whole step in one persistent kernel
        if (sample) launch_fused<T, true>(a, s); else launch_fused<T, false>(a, s);
        prof_end(s);
        ++launches;
        set_launches(launches);
        return (cudaGetLastError() == cudaSuccess) ? SV_OK : SV_ERR_CUDA;
    }
    if (sample) launch_scalar_pass1<T, true>(a, s);
    else launch_scalar_pass1<T, false>(a, s);
    prof_end(s);
    ++launches;
    if (sample) {
        launch_pass2<T, false>(a, s);
        ++launches;
    }
    set_launches(launches);
    return (cudaGetLastError() == cudaSuccess) ? SV_OK : SV_ERR_CUDA;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Requests holding at most this many bytes of logits run on sk::small_kernel.
static std::atomic<size_t> g_small_limit{sk::kDefaultRowBytes};
// Whether small batches of medium requests may run on cv::cluster_kernel.
static std::atomic<int> g_cluster_on{1};
// Limit of the waits on other warps' or CTAs' work (spec_set_wait_budget).
static std::atomic<long long> g_wait_budget{kDefaultWaitBudget};
long long wait_budget() { return g_wait_budget.load(std::memory_order_relaxed); }

// Host-side argument rules of every verification call (workspace aside):
// SV_ERR_INVALID if one is broken, else SV_OK.  B = 0 passes (a no-op call).
sv_status check_verify_args(const void *logits, sv_dtype dt, const float *q, const int32_t *row_offsets,
                            int B, int K, long long rows, int V, float temperature, bool sample,
                            const int32_t *draft, const float *uniforms, const int32_t *out_tokens,
                            const int32_t *accept_len) {
    if (B < 0 || V <= 0 || rows < 0 || (dt != SV_F32 && dt != SV_BF16)) return SV_ERR_INVALID;
    if (!row_offsets && (K < 0 || K > SV_MAX_K)) return SV_ERR_INVALID;
    if (B == 0) return SV_OK;
    if (rows < B || rows > INT_MAX || rows * V >= (1ll << 62)) return SV_ERR_INVALID;
    if (!logits || !out_tokens || !accept_len) return SV_ERR_INVALID;
    if (rows > B && !draft) return SV_ERR_INVALID;
    if (sample && (!(temperature > 0.f) || !std::isfinite(temperature) || !uniforms || (rows > B && !q)))
        return SV_ERR_INVALID;
    return SV_OK;
}

// Common host path of the three logits-in entry points.
static sv_status verify_common(const void *logits, sv_dtype dt, const float *q,
                               const int32_t *row_offsets, int B, int K, long long rows64, int V,
                               float temperature, bool sample, const int32_t *draft,
                               const float *uniforms, int32_t *out_tokens, int32_t *accept_len,
                               float *diag, void *ws, size_t ws_bytes, void *stream) {
    const sv_status arg = check_verify_args(logits, dt, q, row_offsets, B, K, rows64, V, temperature, sample,
                                            draft, uniforms, out_tokens, accept_len);
    if (arg != SV_OK) return arg;
    if (B == 0) {
        set_launches(0);
        return SV_OK;
    }
    if (!ws) return SV_ERR_INVALID;
    const int rows = static_cast<int>(rows64);
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
    a.wait_budget = wait_budget();
    a.csr_ok = row_offsets ? reinterpret_cast<const int *>(w + L.csr_ok) : nullptr;
    set_ws_records(a, w, L);
    a.dec = reinterpret_cast<Decision *>(w + L.dec);
    a.partials = reinterpret_cast<float2 *>(w + L.partials);
    a.tile_mass = reinterpret_cast<float *>(w + L.tile_mass);

    const size_t esize = (dt == SV_F32) ? 4 : 2;
    const bool vec = aligned16(logits) && ((static_cast<size_t>(V) * esize) % 16 == 0) &&
                     (!q || (aligned16(q) && V % 4 == 0));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // rows per request at most: K + 1, or (ragged) what the batch leaves for one request
    const int nr_cap = row_offsets ? std::min(kMaxRowsPerRequest, rows - B + 1) : K + 1;
    const size_t limit = g_small_limit.load(std::memory_order_relaxed);
    const bool small = static_cast<size_t>(nr_cap) * V * esize <= limit &&
                       sk::smem_bytes(nr_cap, V, static_cast<int>(esize)) <= sk::kMaxSmemBytes;
    // a cluster per request: aligned rows, at most two CTAs per SM for the batch, slices in shared memory
    const bool cluster = !small && vec && g_cluster_on.load(std::memory_order_relaxed) != 0 &&
                         nr_cap <= cv::kMaxRows && B <= cv::kMaxB && cv::segs_per_cta(V) <= cv::kMaxSegs &&
                         B * cv::kC <= 2 * sm_count() &&
                         cv::smem_bytes(nr_cap, V, static_cast<int>(esize)) <= cv::kSmemCap;
    if (cluster) a.cv_segs = reinterpret_cast<float *>(w + L.cv_segs);
    if (vec && !small && !cluster && L.rec_overflow &&
        cudaMemsetAsync(w + L.fpart, 0, L.total - L.fpart, s) != cudaSuccess)  // records beyond the fixed region
        return SV_ERR_CUDA;
    const int small_nr = small ? nr_cap : 0, cluster_nr = cluster ? nr_cap : 0;
    if (dt == SV_F32) return run_typed<float>(a, sample, vec, small_nr, cluster_nr, s);
    return run_typed<__nv_bfloat16>(a, sample, vec, small_nr, cluster_nr, s);
}


// Workspace of finish_from_partials (the partials live elsewhere).
size_t finish_workspace_size(int B, int rows, int V) { return ws_layout(B, rows, V, false).total; }


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
    a.wait_budget = wait_budget();
    a.csr_ok = nullptr;
    set_ws_records(a, w, L);
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
    return verify_common(logits, dt, nullptr, nullptr, B, K, static_cast<long long>(B) * (K + 1), V, 0.f, false, draft,
                         nullptr, out_tokens, accept_len, nullptr, ws, ws_bytes, stream);
}

extern "C" sv_status spec_verify_sample(const void *logits, sv_dtype dt, const float *q, int B,
                                        int K, int V, float temperature, const int32_t *draft,
                                        const float *uniforms, int32_t *out_tokens,
                                        int32_t *accept_len, float *diag, void *ws,
                                        size_t ws_bytes, void *stream) {
    if (K < 0 || K > SV_MAX_K || B < 0) return SV_ERR_INVALID;
    return verify_common(logits, dt, q, nullptr, B, K, static_cast<long long>(B) * (K + 1), V, temperature, true, draft,
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

extern "C" const char *spec_last_kernel(void) { return g_last_kernel; }

extern "C" int spec_set_cluster_kernel(int enable) {
    return g_cluster_on.exchange(enable != 0 ? 1 : 0, std::memory_order_relaxed);
}

extern "C" long long spec_set_wait_budget(long long cycles) {
    if (cycles < 0) return -1;
    return g_wait_budget.exchange(cycles == 0 ? kDefaultWaitBudget : cycles, std::memory_order_relaxed);
}

extern "C" size_t spec_set_small_kernel_limit(size_t bytes) {
    return g_small_limit.exchange(bytes, std::memory_order_relaxed);
}
