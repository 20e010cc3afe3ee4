// Verification kernels and the C ABI of libspecverify.so (sm_103a).
//
// Pass 1  stats_decide_kernel   one CTA per (logits row, chunk of the vocabulary)
//         streams the logits once with 128-bit loads and reduces the chunk to
//         (M, s) = (max z c, sum 2^(z c - M)) with c = log2(e)/T (sampling) or
//         to (max z, first argmax) (greedy).  The last CTA of each request
//         (epoch ticket) merges its rows' chunk partials and runs the decide
//         step: accept tests u q(x) <= p(x), first-rejection scan, emitted
//         drafts, AL, and the record of the row the final token comes from.
// Pass 2  residual_kernel       (sampling only) one CTA per (request, 8 tiles
//         of 1024 tokens) of the selected row: r = max(0, p - q) at a
//         rejection or r = p for the bonus, tile masses; the last CTA of the
//         request takes the prefix over tiles in fp64, finds the tile holding
//         u R, and resolves the token inside it with a block scan that is
//         bit-identical to the one that produced the tile's mass.
//
// The operation is the one stated on "Speculative Decoding in Large Language
// Models", section 2 "Modified Rejection Sampling" (accept test, residual
// p'(x)), with the stop at the first mismatch and the extra target token of
// "Co-Designing AI Models Using Speculative Decoding", "What is speculative
// decoding?".  See include/specverify.h for the full contract.
#include <unistd.h>

#include <atomic>
#include <chrono>
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
    int B, K, V, rows, n_chunks, n_tiles, n_parts, n_draft;
    float c;  // log2(e) / T
    uint32_t epoch;
    // workspace
    uint32_t *status;
    const int *csr_ok;
    unsigned long long *tickets1;
    unsigned long long *tickets2;
    Decision *dec;
    float2 *partials;
    float *tile_mass;
};

__device__ __forceinline__ void request_rows(const Args &a, int b, int &r0, int &nr) {
    if (a.row_offsets) {
        r0 = a.row_offsets[b];
        nr = a.row_offsets[b + 1] - r0;
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

// ---------------------------------------------------------------------------
// Decide step of request b (whole CTA).  Runs after every chunk partial of the
// request's rows is visible.
// ---------------------------------------------------------------------------
struct DecideSmem {
    float M[kMaxRowsPerRequest];
    float S[kMaxRowsPerRequest];
    int arg[kMaxRowsPerRequest];
    int bad;
    int kstar;
};

template <typename T, bool kSample>
__device__ void decide(const Args &a, int b, DecideSmem &sh) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int r0, nr;
    request_rows(a, b, r0, nr);
    const int Kb = nr - 1;
    const int d0 = r0 - b;
    if (tid == 0) {
        sh.bad = 0;
        sh.kstar = Kb;
    }
    __syncthreads();
    for (int j = tid; j < Kb; j += kThreads) {
        const int x = a.draft[d0 + j];
        if (x < 0 || x >= a.V) sh.bad = 1;
    }
    __syncthreads();
    if (sh.bad) {
        for (int j = tid; j < nr; j += kThreads) a.out_tokens[r0 + j] = -1;
        if (tid == 0) {
            a.accept_len[b] = 0;
            if (kSample) {
                Decision d{};
                d.valid = 0;
                a.dec[b] = d;
            }
            atomicOr(a.status, SV_FLAG_BAD_TOKEN);
        }
        return;
    }
    // merge the chunk partials of every row of the request (one warp per row)
    for (int j = warp; j < nr; j += kWarps) {
        const float2 *P = a.partials + static_cast<size_t>(r0 + j) * a.n_chunks;
        if (kSample) {
            float M = -INFINITY, s = 0.f;
            for (int c = lane; c < a.n_chunks; c += 32) {
                const float2 v = __ldcg(P + c);
                ms_merge(M, s, v.x, v.y);
            }
            warp_ms_reduce(M, s);
            if (lane == 0) {
                sh.M[j] = M;
                sh.S[j] = s;
            }
        } else {
            float v = -INFINITY;
            int i = 0x7fffffff;
            for (int c = lane; c < a.n_chunks; c += 32) {
                const float2 w = __ldcg(P + c);
                am_merge(v, i, w.x, __float_as_int(w.y));
            }
            warp_am_reduce(v, i);
            if (lane == 0) sh.arg[j] = i;
        }
    }
    __syncthreads();
    // accept tests at every drafted position; k* = the first rejection
    for (int j = tid; j < Kb; j += kThreads) {
        const int x = a.draft[d0 + j];
        bool acc;
        if (kSample) {
            const float z = logit_at<T>(a, static_cast<size_t>(r0 + j) * a.V + x);
            const float p = exp2f(fmaf(z, a.c, -sh.M[j])) / sh.S[j];
            const float qv = __ldg(a.q + static_cast<size_t>(d0 + j) * a.V + x);
            const float u = __ldg(a.uniforms + r0 + j);
            acc = (u * qv <= p);
            if (a.diag) a.diag[d0 + j] = p;
        } else {
            acc = (x == sh.arg[j]);
        }
        if (!acc) atomicMin(&sh.kstar, j);
    }
    __syncthreads();
    const int ks = sh.kstar;
    for (int j = tid; j < nr; j += kThreads) {
        int v = -1;
        if (j < ks) v = a.draft[d0 + j];
        else if (j == ks && !kSample) v = sh.arg[j];
        a.out_tokens[r0 + j] = v;
    }
    if (tid == 0) {
        a.accept_len[b] = ks + 1;
        if (kSample) {
            Decision d;
            d.row = r0 + ks;
            d.qrow = (ks < Kb) ? d0 + ks : -1;
            d.slot = r0 + ks;
            d.valid = 1;
            d.M = sh.M[ks];
            d.invS = 1.f / sh.S[ks];
            d.u = __ldg(a.uniforms + r0 + Kb);
            d.pad = 0;
            a.dec[b] = d;
        }
    }
}

// ---------------------------------------------------------------------------
// Pass 1: per-(row, chunk) statistics + decide by the request's last CTA
// ---------------------------------------------------------------------------
template <typename T, bool kSample, bool kVecPath>
__global__ void __launch_bounds__(kThreads) stats_decide_kernel(Args a) {
    constexpr int VEC = Elem<T>::kVec;
    constexpr int CHUNK = chunk_elems<T>();
    __shared__ float red_a[kWarps];
    __shared__ int red_b[kWarps];
    __shared__ int s_last;
    __shared__ DecideSmem sh;

    if (a.csr_ok && !__ldcg(a.csr_ok)) return;
    const int tid = threadIdx.x;
    const int item = blockIdx.x;
    const int row = item / a.n_chunks;
    const int chunk = item - row * a.n_chunks;
    const int c0 = chunk * CHUNK;
    const int n = min(CHUNK, a.V - c0);
    const T *zrow = reinterpret_cast<const T *>(a.logits) + static_cast<size_t>(row) * a.V + c0;

    // element (i, k) of this thread is token c0 + (i * kThreads + tid) * VEC + k
    float vals[kLoadsPerThread][VEC];
    if (kVecPath) {
        uint4 raw[kLoadsPerThread];
#pragma unroll
        for (int i = 0; i < kLoadsPerThread; ++i) {
            const int e = (i * kThreads + tid) * VEC;
            if (e < n) raw[i] = ld_stream_u4(zrow + e);
            else raw[i] = make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < kLoadsPerThread; ++i) unpack(raw[i], vals[i]);
    } else {
#pragma unroll
        for (int i = 0; i < kLoadsPerThread; ++i)
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                const int e = (i * kThreads + tid) * VEC + k;
                vals[i][k] = (e < n) ? Elem<T>::at(zrow, e) : 0.f;
            }
    }

    float ra = 0.f;
    int rb = 0;
    if (kSample) {
        float bm = -INFINITY;
#pragma unroll
        for (int i = 0; i < kLoadsPerThread; ++i)
#pragma unroll
            for (int k = 0; k < VEC; ++k)
                if ((i * kThreads + tid) * VEC + k < n) bm = fmaxf(bm, vals[i][k]);
        const float M = bm * a.c;
        float s = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int i = 0; i < kLoadsPerThread; ++i)
#pragma unroll
                for (int k = 0; k < VEC; ++k)
                    if ((i * kThreads + tid) * VEC + k < n) s += ex2(fmaf(vals[i][k], a.c, -M));
        }
        float Mw = M, sw = s;
        warp_ms_reduce(Mw, sw);
        if ((tid & 31) == 0) {
            red_a[tid >> 5] = Mw;
            red_b[tid >> 5] = __float_as_int(sw);
        }
        __syncthreads();
        if (tid < 32) {
            float Mx = (tid < kWarps) ? red_a[tid] : -INFINITY;
            float sx = (tid < kWarps) ? __int_as_float(red_b[tid]) : 0.f;
            warp_ms_reduce(Mx, sx);
            ra = Mx;
            rb = __float_as_int(sx);
        }
    } else {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kLoadsPerThread; ++i)
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                const int e = (i * kThreads + tid) * VEC + k;
                if (e < n && (bi == 0x7fffffff || vals[i][k] > bv)) {
                    bv = vals[i][k];
                    bi = c0 + e;
                }
            }
        warp_am_reduce(bv, bi);
        if ((tid & 31) == 0) {
            red_a[tid >> 5] = bv;
            red_b[tid >> 5] = bi;
        }
        __syncthreads();
        if (tid < 32) {
            float vx = (tid < kWarps) ? red_a[tid] : -INFINITY;
            int ix = (tid < kWarps) ? red_b[tid] : 0x7fffffff;
            warp_am_reduce(vx, ix);
            ra = vx;
            rb = ix;
        }
    }
    if (tid == 0) {
        a.partials[static_cast<size_t>(row) * a.n_chunks + chunk] = make_float2(ra, __int_as_float(rb));
        __threadfence();
        const int b = request_of_row(a, row);
        int r0, nr;
        request_rows(a, b, r0, nr);
        const uint32_t cnt = ticket_arrive(a.tickets1 + b, a.epoch);
        s_last = (cnt == static_cast<uint32_t>(nr) * static_cast<uint32_t>(a.n_chunks)) ? b : -1;
        if (s_last >= 0) a.tickets1[b] = 0ull;  // every other CTA of the request has arrived
    }
    __syncthreads();
    if (s_last >= 0) {
        __threadfence();
        decide<T, kSample>(a, s_last, sh);
    }
}

// ---------------------------------------------------------------------------
// Pass 2: residual masses and the inverse-CDF draw
// ---------------------------------------------------------------------------
struct ScanSmem {
    float warp_tot[kWarps];
    float tile_total;
    int found_tile;
    double found_base;
    double R;
    double t;
    int vbest;
    float rbest;
    int zero_fallback;
};

// r(v) for the 4 tokens tile * 1024 + tid * 4 + k.  Same arithmetic (no
// contraction) wherever it is called, so mass and search passes agree bitwise.
template <typename T, bool kVecPath>
__device__ __forceinline__ void tile_values(const T *zrow, const float *qrow, int V, int tile,
                                            float c, float M, float invS, float (&r)[4]) {
    const int e0 = tile * kTileElems + threadIdx.x * 4;
    float z[4], qv[4] = {0.f, 0.f, 0.f, 0.f};
    if (kVecPath && e0 + 4 <= V) {
        if (sizeof(T) == 4) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(zrow + e0));
            z[0] = v.x; z[1] = v.y; z[2] = v.z; z[3] = v.w;
        } else {
            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(zrow + e0));
            z[0] = __uint_as_float(v.x << 16);
            z[1] = __uint_as_float(v.x & 0xffff0000u);
            z[2] = __uint_as_float(v.y << 16);
            z[3] = __uint_as_float(v.y & 0xffff0000u);
        }
        if (qrow) {
            const float4 w = __ldg(reinterpret_cast<const float4 *>(qrow + e0));
            qv[0] = w.x; qv[1] = w.y; qv[2] = w.z; qv[3] = w.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int e = e0 + k;
            z[k] = (e < V) ? Elem<T>::at(zrow, e) : -INFINITY;
            if (qrow) qv[k] = (e < V) ? __ldg(qrow + e) : 0.f;
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (e0 + k < V) {
            const float p = __fmul_rn(ex2(__fmaf_rn(z[k], c, -M)), invS);
            r[k] = qrow ? fmaxf(__fsub_rn(p, qv[k]), 0.f) : p;
        } else {
            r[k] = 0.f;
        }
    }
}

// Running sums of the tile: e[k] = excl(thread) + (r0 + .. + rk), and the tile
// total (the value e[3] of the last thread).  Deterministic.
__device__ __forceinline__ float tile_scan(const float (&r)[4], float (&e)[4], ScanSmem &sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float pre[4];
    pre[0] = r[0];
    pre[1] = __fadd_rn(pre[0], r[1]);
    pre[2] = __fadd_rn(pre[1], r[2]);
    pre[3] = __fadd_rn(pre[2], r[3]);
    const float s = pre[3];
    float incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl = __fadd_rn(incl, y);
    }
    float lane_excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) lane_excl = 0.f;
    __syncthreads();  // protect warp_tot / tile_total from a previous use
    if (lane == 31) sm.warp_tot[warp] = incl;
    __syncthreads();
    float woff = 0.f;
    for (int w = 0; w < warp; ++w) woff = __fadd_rn(woff, sm.warp_tot[w]);
    const float excl = __fadd_rn(woff, lane_excl);
#pragma unroll
    for (int k = 0; k < 4; ++k) e[k] = __fadd_rn(excl, pre[k]);
    if (tid == kThreads - 1) sm.tile_total = e[3];
    __syncthreads();
    return sm.tile_total;
}

template <typename T, bool kVecPath>
__device__ void draw_final(const Args &a, int b, const Decision &d, ScanSmem &sm) {
    const int tid = threadIdx.x, lane = tid & 31;
    const T *zrow = reinterpret_cast<const T *>(a.logits) + static_cast<size_t>(d.row) * a.V;
    const float *qrow = (d.qrow >= 0) ? a.q + static_cast<size_t>(d.qrow) * a.V : nullptr;
    const float *mass = a.tile_mass + static_cast<size_t>(b) * a.n_tiles;
    if (tid == 0) sm.zero_fallback = 0;

    for (int attempt = 0; attempt < 2; ++attempt) {
        // prefix over tile masses in fp64 (warp 0); lane l owns a contiguous group
        if (tid < 32) {
            const int G = (a.n_tiles + 31) / 32;
            const int i0 = min(lane * G, a.n_tiles), i1 = min(i0 + G, a.n_tiles);
            double sum = 0.0;
            for (int i = i0; i < i1; ++i) sum += static_cast<double>(__ldcg(mass + i));
            double incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const double R = __shfl_sync(0xffffffffu, incl, 31);
            double base = __shfl_up_sync(0xffffffffu, incl, 1);  // exclusive offset of the group
            if (lane == 0) base = 0.0;
            const double t = static_cast<double>(d.u) * R;
            int found = -1;
            double fbase = 0.0, P = base;
            for (int i = i0; i < i1; ++i) {
                const double Pn = P + static_cast<double>(__ldcg(mass + i));
                if (found < 0 && Pn > t) {
                    found = i;
                    fbase = P;
                }
                P = Pn;
            }
            const unsigned ball = __ballot_sync(0xffffffffu, found >= 0);
            const int src = ball ? (__ffs(ball) - 1) : 0;
            const int ft = __shfl_sync(0xffffffffu, found, src);
            const double fb = __shfl_sync(0xffffffffu, fbase, src);
            if (lane == 0) {
                sm.found_tile = ball ? ft : -1;
                sm.found_base = fb;
                sm.R = R;
                sm.t = t;
            }
        }
        __syncthreads();
        if (sm.R > 0.0 || attempt == 1) break;
        // empty residual after a rejection: draw from p instead (recompute masses)
        qrow = nullptr;
        if (tid == 0) {
            sm.zero_fallback = 1;
            atomicOr(a.status, SV_FLAG_ZERO_RESIDUAL);
        }
        float *wmass = a.tile_mass + static_cast<size_t>(b) * a.n_tiles;
        for (int tile = 0; tile < a.n_tiles; ++tile) {
            float r[4], e[4];
            tile_values<T, kVecPath>(zrow, qrow, a.V, tile, a.c, d.M, d.invS, r);
            const float tot = tile_scan(r, e, sm);
            if (tid == 0) wmass[tile] = tot;
        }
        __threadfence_block();
        __syncthreads();
    }

    if (tid == 0) {
        sm.vbest = 0x7fffffff;
        sm.rbest = 0.f;
    }
    __syncthreads();
    const int ft = sm.found_tile;
    if (ft >= 0) {
        float r[4], e[4];
        tile_values<T, kVecPath>(zrow, qrow, a.V, ft, a.c, d.M, d.invS, r);
        tile_scan(r, e, sm);
        const int e0 = ft * kTileElems + tid * 4;
        int cand = 0x7fffffff;
#pragma unroll
        for (int k = 3; k >= 0; --k)
            if (e0 + k < a.V && sm.found_base + static_cast<double>(e[k]) > sm.t) cand = e0 + k;
        if (cand != 0x7fffffff) atomicMin(&sm.vbest, cand);
        __syncthreads();
        if (sm.vbest != 0x7fffffff && sm.vbest >= e0 && sm.vbest < e0 + 4) sm.rbest = r[sm.vbest - e0];
    }
    __syncthreads();
    if (sm.vbest == 0x7fffffff) {
        // rounding left u R above every boundary: the largest token with r > 0
        int last_tile = -1;
        for (int i = a.n_tiles - 1; i >= 0; --i)
            if (__ldcg(mass + i) > 0.f) {
                last_tile = i;
                break;
            }
        if (last_tile >= 0) {
            float r[4];
            tile_values<T, kVecPath>(zrow, qrow, a.V, last_tile, a.c, d.M, d.invS, r);
            const int e0 = last_tile * kTileElems + tid * 4;
            int cand = -1;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (e0 + k < a.V && r[k] > 0.f) cand = e0 + k;
            __shared__ int s_max;
            if (tid == 0) s_max = -1;
            __syncthreads();
            if (cand >= 0) atomicMax(&s_max, cand);
            __syncthreads();
            if (s_max >= e0 && s_max < e0 + 4) {
                sm.vbest = s_max;
                sm.rbest = r[s_max - e0];
            }
        }
        __syncthreads();
    }
    if (tid == 0) {
        const int v = (sm.vbest == 0x7fffffff) ? -1 : sm.vbest;
        a.out_tokens[d.slot] = v;
        if (a.diag) {
            a.diag[a.n_draft + 2 * b] = static_cast<float>(sm.R);
            a.diag[a.n_draft + 2 * b + 1] = static_cast<float>(static_cast<double>(sm.rbest) / sm.R);
        }
    }
}

template <typename T, bool kVecPath>
__global__ void __launch_bounds__(kThreads) residual_kernel(Args a) {
    __shared__ ScanSmem sm;
    __shared__ int s_last;
    if (a.csr_ok && !__ldcg(a.csr_ok)) return;
    const int b = blockIdx.x / a.n_parts;
    const int part = blockIdx.x - b * a.n_parts;
    const Decision d = a.dec[b];
    if (!d.valid) return;
    const T *zrow = reinterpret_cast<const T *>(a.logits) + static_cast<size_t>(d.row) * a.V;
    const float *qrow = (d.qrow >= 0) ? a.q + static_cast<size_t>(d.qrow) * a.V : nullptr;
    const int t0 = part * kTilesPerPart;
    const int t1 = min(t0 + kTilesPerPart, a.n_tiles);
    for (int tile = t0; tile < t1; ++tile) {
        float r[4], e[4];
        tile_values<T, kVecPath>(zrow, qrow, a.V, tile, a.c, d.M, d.invS, r);
        const float tot = tile_scan(r, e, sm);
        if (threadIdx.x == 0) a.tile_mass[static_cast<size_t>(b) * a.n_tiles + tile] = tot;
    }
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t cnt = ticket_arrive(a.tickets2 + b, a.epoch);
        s_last = (cnt == static_cast<uint32_t>(a.n_parts)) ? 1 : 0;
        if (s_last) a.tickets2[b] = 0ull;
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        draw_final<T, kVecPath>(a, b, d, sm);
    }
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
    size_t status, csr_ok, tickets1, tickets2, dec, partials, tile_mass, total;
};

static inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static WsLayout ws_layout(int B, int rows, int V) {
    WsLayout L;
    const size_t n_chunks = (static_cast<size_t>(V) + chunk_elems<float>() - 1) / chunk_elems<float>();
    const size_t n_tiles = (static_cast<size_t>(V) + kTileElems - 1) / kTileElems;
    size_t o = 0;
    L.status = o; o = align256(o + 16);
    L.csr_ok = o; o = align256(o + 16);
    L.tickets1 = o; o = align256(o + 8ull * B);
    L.tickets2 = o; o = align256(o + 8ull * B);
    L.dec = o; o = align256(o + sizeof(Decision) * static_cast<size_t>(B));
    L.partials = o; o = align256(o + sizeof(float2) * static_cast<size_t>(rows) * n_chunks);
    L.tile_mass = o; o = align256(o + sizeof(float) * static_cast<size_t>(B) * n_tiles);
    L.total = o;
    return L;
}

// Call epochs start from a per-process value so that two copies of the
// library, or a workspace holding leftovers, do not share a tag sequence.
static uint32_t initial_epoch() {
    static int anchor;
    uint32_t x = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(&anchor) & 0xffffffffu);
    x ^= static_cast<uint32_t>(std::chrono::steady_clock::now().time_since_epoch().count());
    x ^= static_cast<uint32_t>(getpid()) * 2654435761u;
    return x ? x : 1u;
}
static std::atomic<uint32_t> g_epoch{initial_epoch()};
static void *g_prof_begin = nullptr;
static void *g_prof_end = nullptr;
static thread_local int g_last_launches = 0;

uint32_t next_epoch() {
    uint32_t e = g_epoch.fetch_add(1, std::memory_order_relaxed);
    if (e == 0) e = g_epoch.fetch_add(1, std::memory_order_relaxed);
    return e;
}
void prof_begin(cudaStream_t s) {
    if (g_prof_begin) cudaEventRecord(static_cast<cudaEvent_t>(g_prof_begin), s);
}
void prof_end(cudaStream_t s) {
    if (g_prof_end) cudaEventRecord(static_cast<cudaEvent_t>(g_prof_end), s);
}
void set_launches(int n) { g_last_launches = n; }

template <typename T, bool kSample, bool kVecPath>
static void launch_pass1(const Args &a, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>(a.rows) * static_cast<unsigned>(a.n_chunks);
    stats_decide_kernel<T, kSample, kVecPath><<<grid, kThreads, 0, s>>>(a);
}

template <typename T, bool kVecPath>
static void launch_pass2(const Args &a, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>(a.B) * static_cast<unsigned>(a.n_parts);
    residual_kernel<T, kVecPath><<<grid, kThreads, 0, s>>>(a);
}

template <typename T>
static sv_status run_typed(Args &a, bool sample, bool vec, cudaStream_t s) {
    a.n_chunks = (a.V + chunk_elems<T>() - 1) / chunk_elems<T>();
    int launches = 0;
    if (a.row_offsets) {
        csr_check_kernel<<<1, kThreads, 0, s>>>(a, const_cast<int *>(a.csr_ok));
        ++launches;
    }
    prof_begin(s);
    if (sample) {
        if (vec) launch_pass1<T, true, true>(a, s); else launch_pass1<T, true, false>(a, s);
    } else {
        if (vec) launch_pass1<T, false, true>(a, s); else launch_pass1<T, false, false>(a, s);
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
    a.n_parts = (a.n_tiles + kTilesPerPart - 1) / kTilesPerPart;
    a.n_draft = rows - B;
    a.c = sample ? static_cast<float>(1.4426950408889634 / static_cast<double>(temperature)) : 1.f;
    a.epoch = next_epoch();
    a.status = reinterpret_cast<uint32_t *>(w + L.status);
    a.csr_ok = row_offsets ? reinterpret_cast<const int *>(w + L.csr_ok) : nullptr;
    a.tickets1 = reinterpret_cast<unsigned long long *>(w + L.tickets1);
    a.tickets2 = reinterpret_cast<unsigned long long *>(w + L.tickets2);
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
