// Medium requests in small batches: one cluster of CTAs per request (the
// kernel is described below).  The same step as the other verification
// kernels: "Speculative Decoding in Large Language Models", section 2
// "Modified Rejection Sampling", with the stop at the first mismatch and the
// extra target token of "Co-Designing AI Models Using Speculative Decoding",
// "What is speculative decoding?".
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "../../include/specverify.h"
#include "sv_device.cuh"
#include "sv_draw.cuh"
#include "sv_args.cuh"
#include "sv_host.h"
#include "sv_slice.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// Medium requests: one cluster of kC CTAs per request (up to a few hundred KB
// of logits per request, batches of at most two clusters per SM pair).  Each
// CTA copies its contiguous slice of 256-token segments of every row of the
// request into shared memory with bulk copies, reduces each row over its
// slice (max and sum of exponentials, or argmax) and sends the row partials
// to every CTA of the cluster with remote stores.  After a cluster barrier
// every CTA merges the kC partials of each row in rank order (the same
// normalisers everywhere) and runs the accept tests and the first-reject
// scan.  The draw then follows the same slice-total scheme as the LM-head
// finish: r over the CTA's slice of the selected row (z from shared memory,
// q from global memory), segment sums, slice totals to every CTA, one more
// cluster barrier, and the CTA whose slice holds u R draws.  No CTA reads
// another CTA's shared memory.
// ---------------------------------------------------------------------------
namespace cv {

template <typename T, bool kSample>
__global__ void __launch_bounds__(kThreads, 2) cluster_kernel(Args a) {
    extern __shared__ __align__(128) unsigned char cv_smem[];
    __shared__ uint64_t s_bar;
    __shared__ float2 s_wpart[kWarps];      // each warp's partial of its part of a row
    __shared__ float2 s_cta[kC][kMaxRows];  // row partials of every CTA of the cluster (remote stores)
    __shared__ float2 s_row[kMaxRows];      // merged row normalisers
    __shared__ int s_x[kMaxRows];
    __shared__ float s_z[kMaxRows], s_q[kMaxRows], s_u[kMaxRows];
    __shared__ float s_seg[kMaxSegs];
    __shared__ float2 s_tot[2][kC];         // slice totals (double-single), remote stores
    __shared__ int s_ks, s_retry;

    const uint32_t rank = cluster_ctarank();
    const int b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    cluster_arrive_relaxed();  // waited on before the first remote store
    pdl_wait_prior_grid();  // the logits may come from the previous kernel on the stream
    pdl_launch_dependents();
    if (a.csr_ok && !__ldcg(a.csr_ok)) return;  // the same word for every CTA: the cluster leaves together
    int r0, nr;
    request_rows(a, b, r0, nr);
    const int V = a.V, Kb = nr - 1, d0 = r0 - b;
    const int nsp = segs_per_cta(V), ns = (V + kSegElems - 1) / kSegElems;
    const int seg0 = min(static_cast<int>(rank) * nsp, ns), seg1 = min(seg0 + nsp, ns), nloc = seg1 - seg0;
    const int t0 = seg0 * kSegElems, nt = min(seg1 * kSegElems, V) - t0;
    const T *logits = reinterpret_cast<const T *>(a.logits);
    T *zs = reinterpret_cast<T *>(cv_smem);  // row j's slice at zs + j * nsp * 256
    const int slice = nsp * kSegElems;

    // this CTA's slice of every row of the request
    if (tid == 0 && nt > 0) {
        const uint32_t bytes = static_cast<uint32_t>(nt) * sizeof(T);
        mbar_arrive_expect_tx(&s_bar, bytes * static_cast<uint32_t>(nr));
        for (int j = 0; j < nr; ++j)
            bulk_g2s(zs + static_cast<size_t>(j) * slice, logits + static_cast<size_t>(r0 + j) * V + t0, bytes, &s_bar);
    }
    // accept-test operands of draft j = tid, gathered while the copies land
    int xj = -1;
    float zj = 0.f, qj = 0.f, uj = 0.f;
    if (tid < Kb) {
        xj = __ldg(a.draft + d0 + tid);
        if (xj < 0 || xj >= V) {
            xj = -1;
        } else if (kSample) {
            float z4[4];
            const int x4 = xj & ~3;
            load4<T>(logits + static_cast<size_t>(r0 + tid) * V + x4, z4);
            zj = z4[xj - x4];
            qj = __ldg(a.q + static_cast<size_t>(d0 + tid) * V + xj);
            uj = __ldg(a.uniforms + r0 + tid);
        }
        s_x[tid] = xj;
        s_z[tid] = zj;
        s_q[tid] = qj;
        s_u[tid] = uj;
    }
    if (nt > 0 && !mbar_wait_bounded(&s_bar, 0, kDrainBudget) && tid == 0) atomicOr(a.status, SV_FLAG_TIMEOUT);

    // row partials over the slice: row j takes warps [j wpr, (j + 1) wpr), each a part in token order
    const int wpr = nr <= kWarps ? kWarps / nr : 1;
    {
        const int j = warp / wpr, part = warp - j * wpr;
        float ra;
        int rb;
        partial_identity<kSample>(ra, rb);
        if (j < nr) {
            const int nq = nt >> 2;  // 4-token groups of the slice
            const int q0 = (nq * part) / wpr, q1 = (nq * (part + 1)) / wpr;
            const T *row = zs + static_cast<size_t>(j) * slice;
            // four independent accumulators (one per position within a 4-token group) and
            // several groups' loads in flight: the loops are latency-bound otherwise
            if (kSample) {
                float zm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 4
                for (int i = q0 + lane; i < q1; i += 32) {
                    float z[4];
                    load4<T>(row + 4 * i, z);
#pragma unroll
                    for (int k = 0; k < 4; ++k) zm[k] = fmaxf(zm[k], z[k]);
                }
                float zmax = fmaxf(fmaxf(zm[0], zm[1]), fmaxf(zm[2], zm[3]));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
                if (zmax != -INFINITY) {
                    const float Mw = __fmul_rn(zmax, a.c);  // c > 0: the max of c z
                    float sk[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                    for (int i = q0 + lane; i < q1; i += 32) {
                        float z[4];
                        load4<T>(row + 4 * i, z);
#pragma unroll
                        for (int k = 0; k < 4; ++k) sk[k] += ex2(__fmaf_rn(z[k], a.c, -Mw));
                    }
                    float s = (sk[0] + sk[1]) + (sk[2] + sk[3]);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                    ra = Mw;
                    rb = __float_as_int(s);
                }
            } else {
                float bv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                int bi[4] = {0x7fffffff, 0x7fffffff, 0x7fffffff, 0x7fffffff};
#pragma unroll 4
                for (int i = q0 + lane; i < q1; i += 32) {
                    float z[4];
                    load4<T>(row + 4 * i, z);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (z[k] > bv[k]) {  // strict: each stream keeps the lowest index of its maxima
                            bv[k] = z[k];
                            bi[k] = t0 + 4 * i + k;
                        }
                }
#pragma unroll
                for (int k = 1; k < 4; ++k) am_merge(bv[0], bi[0], bv[k], bi[k]);  // lower index on equal values
                warp_am_reduce(bv[0], bi[0]);
                ra = bv[0];
                rb = bi[0];
            }
        }
        if (lane == 0) s_wpart[warp] = make_float2(ra, __int_as_float(rb));
    }
    __syncthreads();
    // this CTA's partial of row j (its warps in order) to every CTA of the cluster, all of them running
    cluster_wait();
    if (tid < nr) {
        float ra;
        int rb;
        partial_identity<kSample>(ra, rb);
        if (tid < kWarps)
            for (int p = 0; p < wpr; ++p) merge_pair<kSample>(ra, rb, s_wpart[tid * wpr + p]);
#pragma unroll
        for (int k = 0; k < kC; ++k) st_dsmem_f32x2(&s_cta[rank][tid], ra, __int_as_float(rb), static_cast<uint32_t>(k));
    }
    cluster_sync();
    if (tid < nr) {
        float ra;
        int rb;
        partial_identity<kSample>(ra, rb);
#pragma unroll
        for (int k = 0; k < kC; ++k) merge_pair<kSample>(ra, rb, s_cta[k][tid]);
        s_row[tid] = make_float2(ra, __int_as_float(rb));
    }
    __syncthreads();

    // accept tests and first-reject scan (warp 0 of every CTA; rank 0 writes the outputs)
    if (warp == 0) {
        bool bad = false;
        for (int j = lane; j < Kb; j += 32) bad |= s_x[j] < 0;
        bad = __any_sync(0xffffffffu, bad);
        int ks = -1;
        for (int jb = 0; !bad && jb < nr && ks < 0; jb += 32) {
            const int j = jb + lane;
            bool rej = false;
            if (j < Kb) {
                const float2 sj = s_row[j];
                if (kSample) {
                    const float p = exp2f(fmaf(s_z[j], a.c, -sj.x)) / sj.y;
                    rej = !(s_u[j] * s_q[j] <= p);
                    if (a.diag && rank == 0) a.diag[d0 + j] = p;
                } else {
                    rej = (s_x[j] != __float_as_int(sj.y));
                }
            }
            const unsigned m = __ballot_sync(0xffffffffu, rej);
            if (m) ks = jb + __ffs(m) - 1;
            else if (jb + 32 >= nr) ks = Kb;
        }
        if (rank == 0) {
            if (bad) {
                for (int j = lane; j < nr; j += 32) a.out_tokens[r0 + j] = -1;
                if (lane == 0) {
                    a.accept_len[b] = 0;
                    atomicOr(a.status, SV_FLAG_BAD_TOKEN);
                }
            } else {
                for (int j = lane; j < nr; j += 32) {
                    int v = -1;
                    if (j < ks) v = s_x[j];
                    else if (j == ks && !kSample) v = __float_as_int(s_row[ks].y);
                    a.out_tokens[r0 + j] = v;
                }
                if (lane == 0) a.accept_len[b] = ks + 1;
            }
        }
        if (lane == 0) s_ks = bad ? -1 : ks;
    }
    __syncthreads();
    // every CTA of the cluster has the same ks: leaving together touches no other CTA's memory
    if (!kSample || s_ks < 0) return;

    const int ks = s_ks;
    const float M = s_row[ks].x, invS = 1.f / s_row[ks].y;
    const T *zsl = zs + static_cast<size_t>(ks) * slice;               // the selected row's slice
    const T *zrow = logits + static_cast<size_t>(r0 + ks) * V;         // and the whole row (fallbacks)
    const float *qrow0 = (ks < Kb) ? a.q + static_cast<size_t>(d0 + ks) * V : nullptr;
    float *gseg = a.cv_segs + static_cast<size_t>(b) * ns;
    // warp 0's share of the local segments and its exclusive prefix within the slice
    const int G = (nloc + 31) / 32;
    const int i0 = min(lane * G, nloc), i1 = min(i0 + G, nloc);
    DS excl{0.f, 0.f};
    int attempt = 0;
    const float *qrow = qrow0;
    for (;; ++attempt) {
        qrow = (attempt == 0) ? qrow0 : nullptr;
        // r over this CTA's segments; a warp's q loads for kQBatch segments are in flight together
        for (int gb = warp; gb < nloc; gb += kQBatch * kWarps) {
            float4 qb[kQBatch][2];
#pragma unroll
            for (int i = 0; i < kQBatch; ++i) {
                const int gl = gb + i * kWarps;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int e = (seg0 + gl) * kSegElems + (j * 32 + lane) * 4;
                    qb[i][j] = (gl < nloc && qrow && e < V) ? __ldg(reinterpret_cast<const float4 *>(qrow + e))
                                                              : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int i = 0; i < kQBatch; ++i) {
                const int gl = gb + i * kWarps;
                if (gl >= nloc) continue;
                const int g = seg0 + gl;
                float r[2][4];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int o = (j * 32 + lane) * 4;
                    const bool in = g * kSegElems + o < V;
                    float z[4] = {0.f, 0.f, 0.f, 0.f};
                    if (in) load4<T>(zsl + gl * kSegElems + o, z);
                    const float qv[4] = {qb[i][j].x, qb[i][j].y, qb[i][j].z, qb[i][j].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float p = __fmul_rn(ex2(__fmaf_rn(z[k], a.c, -M)), invS);
                        r[j][k] = in ? (qrow ? fmaxf(__fsub_rn(p, qv[k]), 0.f) : p) : 0.f;
                    }
                }
                const float s = seg_sum(r);
                if (lane == 0) {
                    s_seg[gl] = s;
                    gseg[g] = s;
                }
            }
        }
        __syncthreads();
        // the slice total, in a fixed order, to every CTA of the cluster
        if (warp == 0) {
            DS sum{0.f, 0.f};
            for (int i = i0; i < i1; ++i) sum = ds_add_f(sum, s_seg[i]);
            DS incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const DS y = ds_shfl_up(incl, o);
                if (lane >= o) incl = ds_add(incl, y);
            }
            excl = ds_shfl_up(incl, 1);
            if (lane == 0) excl = DS{0.f, 0.f};
            const DS tot = ds_shfl(incl, 31);
            if (lane < kC) st_dsmem_f32x2(&s_tot[attempt][rank], tot.hi, tot.lo, static_cast<uint32_t>(lane));
        }
        cluster_sync();
        // the same totals in the same order in every CTA: an empty residual is seen by all of them
        if (attempt == 0 && qrow0 != nullptr) {
            if (tid == 0) {
                DS R{0.f, 0.f};
                for (int k = 0; k < kC; ++k) R = ds_add(R, DS{s_tot[0][k].x, s_tot[0][k].y});
                s_retry = R.hi > 0.f ? 0 : 1;
            }
            __syncthreads();
            if (s_retry) {
                if (rank == 0 && tid == 0) atomicOr(a.status, SV_FLAG_ZERO_RESIDUAL);  // draw from p
                continue;
            }
        }
        break;
    }
    if (warp != 0) return;

    // prefix of the slice totals, R, u R and the CTA whose slice holds u R
    const float u = __ldg(a.uniforms + r0 + Kb);
    DS P{0.f, 0.f}, Pmine{0.f, 0.f};
    DS Pk[kC + 1];
    Pk[0] = P;
#pragma unroll
    for (int k = 0; k < kC; ++k) {
        P = ds_add(P, DS{s_tot[attempt][k].x, s_tot[attempt][k].y});
        Pk[k + 1] = P;
    }
    const DS R = P;
    const DS t = ds_mul_f(R, u);
    int owner = -1, last_pos = -1;
#pragma unroll
    for (int k = kC - 1; k >= 0; --k) {
        if (ds_gt(Pk[k + 1], t)) owner = k;
        if (last_pos < 0 && s_tot[attempt][k].x > 0.f) last_pos = k;
    }
#pragma unroll
    for (int k = 0; k < kC; ++k)
        if (k == static_cast<int>(rank)) Pmine = Pk[k];
    const bool past_end = owner < 0;  // u R at or above every boundary: the last r > 0
    if (past_end) owner = last_pos < 0 ? 0 : last_pos;
    if (owner != static_cast<int>(rank)) return;

    int vstar = -1;
    float rstar = 0.f;
    if (!past_end) {
        // the first local segment whose running sum passes u R
        DS Pl = ds_add(Pmine, excl);
        int found = -1;
        DS fb{0.f, 0.f};
        for (int i = i0; i < i1; ++i) {
            const DS Pn = ds_add_f(Pl, s_seg[i]);
            if (found < 0 && ds_gt(Pn, t)) {
                found = i;
                fb = Pl;
            }
            Pl = Pn;
        }
        const unsigned ball = __ballot_sync(0xffffffffu, found >= 0);
        int next = seg1;  // sums short of u R: the next r > 0 after the slice
        if (ball) {
            const int src = __ffs(ball) - 1;
            const int gl = __shfl_sync(0xffffffffu, found, src);
            const int fseg = seg0 + gl;
            const DS fbase = ds_shfl(fb, src);
            float r[2][4];
            seg_r<T>(zsl + gl * kSegElems, qrow ? qrow + static_cast<size_t>(fseg) * kSegElems : nullptr, fseg, V,
                     a.c, M, invS, lane, r);
            const TileScan ts = warp_seg_scan(r, fseg, V, fbase, t, lane);
            vstar = ts.v;
            rstar = ts.rv;
            next = fseg + 1;
        }
        if (vstar < 0)
            vstar = find_positive<T, true>(zrow, qrow, V, ns, a.c, M, invS, s_seg, gseg, seg0, seg1, next, lane,
                                           &rstar);
    }
    if (vstar < 0)
        vstar = find_positive<T, false>(zrow, qrow, V, ns, a.c, M, invS, s_seg, gseg, seg0, seg1, ns - 1, lane,
                                        &rstar);
    if (lane == 0) {
        a.out_tokens[r0 + ks] = vstar;
        if (a.diag) {
            const float Rf = __fadd_rn(R.hi, R.lo);
            a.diag[a.n_draft + 2 * b] = Rf;
            a.diag[a.n_draft + 2 * b + 1] = vstar >= 0 ? __fdiv_rn(rstar, Rf) : 0.f;
        }
    }
}

}  // namespace cv

template <typename T, bool kSample>
static cudaError_t launch_cluster(const Args &a, int nr_cap, cudaStream_t s) {
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!configured[dev]) {
        cudaFuncSetAttribute(cv::cluster_kernel<T, kSample>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(cv::kSmemCap));
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cv::kC, static_cast<unsigned>(a.B));
    cfg.blockDim = dim3(cv::kThreads);
    cfg.dynamicSmemBytes = cv::smem_bytes(nr_cap, a.V, static_cast<int>(sizeof(T)));
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cv::kC;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, cv::cluster_kernel<T, kSample>, a);
}

cudaError_t launch_cluster_kernel(const Args &a, int nr_cap, bool sample, bool bf16, cudaStream_t s) {
    if (bf16) return sample ? launch_cluster<__nv_bfloat16, true>(a, nr_cap, s) : launch_cluster<__nv_bfloat16, false>(a, nr_cap, s);
    return sample ? launch_cluster<float, true>(a, nr_cap, s) : launch_cluster<float, false>(a, nr_cap, s);
}

}  // namespace sv
