// Small vocabularies: one CTA per request (the kernel is described below).
// The same step as the other verification kernels: "Speculative Decoding in
// Large Language Models", section 2 "Modified Rejection Sampling", with the
// stop at the first mismatch and the extra target token of "Co-Designing AI
// Models Using Speculative Decoding", "What is speculative decoding?".
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "../../include/specverify.h"
#include "sv_device.cuh"
#include "sv_draw.cuh"
#include "sv_args.cuh"
#include "sv_host.h"

namespace sv {

// ---------------------------------------------------------------------------
// Small vocabularies: one CTA per request holds all of the request's logits
// rows in shared memory and runs every step on chip (row normalisers, accept
// tests and first-reject scan, residual row, inverse-CDF draw), with no
// cross-CTA records and no polling.  Chosen when the rows of one request
// take at most a set limit (48 KB by default), so that a batch of many small requests
// runs one request per CTA, several CTAs per SM, and a single request is
// one short kernel.
// ---------------------------------------------------------------------------
namespace sk {

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
    return __uint_as_float(static_cast<uint32_t>(__bfloat16_as_ushort(v)) << 16);
}

// Copy n elements of the request's rows into shared memory (16-byte vectors
// when both ends allow, elements otherwise).  A thread issues up to kCopyBatch
// loads before it stores any of them: one round trip instead of one per load.
constexpr int kCopyBatch = 6;  // six loads per thread in flight keep 5 CTAs per SM resident (48 registers)
template <typename T>
__device__ __forceinline__ void load_rows(T *dst, const T *src, size_t n, int tid) {
    const size_t bytes = n * sizeof(T);
    if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0 && (bytes & 15u) == 0) {
        const uint4 *s = reinterpret_cast<const uint4 *>(src);
        uint4 *d = reinterpret_cast<uint4 *>(dst);
        const size_t nv = bytes / 16;
        for (size_t i0 = tid; i0 < nv; i0 += static_cast<size_t>(kThreads) * kCopyBatch) {
            uint4 v[kCopyBatch];
#pragma unroll
            for (int k = 0; k < kCopyBatch; ++k) {
                const size_t i = i0 + static_cast<size_t>(k) * kThreads;
                if (i < nv) v[k] = __ldcs(s + i);
            }
#pragma unroll
            for (int k = 0; k < kCopyBatch; ++k) {
                const size_t i = i0 + static_cast<size_t>(k) * kThreads;
                if (i < nv) d[i] = v[k];
            }
        }
    } else {
        for (size_t i0 = tid; i0 < n; i0 += static_cast<size_t>(kThreads) * kCopyBatch) {
            T v[kCopyBatch];
#pragma unroll
            for (int k = 0; k < kCopyBatch; ++k) {
                const size_t i = i0 + static_cast<size_t>(k) * kThreads;
                if (i < n) v[k] = src[i];
            }
#pragma unroll
            for (int k = 0; k < kCopyBatch; ++k) {
                const size_t i = i0 + static_cast<size_t>(k) * kThreads;
                if (i < n) dst[i] = v[k];
            }
        }
    }
}

template <typename T, bool kSample>
__global__ void __launch_bounds__(kThreads) small_kernel(Args a, int nr_cap) {
    extern __shared__ __align__(16) unsigned char smem[];
    pdl_wait_prior_grid();  // inputs may come from the previous kernel on the stream
    pdl_launch_dependents();
    if (a.csr_ok && !__ldcg(a.csr_ok)) return;
    const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int r0, nr;
    request_rows(a, b, r0, nr);
    const int V = a.V, Kb = nr - 1, d0 = r0 - b;
    T *zs = reinterpret_cast<T *>(smem);
    float2 *st = reinterpret_cast<float2 *>(smem + a16(static_cast<size_t>(nr_cap) * V * sizeof(T)));
    float *rr = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(st) + a16(static_cast<size_t>(nr_cap) * 8));
    DS *ts = reinterpret_cast<DS *>(reinterpret_cast<unsigned char *>(rr) + a16(static_cast<size_t>(V) * 4));
    __shared__ int s_bad, s_ks, s_best;

    // drafts of the first 32 rows: their gathers are in flight during the copy
    int x = 0;
    float qv = 0.f, u = 0.f;
    bool bad = false;
    if (warp == 0) {
        if (lane < Kb) {
            x = __ldg(a.draft + d0 + lane);
            bad = (x < 0 || x >= V);
            if (kSample && !bad) {
                qv = __ldg(a.q + static_cast<size_t>(d0 + lane) * V + x);
                u = __ldg(a.uniforms + r0 + lane);
            }
        }
        for (int j = 32 + lane; j < Kb; j += 32) {
            const int y = __ldg(a.draft + d0 + j);
            bad |= (y < 0 || y >= V);
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) s_bad = bad ? 1 : 0;
    }
    load_rows<T>(zs, reinterpret_cast<const T *>(a.logits) + static_cast<size_t>(r0) * V,
                 static_cast<size_t>(nr) * V, tid);
    __syncthreads();

    // row normalisers: warp w takes rows w, w + 8, ...
    for (int j = warp; j < nr; j += kWarps) {
        const T *row = zs + static_cast<size_t>(j) * V;
        if (kSample) {
            float zmax = -INFINITY;
            for (int v = lane; v < V; v += 32) zmax = fmaxf(zmax, to_f<T>(row[v]));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
            const float M = __fmul_rn(zmax, a.c);  // c > 0: the max of c z
            float s = 0.f;
            for (int v = lane; v < V; v += 32) s += ex2(__fmaf_rn(to_f<T>(row[v]), a.c, -M));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) st[j] = make_float2(M, s);
        } else {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int v = lane; v < V; v += 32) {
                const float zv = to_f<T>(row[v]);
                if (zv > bv) {  // strict: the lowest index of this lane's maxima
                    bv = zv;
                    bi = v;
                }
            }
            warp_am_reduce(bv, bi);
            if (lane == 0) st[j] = make_float2(bv, __int_as_float(bi));
        }
    }
    __syncthreads();

    // accept tests and first-reject scan (warp 0; lane j holds row jb + j)
    if (warp == 0) {
        int ks = -1;
        if (!s_bad) {
            for (int jb = 0; jb < nr && ks < 0; jb += 32) {
                const int j = jb + lane;
                if (jb > 0 && j < Kb) {
                    x = __ldg(a.draft + d0 + j);
                    if (kSample) {
                        qv = __ldg(a.q + static_cast<size_t>(d0 + j) * V + x);
                        u = __ldg(a.uniforms + r0 + j);
                    }
                }
                bool rej = false;
                if (j < Kb) {
                    const float2 sj = st[j];
                    if (kSample) {
                        const float z = to_f<T>(zs[static_cast<size_t>(j) * V + x]);
                        const float p = exp2f(fmaf(z, a.c, -sj.x)) / sj.y;
                        rej = !(u * qv <= p);
                        if (a.diag) a.diag[d0 + j] = p;
                    } else {
                        rej = (x != __float_as_int(sj.y));
                    }
                }
                const unsigned m = __ballot_sync(0xffffffffu, rej);
                if (m) ks = jb + __ffs(m) - 1;
                else if (jb + 32 >= nr) ks = Kb;
            }
        }
        if (s_bad) {
            for (int j = lane; j < nr; j += 32) a.out_tokens[r0 + j] = -1;
            if (lane == 0) {
                a.accept_len[b] = 0;
                atomicOr(a.status, SV_FLAG_BAD_TOKEN);
            }
        } else {
            for (int j = lane; j < nr; j += 32) {
                int v = -1;
                if (j < ks) v = __ldg(a.draft + d0 + j);
                else if (j == ks && !kSample) v = __float_as_int(st[ks].y);
                a.out_tokens[r0 + j] = v;
            }
            if (lane == 0) a.accept_len[b] = ks + 1;
        }
        if (lane == 0) s_ks = s_bad ? -1 : ks;
    }
    __syncthreads();
    if (!kSample || s_ks < 0) return;

    // residual (or bonus) row ks: r(v) into shared memory, each thread a contiguous run of tokens
    const int ks = s_ks;
    const float M = st[ks].x, invS = 1.f / st[ks].y;
    const float *qrow = (ks < Kb) ? a.q + static_cast<size_t>(d0 + ks) * V : nullptr;
    const T *zr = zs + static_cast<size_t>(ks) * V;
    const float uK = __ldg(a.uniforms + r0 + Kb);
    const int L = (V + kThreads - 1) / kThreads;
    const int v0 = min(tid * L, V), v1 = min(v0 + L, V);
    DS P{0.f, 0.f}, incl{0.f, 0.f}, R{0.f, 0.f};
    for (int attempt = 0; attempt < 2; ++attempt) {
        DS sum{0.f, 0.f};
        // the run's q values are fetched kCopyBatch at a time ahead of their use
        for (int vb = v0; vb < v1; vb += kCopyBatch) {
            float qv[kCopyBatch];
#pragma unroll
            for (int k = 0; k < kCopyBatch; ++k) qv[k] = (qrow && vb + k < v1) ? __ldg(qrow + vb + k) : 0.f;
#pragma unroll
            for (int k = 0; k < kCopyBatch; ++k) {
                const int v = vb + k;
                if (v < v1) {
                    const float p = __fmul_rn(ex2(__fmaf_rn(to_f<T>(zr[v]), a.c, -M)), invS);
                    const float r = qrow ? fmaxf(__fsub_rn(p, qv[k]), 0.f) : p;
                    rr[v] = r;
                    sum = ds_add_f(sum, r);
                }
            }
        }
        // block-wide inclusive scan of the per-thread sums (double-single)
        incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const DS y = ds_shfl_up(incl, o);
            if (lane >= o) incl = ds_add(incl, y);
        }
        if (lane == 31) ts[warp] = incl;
        __syncthreads();
        DS wpre{0.f, 0.f};
        for (int w = 0; w < warp; ++w) wpre = ds_add(wpre, ts[w]);
        R = ts[0];
        for (int w = 1; w < kWarps; ++w) R = ds_add(R, ts[w]);
        incl = ds_add(wpre, incl);
        P = ds_add(incl, DS{-sum.hi, -sum.lo});
        __syncthreads();
        if (R.hi > 0.f || attempt == 1) break;
        // empty residual after a rejection: draw from p instead
        qrow = nullptr;
        if (tid == 0) atomicOr(a.status, SV_FLAG_ZERO_RESIDUAL);
    }
    const DS t = ds_mul_f(R, uK);
    // the first thread whose run holds u R scans it in token order
    if (tid == 0) s_best = 0x7fffffff;
    __syncthreads();
    const bool holds = v0 < v1 && ds_gt(incl, t) && !ds_gt(P, t);
    if (holds) atomicMin(&s_best, tid);
    __syncthreads();
    const int owner = s_best;
    __syncthreads();
    if (tid == 0) s_best = 0x7fffffff;  // reused below: the drawn token
    __syncthreads();
    if (tid == owner) {
        DS run = P;
        int vs = -1;
        for (int v = v0; v < v1; ++v) {
            run = ds_add_f(run, rr[v]);
            if (ds_gt(run, t)) {
                vs = v;
                break;
            }
        }
        s_best = vs >= 0 ? vs : -(v1 + 1);  // < 0: the sums ended short of u R at v1
    }
    __syncthreads();
    int vstar = s_best;  // >= 0 drawn; < 0 the owner's sums ended short; 0x7fffffff no owner
    __syncthreads();
    if (vstar < 0) {
        // rounding: the next token with r > 0 after the owner's run
        const int from = -(vstar + 1);
        if (tid == 0) s_best = 0x7fffffff;
        __syncthreads();
        for (int v = max(v0, from); v < v1; ++v)
            if (rr[v] > 0.f) {
                atomicMin(&s_best, v);
                break;
            }
        __syncthreads();
        vstar = s_best;
        __syncthreads();
    }
    if (vstar == 0x7fffffff) {
        // u R at or above every boundary: the last token with r > 0
        if (tid == 0) s_best = -1;
        __syncthreads();
        for (int v = v1 - 1; v >= v0; --v)
            if (rr[v] > 0.f) {
                atomicMax(&s_best, v);
                break;
            }
        __syncthreads();
        vstar = s_best;
    }
    if (tid == 0) {
        a.out_tokens[r0 + ks] = vstar;
        if (a.diag) {
            const float Rf = __fadd_rn(R.hi, R.lo);
            a.diag[a.n_draft + 2 * b] = Rf;
            a.diag[a.n_draft + 2 * b + 1] = vstar >= 0 ? __fdiv_rn(rr[vstar], Rf) : 0.f;
        }
    }
}

}  // namespace sk

// One CTA per request, the request's rows in shared memory (sk::small_kernel).
template <typename T, bool kSample>
static cudaError_t launch_small(const Args &a, int nr_cap, cudaStream_t s) {
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!configured[dev]) {
        cudaFuncSetAttribute(sk::small_kernel<T, kSample>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sk::kMaxSmemBytes));
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.B);
    cfg.blockDim = dim3(sk::kThreads);
    cfg.dynamicSmemBytes = sk::smem_bytes(nr_cap, a.V, sizeof(T));
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sk::small_kernel<T, kSample>, a, nr_cap);
}

cudaError_t launch_small_kernel(const Args &a, int nr_cap, bool sample, bool bf16, cudaStream_t s) {
    if (bf16) return sample ? launch_small<__nv_bfloat16, true>(a, nr_cap, s) : launch_small<__nv_bfloat16, false>(a, nr_cap, s);
    return sample ? launch_small<float, true>(a, nr_cap, s) : launch_small<float, false>(a, nr_cap, s);
}

}  // namespace sv
