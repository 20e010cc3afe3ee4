// Device helpers shared by the final draws of the verifier kernels and the
// draft sampler: double-single prefix sums, the 256-token segment loader and
// the in-segment running-sum scan.
#pragma once

#include <cstdint>

#include "sv_device.cuh"

namespace sv {

// Row partials: (M, S) of an online softmax (sampling) or (max, argmax) (greedy).
template <bool kSample>
__device__ __forceinline__ void partial_identity(float &ra, int &rb) {
    ra = -INFINITY;
    rb = kSample ? __float_as_int(0.f) : 0x7fffffff;
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

struct TileScan {
    int v;       // found token (kFind) or -1
    float rv;    // its r(v)
    float mass;  // tile mass
};

// r(v) of the 8 tokens a lane holds in 256-token segment g of a row: token
// g * 256 + (j * 32 + lane) * 4 + k, j < 2, k < 4; zero beyond V.  Same
// arithmetic as res_lane_sum (V is a multiple of 4 on this path).
template <typename T>
__device__ __forceinline__ void seg_load_r(const T *zrow, const float *qrow, int V, int g, float c, float M,
                                           float invS, int lane, float (&r)[2][4]) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int e0 = g * kSegElems + (j * 32 + lane) * 4;
        float z[4] = {0.f, 0.f, 0.f, 0.f}, qv[4] = {0.f, 0.f, 0.f, 0.f};
        const bool in = e0 < V;
        if (in) {
            if constexpr (sizeof(T) == 4) {
                const float4 w = __ldcs(reinterpret_cast<const float4 *>(zrow + e0));
                z[0] = w.x; z[1] = w.y; z[2] = w.z; z[3] = w.w;
            } else {
                const uint2 w = __ldcs(reinterpret_cast<const uint2 *>(zrow + e0));
                z[0] = __uint_as_float(w.x << 16);
                z[1] = __uint_as_float(w.x & 0xffff0000u);
                z[2] = __uint_as_float(w.y << 16);
                z[3] = __uint_as_float(w.y & 0xffff0000u);
            }
            if (qrow) {
                const float4 w = __ldcs(reinterpret_cast<const float4 *>(qrow + e0));
                qv[0] = w.x; qv[1] = w.y; qv[2] = w.z; qv[3] = w.w;
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float p = __fmul_rn(ex2(__fmaf_rn(z[k], c, -M)), invS);
            r[j][k] = in ? (qrow ? fmaxf(__fsub_rn(p, qv[k]), 0.f) : p) : 0.f;
        }
    }
}

// Double-single arithmetic: an unevaluated sum hi + lo of two fp32 values
// (about 48 significant bits), from error-free transformations (Knuth's
// TwoSum; the product error from one fma).  FP64 runs at a small fraction of
// the fp32 rate on this GPU, and the draw's prefix sums sit on the critical
// path, so they are kept in this form instead.
struct DS {
    float hi, lo;
};
__device__ __forceinline__ DS ds_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return DS{s, e};
}
__device__ __forceinline__ DS ds_norm(float s, float e) {
    const float hi = __fadd_rn(s, e);
    return DS{hi, __fsub_rn(e, __fsub_rn(hi, s))};
}
__device__ __forceinline__ DS ds_add(DS a, DS b) {
    const DS t = ds_two_sum(a.hi, b.hi);
    return ds_norm(t.hi, __fadd_rn(t.lo, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ DS ds_add_f(DS a, float b) {
    const DS t = ds_two_sum(a.hi, b);
    return ds_norm(t.hi, __fadd_rn(t.lo, a.lo));
}
__device__ __forceinline__ DS ds_mul_f(DS a, float b) {
    const float p = __fmul_rn(a.hi, b);
    const float e = __fmaf_rn(a.lo, b, __fmaf_rn(a.hi, b, -p));
    return ds_norm(p, e);
}
// a > b
__device__ __forceinline__ bool ds_gt(DS a, DS b) {
    const DS d = ds_add(a, DS{-b.hi, -b.lo});
    return d.hi > 0.f || (d.hi == 0.f && d.lo > 0.f);
}
__device__ __forceinline__ DS ds_shfl_up(DS a, int o) {
    return DS{__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ DS ds_shfl(DS a, int src) {
    return DS{__shfl_sync(0xffffffffu, a.hi, src), __shfl_sync(0xffffffffu, a.lo, src)};
}

// Running sums of a segment in token order (fp32 within the segment, on top
// of the double-single prefix base_p of the segments before it): the first
// token whose running sum passes t, or -1.
__device__ __forceinline__ TileScan warp_seg_scan(const float (&r)[2][4], int g, int V, DS base_p, DS t, int lane) {
    float base = 0.f;
    TileScan res{-1, 0.f, 0.f};
    // base_p + x > t is tested as x > t - base_p, formed once per segment
    const DS d = ds_add(t, DS{-base_p.hi, -base_p.lo});
#pragma unroll
    for (int j = 0; j < 2; ++j) {
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
        int cand = -1;
        const int e0 = g * kSegElems + (j * 32 + lane) * 4;
#pragma unroll
        for (int k = 3; k >= 0; --k)
            if (e0 + k < V && ds_gt(DS{__fadd_rn(head, pre[k]), 0.f}, d)) cand = k;
        const unsigned m = __ballot_sync(0xffffffffu, cand >= 0);
        if (m && res.v < 0) {
            const int src = __ffs(m) - 1;
            const int ck = __shfl_sync(0xffffffffu, cand, src);
            float rsel = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (k == ck) rsel = r[j][k];
            res.v = g * kSegElems + (j * 32 + src) * 4 + ck;
            res.rv = __shfl_sync(0xffffffffu, rsel, src);
        }
        base = __fadd_rn(base, seg);
    }
    return res;
}

// Sum of a segment's r(v) in a fixed order (the slow path below uses it twice).
__device__ __forceinline__ float seg_sum(const float (&r)[2][4]) {
    float m = ((r[0][0] + r[0][1]) + (r[0][2] + r[0][3])) + ((r[1][0] + r[1][1]) + (r[1][2] + r[1][3]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m += __shfl_xor_sync(0xffffffffu, m, o);
    return m;
}

}  // namespace sv
