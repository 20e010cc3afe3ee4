// Per-segment helpers shared by the kernels that split a request's vocabulary
// into per-CTA slices of 256-token segments (cluster.cu, lmhead.cu): r over
// one segment, a segment's mass, and the warp-wide searches for the next or
// last token with r > 0 that the draw's rounding fallbacks use.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "sv_device.cuh"

namespace sv {

// Four consecutive logits (16-byte vectors of fp32, 8-byte of bf16) as floats.
template <typename T>
__device__ __forceinline__ void load4(const T *p, float (&z)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float *p, float (&z)[4]) {
    const float4 w = *reinterpret_cast<const float4 *>(p);
    z[0] = w.x; z[1] = w.y; z[2] = w.z; z[3] = w.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16 *p, float (&z)[4]) {
    const uint2 w = *reinterpret_cast<const uint2 *>(p);
    z[0] = __uint_as_float(w.x << 16);
    z[1] = __uint_as_float(w.x & 0xffff0000u);
    z[2] = __uint_as_float(w.y << 16);
    z[3] = __uint_as_float(w.y & 0xffff0000u);
}

// r(v) of the 8 tokens a lane holds in 256-token segment g (token g * 256 +
// (j * 32 + lane) * 4 + k): zseg points at the segment's first logit (in
// shared or global memory), qseg at its q values or nullptr (r = p).
template <typename T>
__device__ __forceinline__ void seg_r(const T *zseg, const float *qseg, int g, int V, float c, float M, float invS,
                                      int lane, float (&r)[2][4]) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int o = (j * 32 + lane) * 4;
        const bool in = g * kSegElems + o < V;
        float z[4] = {0.f, 0.f, 0.f, 0.f}, qv[4] = {0.f, 0.f, 0.f, 0.f};
        if (in) {
            load4<T>(zseg + o, z);
            if (qseg) {
                const float4 w = __ldg(reinterpret_cast<const float4 *>(qseg + o));
                qv[0] = w.x; qv[1] = w.y; qv[2] = w.z; qv[3] = w.w;
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float p = __fmul_rn(ex2(__fmaf_rn(z[k], c, -M)), invS);
            r[j][k] = in ? (qseg ? fmaxf(__fsub_rn(p, qv[k]), 0.f) : p) : 0.f;
        }
    }
}

// Segment g's mass: this CTA's own segments from shared memory, the others'
// from the global scratch row (written before the cluster barrier).
__device__ __forceinline__ float seg_mass(const float *s_seg, const float *gseg, int g, int seg0, int seg1) {
    return (g >= seg0 && g < seg1) ? s_seg[g - seg0] : __ldcg(gseg + g);
}

// First token with r > 0 at or after segment g0 (forward) or the last at or
// before it (backward), its r in *rv; -1 if none.  Warp-wide, 32 segment
// masses per step, r recomputed from the global rows.
template <typename T, bool kForward>
__device__ int find_positive(const T *zrow, const float *qrow, int V, int ns, float c, float M, float invS,
                             const float *s_seg, const float *gseg, int seg0, int seg1, int g0, int lane, float *rv) {
    for (int base = g0; kForward ? base < ns : base >= 0; base += kForward ? 32 : -32) {
        const int g = kForward ? base + lane : base - lane;
        const bool has = (kForward ? g < ns : g >= 0) && seg_mass(s_seg, gseg, g, seg0, seg1) > 0.f;
        const unsigned m = __ballot_sync(0xffffffffu, has);
        if (!m) continue;
        const int gs = __shfl_sync(0xffffffffu, g, __ffs(m) - 1);
        float r[2][4];
        seg_r<T>(zrow + static_cast<size_t>(gs) * kSegElems, qrow ? qrow + static_cast<size_t>(gs) * kSegElems : nullptr,
                 gs, V, c, M, invS, lane, r);
        int loc = kForward ? 0x7fffffff : -1;
        float rloc = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int jj = kForward ? 1 - j : j, kk = kForward ? 3 - k : k;  // keep the extreme one
                if (r[jj][kk] > 0.f) {
                    loc = (jj * 32 + lane) * 4 + kk;
                    rloc = r[jj][kk];
                }
            }
        const int best = kForward ? __reduce_min_sync(0xffffffffu, loc) : __reduce_max_sync(0xffffffffu, loc);
        if (kForward ? best == 0x7fffffff : best < 0) continue;  // a positive sum of nothing: cannot happen
        const unsigned mm = __ballot_sync(0xffffffffu, loc == best);
        *rv = __shfl_sync(0xffffffffu, rloc, __ffs(mm) - 1);
        return gs * kSegElems + best;
    }
    return -1;
}

}  // namespace sv
