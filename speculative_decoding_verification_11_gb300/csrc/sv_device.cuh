// Device helpers shared by the verification kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr int kThreads = 256;          // every verification kernel runs 8 warps
constexpr int kWarps = kThreads / 32;
constexpr int kLoadsPerThread = 8;     // 16-byte loads in flight per thread per chunk
constexpr int kTileElems = kThreads * 4;  // residual tile: 4 tokens per thread
constexpr int kTilesPerPart = 8;          // residual CTA covers 8 tiles
constexpr int kMaxRowsPerRequest = 256;   // SV_MAX_K + 1

// Elements per 16-byte vector and per stats chunk for each logits type.
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kVec = 4;
    static __device__ __forceinline__ float at(const float *p, size_t i) { return __ldg(p + i); }
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
    static __device__ __forceinline__ float at(const __nv_bfloat16 *p, size_t i) {
        const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(p) + i);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
};
template <typename T> __host__ __device__ constexpr int chunk_elems() { return kThreads * kLoadsPerThread * Elem<T>::kVec; }

// 2^x on the MUFU unit (flushes subnormal results to zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 128-bit streaming load that does not allocate in L1 (each logit is read once).
__device__ __forceinline__ uint4 ld_stream_u4(const void *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// Unpack a 16-byte vector into floats.
__device__ __forceinline__ void unpack(const uint4 &v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack(const uint4 &v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// (M, s) represents sum_i 2^(y_i - M).  Merge two such pairs.
__device__ __forceinline__ void ms_merge(float &M, float &s, float M2, float s2) {
    const float Mn = fmaxf(M, M2);
    if (Mn == -INFINITY) {
        M = Mn;
        s = 0.f;
        return;
    }
    s = s * ex2(M - Mn) + s2 * ex2(M2 - Mn);
    M = Mn;
}

// Argmax pair: larger value wins, lower index on equal values.
__device__ __forceinline__ void am_merge(float &v, int &i, float v2, int i2) {
    if (v2 > v || (v2 == v && i2 < i)) {
        v = v2;
        i = i2;
    }
}

__device__ __forceinline__ void warp_ms_reduce(float &M, float &s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float M2 = __shfl_xor_sync(0xffffffffu, M, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        ms_merge(M, s, M2, s2);
    }
}

__device__ __forceinline__ void warp_am_reduce(float &v, int &i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
        am_merge(v, i, v2, i2);
    }
}

// Epoch ticket: the high word holds the call's epoch, the low word the number
// of CTAs of this call that arrived.  A stale word from an earlier call
// (epoch differs) restarts at one, so the workspace never needs clearing.
// Lock-free: every failed CAS means another CTA's update went through.
__device__ __forceinline__ uint32_t ticket_arrive(unsigned long long *t, uint32_t epoch) {
    unsigned long long cur = *reinterpret_cast<volatile unsigned long long *>(t);
    while (true) {
        const unsigned long long nxt = (static_cast<uint32_t>(cur >> 32) == epoch)
                                           ? cur + 1ull
                                           : ((static_cast<unsigned long long>(epoch) << 32) | 1ull);
        const unsigned long long prev = atomicCAS(t, cur, nxt);
        if (prev == cur) return static_cast<uint32_t>(nxt & 0xffffffffull);
        cur = prev;
    }
}

}  // namespace sv
