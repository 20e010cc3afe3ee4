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
constexpr int kMaxRowsPerRequest = 256;   // SV_MAX_K + 1
constexpr int kSegElems = 256;            // fused kernel: residual masses are kept per 256-token segment
constexpr int kResStageElems = 4096;      // fused kernel: tokens of one residual ring stage
constexpr int kResBlockStages = 4;        // fused kernel: stages per residual work block
constexpr int kResBlockElems = kResStageElems * kResBlockStages;

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

}  // namespace sv

namespace sv {

// ---------------------------------------------------------------------------
// mbarrier / bulk-copy primitives (inline PTX, sm_90+ forms valid on sm_103a)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: gives up after `budget` SM clock cycles and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, long long budget) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > budget) return false;
    }
    return true;
}

// Global -> shared bulk copy completing on an mbarrier (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// The same copy with an L2 eviction-priority hint (a policy from createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Release / acquire helpers for the per-request tickets.
__device__ __forceinline__ uint32_t atom_add_release_gpu(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

}  // namespace sv

namespace sv {

// ---------------------------------------------------------------------------
// Thread-block cluster primitives
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Split cluster barrier: every thread arrives as the kernel starts and waits
// before its first access to another CTA's shared memory, which is only valid
// once every CTA of the cluster is running.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// Whole-cluster barrier; release/acquire orders shared-memory writes before it
// with distributed-shared-memory reads after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Read a float from the shared memory of CTA `rank` of this cluster at the
// address that `p` has in this CTA.
__device__ __forceinline__ float ld_dsmem_f32(const float *p, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(p)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// Store two floats into the shared memory of CTA `rank` of this cluster, at
// the address that `p` has in this CTA (8-byte aligned).  Visible to that CTA
// after the next cluster barrier.
__device__ __forceinline__ void st_dsmem_f32x2(float2 *p, float a, float b, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(p)), "r"(rank));
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(remote), "f"(a), "f"(b) : "memory");
}

}  // namespace sv

namespace sv {
// Programmatic dependent launch: let the next kernel in the stream be
// scheduled early / wait for the previous kernel's completion and memory.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
}  // namespace sv
