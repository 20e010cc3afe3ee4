// Fused LM-head front end (sm_103a): z = hidden . W_vocab on the 5th-generation
// tensor cores, with the verifier's per-row statistics taken in the epilogue.
//
// This is the GEMM whose M grows from B to B (1 + D) under speculation
// ("Co-Designing AI Models Using Speculative Decoding", Guideline 1): all
// M = B (K+1) <= 128 rows of hidden are one tcgen05 M tile, and the kernel
// streams W_vocab (kept as its transpose, V x d, K-major) once.
//
// Persistent CTA per SM over BN-wide vocabulary tiles (BN in {256, 224, 192,
// 128}, chosen per call so that the last wave of tiles is as full as possible):
//   warp 0    TMA producer: 128 x 64 hidden tile + BN x 64 W tile per stage
//             (128-byte swizzle), 4-6 stage ring (full/empty mbarriers); W is
//             streamed with an evict-first L2 hint, hidden with evict-last.
//   warp 1    TMEM allocator and single-thread MMA issuer: 4 tcgen05.mma
//             (kind::f16, bf16 x bf16 -> fp32, M=128, N=BN, K=16) per stage
//             into one of two BN-column TMEM accumulators; tcgen05.commit
//             frees the stage and, after the last k step, publishes the tile.
//   warps 2-5 epilogue: tcgen05.ld of the accumulator (thread = row); each
//             row keeps one running partial (M, s) = (max z c, sum 2^(z c - M))
//             or (max z, first argmax) over all tiles of its CTA, written once
//             at the end, and in sampling mode an fp32 copy of the tiles'
//             logits for the decide gathers and the residual draw.
// The decide step and the residual draw then run over these partials and
// logits (finish_from_partials in verify.cu).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "../../include/specverify.h"
#include "sv_args.cuh"
#include "sv_device.cuh"
#include "sv_draw.cuh"
#include "sv_host.h"
#include "sv_slice.cuh"

namespace sv {
namespace lm {

constexpr int BM = 128;                 // rows of the M tile (all rows of the batch)
constexpr int BK = 64;                  // hidden-size slice per stage: 128 bytes of bf16
constexpr int UK = 16;                  // K of one tcgen05.mma kind::f16
constexpr int kABytes = BM * BK * 2;    // 16 KB
constexpr int kEpiWarps = 4;
constexpr int kThreadsLm = (2 + kEpiWarps) * 32;
constexpr int kLmSmemBudget = 204800;   // shared bytes for the operand ring

// Vocabulary tile width BN (a multiple of 32, <= 256) and the ring depth that
// fits the shared-memory budget.
template <int BN> struct Tile {
    static constexpr int kBBytes = BN * BK * 2;
    static constexpr int kStages = (kLmSmemBudget / (kABytes + kBBytes)) < 6 ? (kLmSmemBudget / (kABytes + kBBytes)) : 6;
    static constexpr int kTmemCols = 2 * BN <= 256 ? 256 : 512;  // two fp32 accumulators, power of two
    // tcgen05 instruction descriptor, kind::f16: D f32, A bf16, B bf16, both
    // K-major, N >> 3 at bit 17, M >> 4 at bit 24.
    static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                       (static_cast<uint32_t>(BN >> 3) << 17) |
                                       (static_cast<uint32_t>(BM >> 4) << 24);
};

template <int BN> struct LmSmem {
    alignas(1024) unsigned char a[Tile<BN>::kStages][kABytes];
    alignas(1024) unsigned char b[Tile<BN>::kStages][Tile<BN>::kBBytes];
    uint64_t full[Tile<BN>::kStages];
    uint64_t empty[Tile<BN>::kStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
    // each epilogue warp's 32 x 32 block of the logits copy, 128-byte swizzled, for a bulk tensor store
    alignas(1024) float stage[kEpiWarps][32 * 32];
};

struct LmArgs {
    int M, d, V, n_tiles;
    float c;          // log2(e) / T
    float *spill;     // M x V fp32 logits (sampling), or nullptr
    int spill_keep;   // 1: the spill is read back from L2 soon (stores at evict_last priority)
    int spill_tma;    // 1: the spill is written by bulk tensor stores through the third tensor map
    float2 *partials; // M x gridDim.x: one merged partial per row and CTA
    uint32_t *status;
    long long wait_budget;  // SM cycles a wait on another warp's work may take (own copies and MMAs: kDrainBudget)
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
// 16-byte global store with an L2 eviction-priority policy.
__device__ __forceinline__ void st_f32x4_hint(float *p, float a, float b, float c, float d, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d), "l"(pol)
                 : "memory");
}

// Invalidate the 128-byte L2 lines that lie wholly inside [begin, end) without
// writing them back (their contents become indeterminate); thread i of n takes
// lines i, i + n, ...  For scratch that nobody reads again.
__device__ __forceinline__ void discard_l2_range(const void *begin, const void *end, int i, int n) {
    const uintptr_t b = (reinterpret_cast<uintptr_t>(begin) + 127u) & ~static_cast<uintptr_t>(127u);
    const uintptr_t e = reinterpret_cast<uintptr_t>(end) & ~static_cast<uintptr_t>(127u);
    for (uintptr_t l = b + static_cast<uintptr_t>(i) * 128u; l < e; l += static_cast<uintptr_t>(n) * 128u)
        asm volatile("discard.global.L2 [%0], 128;" ::"l"(l) : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), sm_100 form.
__device__ __forceinline__ uint64_t smem_desc_sw128(const void *p) {
    const uint64_t addr = smem_addr(p);
    uint64_t d = 0;
    d |= (addr >> 4) & 0x3FFFull;        // start address, 16-byte units
    d |= 1ull << 16;                     // leading byte offset (unused for swizzled K-major)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;  // stride byte offset
    d |= 1ull << 46;                     // descriptor version
    d |= 2ull << 61;                     // 128-byte swizzle
    return d;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Bulk tensor store of a box from shared memory, tracked by the issuing thread's bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int x, int y, uint64_t policy) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_addr(src)), "r"(x), "r"(y), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The thread's committed bulk stores have read their shared memory / have completed.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Order this thread's generic-proxy shared-memory writes before later async-proxy reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <bool kSample, int BN>
__global__ void __launch_bounds__(kThreadsLm, 1)
    lmhead_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, LmArgs a) {
    constexpr int kStagesLm = Tile<BN>::kStages;
    constexpr int kBBytes = Tile<BN>::kBBytes;
    constexpr int kTmemCols = Tile<BN>::kTmemCols;
    extern __shared__ unsigned char smem_raw[];
    LmSmem<BN> &sm =
        *reinterpret_cast<LmSmem<BN> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nk = a.d / BK;
    if (tid == 0) {
        for (int s = 0; s < kStagesLm; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.acc_full[i], 1);
            mbar_init(&sm.acc_empty[i], kEpiWarps);
        }
        mbar_init(&sm.mma_done, 1);
        sm.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&sm.tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    volatile int *abort_flag = &sm.abort;
    auto timeout = [&]() {
        *abort_flag = 1;
        atomicOr(a.status, SV_FLAG_TIMEOUT);
    };

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_h = l2_policy_evict_last();
            int kg = 0;
            for (int t = blockIdx.x; t < a.n_tiles && !*abort_flag; t += gridDim.x) {
                for (int kb = 0; kb < nk; ++kb, ++kg) {
                    const int s = kg % kStagesLm;
                    if (kg >= kStagesLm &&
                        !mbar_wait_bounded(&sm.empty[s], ((kg / kStagesLm) - 1) & 1, a.wait_budget)) {
                        timeout();
                        break;
                    }
                    mbar_arrive_expect_tx(&sm.full[s], kABytes + kBBytes);
                    tma_load_2d(sm.a[s], &tmA, kb * BK, 0, &sm.full[s], pol_h);
                    tma_load_2d(sm.b[s], &tmB, kb * BK, t * BN, &sm.full[s], pol_w);
                }
            }
            // let every copy issued into the ring land before the CTA can leave
            for (int kk = max(0, kg - kStagesLm); kk < kg; ++kk)
                mbar_wait_bounded(&sm.full[kk % kStagesLm], (kk / kStagesLm) & 1, kDrainBudget);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int kg = 0, ti = 0;
            for (int t = blockIdx.x; t < a.n_tiles && !*abort_flag; t += gridDim.x, ++ti) {
                const int buf = ti & 1;
                if (ti >= 2 && !mbar_wait_bounded(&sm.acc_empty[buf], ((ti / 2) - 1) & 1, a.wait_budget)) {
                    timeout();
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * BN);
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb, ++kg) {
                    const int s = kg % kStagesLm;
                    if (!mbar_wait_bounded(&sm.full[s], (kg / kStagesLm) & 1, a.wait_budget)) {
                        timeout();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = smem_desc_sw128(sm.a[s]);
                    const uint64_t bd = smem_desc_sw128(sm.b[s]);
#pragma unroll
                    for (int kk = 0; kk < BK / UK; ++kk)  // advance 32 bytes (16 bf16) inside the swizzle atom
                        tc_mma(d_tmem, ad + 2ull * kk, bd + 2ull * kk, Tile<BN>::kIdesc, (kb | kk) ? 1u : 0u);
                    tc_commit(&sm.empty[s]);
                }
                if (!ok) break;
                tc_commit(&sm.acc_full[buf]);
            }
            // all issued MMAs complete before TMEM is released
            tc_commit(&sm.mma_done);
            mbar_wait_bounded(&sm.mma_done, 0, kDrainBudget);  // own MMAs, before TMEM is released
        }
    } else {
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const bool live = row < a.M;
        const bool vec_store = (a.V & 3) == 0;
        const uint64_t keep_pol = l2_evict_last_policy();
        float *stage = sm.stage[quad];
        // running partial of this row over every tile of the CTA
        float Mr = -INFINITY, Sr = 0.f;
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        int ti = 0;
        for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x, ++ti) {
            const int buf = ti & 1;
            if (!mbar_wait_bounded(&sm.acc_full[buf], (ti / 2) & 1, a.wait_budget)) timeout();
            if (*abort_flag) break;
            tc_fence_after();
            const int n0 = t * BN;
#pragma unroll 1
            for (int cb = 0; cb < BN / 32; ++cb) {
                float v[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(buf * BN + cb * 32),
                          v);
                const int col0 = n0 + cb * 32;
                const int nvalid = min(32, a.V - col0);
                if (nvalid <= 0) continue;  // the same for the whole warp
                if (kSample && a.spill_tma) {
                    // the warp's 32 x 32 block of the copy: every lane stages its row (rows past M
                    // and columns past V are clipped by the tensor map), one lane stores the box
                    if (lane == 0) bulk_wait_read_all();  // the previous store has read the stage
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)  // 16-byte chunk j of row `lane`, 128-byte swizzle
                        *reinterpret_cast<float4 *>(stage + lane * 32 + ((j ^ (lane & 7)) * 4)) =
                            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, stage, col0, quad * 32, a.spill_keep ? keep_pol : l2_evict_normal_policy());
                        bulk_commit();
                    }
                }
                if (!live) continue;
                if (kSample) {
                    float m = -INFINITY;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < nvalid) m = fmaxf(m, v[i]);
                    if (m != -INFINITY) {
                        const float Mn = fmaxf(Mr, m * a.c);
                        float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (i < nvalid) sacc[i & 3] += ex2(fmaf(v[i], a.c, -Mn));
                        Sr = Sr * ex2(Mr - Mn) + ((sacc[0] + sacc[1]) + (sacc[2] + sacc[3]));
                        Mr = Mn;
                    }
                    float *dst = a.spill + static_cast<size_t>(row) * a.V + col0;
                    if (a.spill_tma) {
                        // stored above
                    } else if (vec_store && nvalid == 32 && a.spill_keep) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) st_f32x4_hint(dst + i, v[i], v[i + 1], v[i + 2], v[i + 3], keep_pol);
                    } else if (vec_store && nvalid == 32) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4 *>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (i < nvalid) dst[i] = v[i];
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < nvalid && (bi == 0x7fffffff || v[i] > bv)) {
                            bv = v[i];
                            bi = col0 + i;
                        }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.acc_empty[buf]);  // accumulator drained
        }
        if (kSample && a.spill_tma && lane == 0) bulk_wait_all();  // the copy is complete before the kernel ends
        if (live)
            a.partials[static_cast<size_t>(row) * gridDim.x + blockIdx.x] =
                kSample ? make_float2(Mr, Sr) : make_float2(bv, __int_as_float(bi));
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Row-major bf16 matrix of `rows` x `cols` read in boxes of box_rows x 64.
static bool encode_bf16_kmajor(CUtensorMap *map, const void *base, int rows, int cols, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The M x V fp32 logits copy as 32 x 32 boxes, 128-byte swizzled (rows of V floats, V a multiple of 4).
static bool encode_f32_rows(CUtensorMap *map, const float *base, int rows, int cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct LmLayout {
    size_t finish, partials, segs, spill, total;
};

static inline size_t a256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Tile width that fills the last wave of tiles best (ties: the wider tile).
static int choose_bn(int V, int sms) {
    const int cands[4] = {256, 224, 192, 128};
    int best = 256;
    double best_eff = -1.0;
    for (int bn : cands) {
        const long long tiles = (V + bn - 1) / bn;
        const long long waves = (tiles + sms - 1) / sms;
        const double eff = static_cast<double>(tiles) / static_cast<double>(waves * sms);
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = bn;
        }
    }
    return best;
}

constexpr int kMaxLmGrid = 1024;  // partials are sized for at most this many CTAs

static LmLayout lm_layout(int B, int K, int V) {
    const int M = B * (K + 1);
    const size_t n_tiles = kMaxLmGrid;  // one partial per row and CTA
    LmLayout L;
    size_t o = 0;
    L.finish = o;
    o = a256(o + finish_workspace_size(B, M, V));
    L.partials = o;
    o = a256(o + sizeof(float2) * static_cast<size_t>(M) * n_tiles);
    L.segs = o;  // per request, one sum per 256-token segment (the cluster finish's scratch)
    o = a256(o + sizeof(float) * static_cast<size_t>(B) * ((V + kSegElems - 1) / kSegElems));
    L.spill = o;
    o = a256(o + sizeof(float) * static_cast<size_t>(M) * V);
    L.total = o;
    return L;
}

// Launch with `grid` CTAs (grid <= n_tiles, <= kMaxLmGrid).
template <bool kSample, int BN>
static void launch_gemm(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc, const LmArgs &a, int grid,
                        cudaStream_t s) {
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    static_assert(sizeof(LmSmem<BN>) + 1024 <= 232448, "shared memory of one CTA on this GPU");
    const int smem = static_cast<int>(sizeof(LmSmem<BN>)) + 1024;
    if (!configured[dev]) {
        cudaFuncSetAttribute(lmhead_gemm_kernel<kSample, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        configured[dev] = true;
    }
    lmhead_gemm_kernel<kSample, BN><<<grid, kThreadsLm, smem, s>>>(ta, tb, tc, a);
}

template <bool kSample>
static void launch_gemm_bn(int bn, const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc, const LmArgs &a,
                           int grid, cudaStream_t s) {
    switch (bn) {
        case 224: launch_gemm<kSample, 224>(ta, tb, tc, a, grid, s); break;
        case 192: launch_gemm<kSample, 192>(ta, tb, tc, a, grid, s); break;
        case 128: launch_gemm<kSample, 128>(ta, tb, tc, a, grid, s); break;
        default: launch_gemm<kSample, 256>(ta, tb, tc, a, grid, s); break;
    }
}

// ---------------------------------------------------------------------------
// Draft sampling (the step before verification): q = softmax(h . W / T) and
// x ~ q for every draft row.  The GEMM above writes the fp32 logits straight
// into the caller's q buffer and one (M, S) partial per row and CTA; then one
// CTA per row merges the partials, turns the row into q in place and draws x
// by inverse CDF with a Philox4x32-10 uniform.
// ---------------------------------------------------------------------------
constexpr int kDraftThreads = 1024;
constexpr int kDraftWarps = kDraftThreads / 32;
static_assert(kDraftWarps == 32, "the warp totals are scanned by one warp");
constexpr int kMaxDraftSegs = 4096;  // V <= 4096 x 256 tokens
constexpr uint32_t kDraftStream = 1;  // Philox stream of the draft draws
constexpr int kDraftBatch = 4;        // segments whose logits a warp loads before using any

// First output word of Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel
// random numbers: as easy as 1, 2, 3", SC 2011) at counter (index low word,
// stream, index high word, 0) and key (seed low word, seed high word).
__device__ __forceinline__ uint32_t philox_w0(uint64_t seed, uint64_t index, uint32_t stream) {
    uint32_t c0 = static_cast<uint32_t>(index), c1 = stream, c2 = static_cast<uint32_t>(index >> 32), c3 = 0u;
    uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return c0;
}

// u = ((w0 >> 9) + 1/2) 2^-23, exact in fp32, in (0, 1).
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint64_t index, uint32_t stream) {
    const uint32_t w = philox_w0(seed, index, stream);
    return __fmul_rn(__fadd_rn(__uint2float_rn(w >> 9), 0.5f), 1.0f / 8388608.0f);
}

template <bool kSample>
__global__ void __launch_bounds__(kDraftThreads) draft_finish_kernel(float *q, const float2 *partials, int n_parts,
                                                                     int V, float c, uint64_t seed, uint64_t offset,
                                                                     int32_t *x_out, float *u_out) {
    pdl_wait_prior_grid();  // the logits and partials come from the GEMM before it
    pdl_launch_dependents();
    const int row = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    __shared__ float2 s_part[kDraftWarps];
    __shared__ float s_segsum[kMaxDraftSegs];
    __shared__ DS s_wtot[kDraftWarps], s_wincl[kDraftWarps];
    __shared__ int s_owner, s_vstar;
    __shared__ float s_u;

    // merge the row's partials in a fixed order (per warp, then warp 0 over the warps)
    float ra;
    int rb;
    partial_identity<kSample>(ra, rb);
    for (int i = tid; i < n_parts; i += kDraftThreads)
        merge_pair<kSample>(ra, rb, partials[static_cast<size_t>(row) * n_parts + i]);
    warp_partial_reduce<kSample>(ra, rb);
    if (lane == 0) s_part[warp] = make_float2(ra, __int_as_float(rb));
    if (tid == 0) {
        s_owner = 0x7fffffff;
        s_vstar = -1;
        s_u = kSample ? philox_uniform(seed, offset + static_cast<uint64_t>(row), kDraftStream) : 0.f;
    }
    __syncthreads();
    if (warp == 0) {
        const float2 w = s_part[lane];
        ra = w.x;
        rb = __float_as_int(w.y);
        warp_partial_reduce<kSample>(ra, rb);
        if (lane == 0) s_part[0] = make_float2(ra, __int_as_float(rb));
    }
    __syncthreads();
    if (!kSample) {  // greedy drafting: the argmax
        if (tid == 0) x_out[row] = __float_as_int(s_part[0].y);
        return;
    }
    const float M = s_part[0].x, invS = 1.f / s_part[0].y;
    const float u = s_u;
    float *qrow = q + static_cast<size_t>(row) * V;
    const int ns = (V + kSegElems - 1) / kSegElems;
    const int G = (ns + kDraftWarps - 1) / kDraftWarps;
    const int g0 = min(warp * G, ns), g1 = min(g0 + G, ns);

    // pass 1: each warp turns its segments into q (in place) and sums them in order.  The logits of
    // kDraftBatch segments are loaded before any is used, so that a warp keeps that many 1 KB reads
    // in flight (the row comes from L2; one segment at a time left the loads latency-bound).
    DS wt{0.f, 0.f};
    for (int gb = g0; gb < g1; gb += kDraftBatch) {
        float4 zb[kDraftBatch][2];
#pragma unroll
        for (int b = 0; b < kDraftBatch; ++b)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int e0 = (gb + b) * kSegElems + (j * 32 + lane) * 4;
                zb[b][j] = (gb + b < g1 && e0 < V) ? __ldcs(reinterpret_cast<const float4 *>(qrow + e0))
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
        for (int b = 0; b < kDraftBatch; ++b) {
            const int g = gb + b;
            if (g >= g1) break;
            float r[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int e0 = g * kSegElems + (j * 32 + lane) * 4;
                const float z[4] = {zb[b][j].x, zb[b][j].y, zb[b][j].z, zb[b][j].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) r[j][k] = e0 < V ? __fmul_rn(ex2(__fmaf_rn(z[k], c, -M)), invS) : 0.f;
                if (e0 < V) *reinterpret_cast<float4 *>(qrow + e0) = make_float4(r[j][0], r[j][1], r[j][2], r[j][3]);
            }
            const float m = seg_sum(r);
            if (lane == 0) s_segsum[g] = m;
            wt = ds_add_f(wt, m);
        }
    }
    if (lane == 0) s_wtot[warp] = wt;
    __syncthreads();
    // inclusive prefix of the warp totals (one warp, shuffle scan), then the owner: the warp whose range
    // holds u R.  Lower and upper ends of every range come from the same scan, so exactly one warp owns
    // any u R below the total.
    if (warp == 0) {
        DS p = s_wtot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const DS y = ds_shfl_up(p, o);
            if (lane >= o) p = ds_add(y, p);
        }
        s_wincl[lane] = p;
    }
    __syncthreads();
    const DS R = s_wincl[kDraftWarps - 1];
    const DS Pw = warp > 0 ? s_wincl[warp - 1] : DS{0.f, 0.f};
    const DS t = ds_mul_f(R, u);
    if (lane == 0 && g0 < g1 && !ds_gt(Pw, t) && ds_gt(s_wincl[warp], t)) atomicMin(&s_owner, warp);
    __syncthreads();

    // the owning warp finds the segment, then the token, in token order
    if (warp == s_owner) {
        DS P = Pw, fbase{0.f, 0.f};
        int fseg = -1;
        for (int g = g0; g < g1; ++g) {
            const DS Pn = ds_add_f(P, s_segsum[g]);
            // the range holds u R; if its running sum falls short by rounding, its last segment
            if (ds_gt(Pn, t) || g == g1 - 1) {
                fseg = g;
                fbase = P;
                break;
            }
            P = Pn;
        }
        int vstar = -1;
        if (fseg >= 0) {
            float r[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int e0 = fseg * kSegElems + (j * 32 + lane) * 4;
                const float4 w = (e0 < V) ? *reinterpret_cast<const float4 *>(qrow + e0) : make_float4(0.f, 0.f, 0.f, 0.f);
                r[j][0] = w.x;
                r[j][1] = w.y;
                r[j][2] = w.z;
                r[j][3] = w.w;
            }
            vstar = warp_seg_scan(r, fseg, V, fbase, t, lane).v;
            // sums that end short of u R inside the segment: the next token with q > 0
            for (int g = fseg + 1; g < ns && vstar < 0; ++g) {
                int loc = 0x7fffffff;
#pragma unroll
                for (int j = 1; j >= 0; --j) {
                    const int e0 = g * kSegElems + (j * 32 + lane) * 4;
                    if (e0 < V) {
                        const float4 w = *reinterpret_cast<const float4 *>(qrow + e0);
                        if (w.w > 0.f) loc = e0 + 3;
                        if (w.z > 0.f) loc = e0 + 2;
                        if (w.y > 0.f) loc = e0 + 1;
                        if (w.x > 0.f) loc = e0;
                    }
                }
                const int best = __reduce_min_sync(0xffffffffu, loc);
                if (best != 0x7fffffff) vstar = best;
            }
        }
        if (lane == 0) s_vstar = vstar;
    }
    __syncthreads();
    int vstar = s_vstar;
    if (vstar < 0) {
        // u R at or above every boundary: the last token with q > 0
        for (int v = V - 1 - tid; v >= 0; v -= kDraftThreads)
            if (qrow[v] > 0.f) {
                atomicMax(&s_vstar, v);
                break;
            }
        __syncthreads();
        vstar = s_vstar;
    }
    if (tid == 0) {
        x_out[row] = vstar;
        if (u_out) u_out[row] = u;
    }
}

// ---------------------------------------------------------------------------
// Verification after the LM-head GEMM, one cluster of kFinC CTAs per request.
// The GEMM left the fp32 logits (the spill, mostly in L2) and one partial per
// row and GEMM CTA.  Every CTA merges the request's row partials and runs the
// accept tests and the first-reject scan (the same result in each; rank 0
// writes it).  For the final draw each CTA computes r over its contiguous
// slice of 256-token segments straight from L2 into registers, keeps the
// segment sums in shared memory (and in a global scratch row), and sends its
// slice total to every CTA of the cluster with remote stores.  After one
// cluster barrier each CTA holds all slice totals, computes the same prefix,
// R and u R, and the one CTA whose slice holds u R finds the segment in its
// own shared memory and the token in that segment (double-single prefix,
// in-segment running sums, the usual rounding fallbacks).  Nothing reads
// another CTA's shared memory after the barrier, so no CTA waits for another
// to finish.
// ---------------------------------------------------------------------------
constexpr int kFinC = 8;            // CTAs per request
constexpr int kFinThreads = 512;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kFinBatch = 2;        // segments whose loads a warp holds in flight at once
constexpr int kFinMaxSegs = 96;     // segments per CTA: V <= kFinC x 96 x 256 = 196608

__host__ __device__ constexpr int fin_segs_per_cta(int V) {
    return ((V + kSegElems - 1) / kSegElems + kFinC - 1) / kFinC;
}

// The 8 tokens a lane holds in 256-token segment g: token g * 256 + (j * 32 +
// lane) * 4 + k, j < 2, k < 4 (zero beyond V).  Loading and computing are
// split so that a warp can hold several segments' loads in flight.
__device__ __forceinline__ void fin_fetch(const float *zrow, const float *qrow, int V, int g, int lane,
                                          float4 (&z)[2], float4 (&qv)[2]) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int e0 = g * kSegElems + (j * 32 + lane) * 4;
        const bool in = e0 < V;
        z[j] = in ? __ldcs(reinterpret_cast<const float4 *>(zrow + e0)) : make_float4(0.f, 0.f, 0.f, 0.f);
        qv[j] = (in && qrow) ? __ldcs(reinterpret_cast<const float4 *>(qrow + e0)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}
// r(v) = max(0, p(v) - q(v)) of those tokens (p(v) alone without a q row),
// p(v) = 2^(z(v) c - M) / S.
__device__ __forceinline__ void fin_r(const float4 (&z)[2], const float4 (&qv)[2], bool has_q, int V, int g,
                                      int lane, float c, float M, float invS, float (&r)[2][4]) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const bool in = g * kSegElems + (j * 32 + lane) * 4 < V;
        const float zz[4] = {z[j].x, z[j].y, z[j].z, z[j].w}, qq[4] = {qv[j].x, qv[j].y, qv[j].z, qv[j].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float p = __fmul_rn(ex2(__fmaf_rn(zz[k], c, -M)), invS);
            r[j][k] = in ? (has_q ? fmaxf(__fsub_rn(p, qq[k]), 0.f) : p) : 0.f;
        }
    }
}

template <bool kSample>
__global__ void __launch_bounds__(kFinThreads, 2) verify_finish_kernel(const float *spill, const float2 *partials,
                                                                    int n_parts, const float *q, int K, int V,
                                                                    float c, const int32_t *draft,
                                                                    const float *uniforms, int32_t *out_tokens,
                                                                    int32_t *accept_len, float *diag,
                                                                    uint32_t *status, float *seg_scratch, int B) {
    cluster_arrive_relaxed();  // waited on before the first remote store
    pdl_wait_prior_grid();  // the spill and the partials come from the GEMM before it
    pdl_launch_dependents();
    const uint32_t rank = cluster_ctarank();
    const int b = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nr = K + 1, r0 = b * nr, d0 = b * K, n_draft = B * K;
    const int nsp = fin_segs_per_cta(V), ns = (V + kSegElems - 1) / kSegElems;
    const int seg0 = min(static_cast<int>(rank) * nsp, ns), seg1 = min(seg0 + nsp, ns), nloc = seg1 - seg0;
    __shared__ float2 s_row[SV_MAX_K + 1];
    __shared__ int s_x[SV_MAX_K];
    __shared__ float s_z[SV_MAX_K], s_q[SV_MAX_K], s_u[SV_MAX_K];
    __shared__ float s_seg[kFinMaxSegs];
    __shared__ float2 s_tot[2][kFinC];  // slice totals (double-single), written by every CTA of the cluster
    __shared__ int s_ks, s_retry;

    // accept-test operands of draft j = tid: independent of the merge below, so issued first
    int xj = -1;
    float zj = 0.f, qj = 0.f, uj = 0.f;
    if (tid < K) {
        xj = __ldg(draft + d0 + tid);
        if (xj < 0 || xj >= V) {
            xj = -1;
        } else if (kSample) {
            zj = __ldcg(spill + static_cast<size_t>(r0 + tid) * V + xj);
            qj = __ldg(q + static_cast<size_t>(d0 + tid) * V + xj);
            uj = __ldg(uniforms + r0 + tid);
        }
    }
    // row normalisers: warp w merges rows w, w + 16, ... over the GEMM's CTAs, in order
    for (int j = warp; j < nr; j += kFinWarps) {
        float ra;
        int rb;
        partial_identity<kSample>(ra, rb);
        for (int i = lane; i < n_parts; i += 32)
            merge_pair<kSample>(ra, rb, partials[static_cast<size_t>(r0 + j) * n_parts + i]);
        warp_partial_reduce<kSample>(ra, rb);
        if (lane == 0) s_row[j] = make_float2(ra, __int_as_float(rb));
    }
    if (tid < K) {
        s_x[tid] = xj;
        s_z[tid] = zj;
        s_q[tid] = qj;
        s_u[tid] = uj;
    }
    __syncthreads();

    // accept tests and first-reject scan (warp 0 of every CTA; rank 0 writes the outputs)
    if (warp == 0) {
        bool bad = false;
        for (int j = lane; j < K; j += 32) bad |= s_x[j] < 0;
        bad = __any_sync(0xffffffffu, bad);
        int ks = -1;
        for (int jb = 0; !bad && jb < nr && ks < 0; jb += 32) {
            const int j = jb + lane;
            bool rej = false;
            if (j < K) {
                const float2 sj = s_row[j];
                if (kSample) {
                    const float p = exp2f(fmaf(s_z[j], c, -sj.x)) / sj.y;
                    rej = !(s_u[j] * s_q[j] <= p);
                    if (diag && rank == 0) diag[d0 + j] = p;
                } else {
                    rej = (s_x[j] != __float_as_int(sj.y));
                }
            }
            const unsigned m = __ballot_sync(0xffffffffu, rej);
            if (m) ks = jb + __ffs(m) - 1;
            else if (jb + 32 >= nr) ks = K;
        }
        if (rank == 0) {
            if (bad) {
                for (int j = lane; j < nr; j += 32) out_tokens[r0 + j] = -1;
                if (lane == 0) {
                    accept_len[b] = 0;
                    atomicOr(status, SV_FLAG_BAD_TOKEN);
                }
            } else {
                for (int j = lane; j < nr; j += 32) {
                    int v = -1;
                    if (j < ks) v = s_x[j];
                    else if (j == ks && !kSample) v = __float_as_int(s_row[ks].y);
                    out_tokens[r0 + j] = v;
                }
                if (lane == 0) accept_len[b] = ks + 1;
            }
        }
        if (lane == 0) s_ks = bad ? -1 : ks;
    }
    __syncthreads();
    // every CTA of the cluster has the same ks: leaving together touches no other CTA's memory
    if (!kSample || s_ks < 0) return;
    cluster_wait();  // every CTA of the cluster is running: remote stores below are safe

    const int ks = s_ks;
    const float M = s_row[ks].x, invS = 1.f / s_row[ks].y;
    const float *zrow = spill + static_cast<size_t>(r0 + ks) * V;
    const float *qrow0 = (ks < K) ? q + static_cast<size_t>(d0 + ks) * V : nullptr;
    float *gseg = seg_scratch + static_cast<size_t>(b) * ns;
    // warp 0's share of the local segments and its exclusive prefix within the slice
    const int G = (nloc + 31) / 32;
    const int i0 = min(lane * G, nloc), i1 = min(i0 + G, nloc);
    DS excl{0.f, 0.f};
    int attempt = 0;
    const float *qrow = qrow0;
    for (;; ++attempt) {
        qrow = (attempt == 0) ? qrow0 : nullptr;
        // r over this CTA's segments, kFinBatch segments per warp in flight
        for (int gb = seg0 + warp; gb < seg1; gb += kFinBatch * kFinWarps) {
            float4 zb[kFinBatch][2], qb[kFinBatch][2];
#pragma unroll
            for (int i = 0; i < kFinBatch; ++i) {
                const int g = gb + i * kFinWarps;
                if (g < seg1) fin_fetch(zrow, qrow, V, g, lane, zb[i], qb[i]);
            }
#pragma unroll
            for (int i = 0; i < kFinBatch; ++i) {
                const int g = gb + i * kFinWarps;
                if (g < seg1) {
                    float r[2][4];
                    fin_r(zb[i], qb[i], qrow != nullptr, V, g, lane, c, M, invS, r);
                    const float s = seg_sum(r);
                    if (lane == 0) {
                        s_seg[g - seg0] = s;
                        gseg[g] = s;
                    }
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
            if (lane < kFinC) st_dsmem_f32x2(&s_tot[attempt][rank], tot.hi, tot.lo, static_cast<uint32_t>(lane));
        }
        cluster_sync();
        // the same totals in the same order in every CTA: an empty residual is seen by all of them
        if (attempt == 0 && qrow0 != nullptr) {
            if (tid == 0) {
                DS R{0.f, 0.f};
                for (int k = 0; k < kFinC; ++k) R = ds_add(R, DS{s_tot[0][k].x, s_tot[0][k].y});
                s_retry = R.hi > 0.f ? 0 : 1;
            }
            __syncthreads();
            if (s_retry) {
                if (rank == 0 && tid == 0) atomicOr(status, SV_FLAG_ZERO_RESIDUAL);  // draw from p
                continue;
            }
        }
        break;
    }
    if (warp != 0) {
        // every CTA's gathers are behind the barrier: the other rows' slices are read by nobody
        // again, so warps 1.. drop their L2 lines unwritten while warp 0 draws
        const int t1 = min(seg1 * kSegElems, V), t0s = seg0 * kSegElems;
        for (int j = 0; j < nr; ++j)
            if (j != ks && t1 > t0s)
                discard_l2_range(spill + static_cast<size_t>(r0 + j) * V + t0s, spill + static_cast<size_t>(r0 + j) * V + t1,
                                 tid - 32, kFinThreads - 32);
        return;
    }

    // prefix of the slice totals, R, u R and the CTA whose slice holds u R
    const float u = __ldg(uniforms + r0 + K);
    DS P{0.f, 0.f}, Pmine{0.f, 0.f};
    DS Pk[kFinC + 1];
    Pk[0] = P;
#pragma unroll
    for (int k = 0; k < kFinC; ++k) {
        P = ds_add(P, DS{s_tot[attempt][k].x, s_tot[attempt][k].y});
        Pk[k + 1] = P;
    }
    const DS R = P;
    const DS t = ds_mul_f(R, u);
    int owner = -1, last_pos = -1;
#pragma unroll
    for (int k = kFinC - 1; k >= 0; --k) {
        if (ds_gt(Pk[k + 1], t)) owner = k;
        if (last_pos < 0 && s_tot[attempt][k].x > 0.f) last_pos = k;
    }
#pragma unroll
    for (int k = 0; k < kFinC; ++k)
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
            const int fseg = seg0 + __shfl_sync(0xffffffffu, found, src);
            const DS fbase = ds_shfl(fb, src);
            float r[2][4];
            seg_r<float>(zrow + static_cast<size_t>(fseg) * kSegElems,
                         qrow ? qrow + static_cast<size_t>(fseg) * kSegElems : nullptr, fseg, V, c, M, invS, lane, r);
            const TileScan ts = warp_seg_scan(r, fseg, V, fbase, t, lane);
            vstar = ts.v;
            rstar = ts.rv;
            next = fseg + 1;
        }
        if (vstar < 0)
            vstar = find_positive<float, true>(zrow, qrow, V, ns, c, M, invS, s_seg, gseg, seg0, seg1, next, lane,
                                            &rstar);
    }
    if (vstar < 0)
        vstar = find_positive<float, false>(zrow, qrow, V, ns, c, M, invS, s_seg, gseg, seg0, seg1, ns - 1, lane,
                                         &rstar);
    if (lane == 0) {
        out_tokens[r0 + ks] = vstar;
        if (diag) {
            const float Rf = __fadd_rn(R.hi, R.lo);
            diag[n_draft + 2 * b] = Rf;
            diag[n_draft + 2 * b + 1] = __fdiv_rn(rstar, Rf);
        }
    }
}

}  // namespace lm
}  // namespace sv

using namespace sv;

extern "C" size_t spec_lmhead_workspace_size(int B, int K, int d, int V) {
    (void)d;
    if (B <= 0 || K < 0 || V <= 0) return 256;
    return lm::lm_layout(B, K, V).total;
}

extern "C" sv_status spec_lmhead_verify(const void *hidden, const void *w_vocab_t, int d, const float *q, int B,
                                        int K, int V, float temperature, const int32_t *draft,
                                        const float *uniforms, int32_t *out_tokens, int32_t *accept_len,
                                        float *diag, void *ws, size_t ws_bytes, void *stream) {
    if (B < 0 || K < 0 || K > SV_MAX_K || V <= 0 || !(temperature >= 0.f) || !std::isfinite(temperature))
        return SV_ERR_INVALID;
    if (B == 0) {
        set_launches(0);
        return SV_OK;
    }
    const int M = B * (K + 1);
    const bool sample = temperature > 0.f;
    if (M > lm::BM || d < lm::BK || d % lm::BK != 0) return SV_ERR_INVALID;
    if (!hidden || !w_vocab_t || !out_tokens || !accept_len || !ws) return SV_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(hidden) & 15u) || (reinterpret_cast<uintptr_t>(w_vocab_t) & 15u))
        return SV_ERR_INVALID;
    if (K > 0 && !draft) return SV_ERR_INVALID;
    if (sample && (!uniforms || (K > 0 && !q))) return SV_ERR_INVALID;
    const lm::LmLayout L = lm::lm_layout(B, K, V);
    if (ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return SV_ERR_WORKSPACE;

    const int bn = lm::choose_bn(V, sm_count());
    const int n_tiles = (V + bn - 1) / bn;
    int grid = n_tiles < sm_count() ? n_tiles : sm_count();
    if (grid > lm::kMaxLmGrid) grid = lm::kMaxLmGrid;
    CUtensorMap ta, tb;
    if (!lm::encode_bf16_kmajor(&ta, hidden, M, d, lm::BM) || !lm::encode_bf16_kmajor(&tb, w_vocab_t, V, d, bn))
        return SV_ERR_CUDA;
    char *w = static_cast<char *>(ws);
    lm::LmArgs a;
    a.M = M;
    a.d = d;
    a.V = V;
    a.n_tiles = n_tiles;
    a.c = sample ? static_cast<float>(1.4426950408889634 / static_cast<double>(temperature)) : 1.f;
    a.spill = sample ? reinterpret_cast<float *>(w + L.spill) : nullptr;
    a.partials = reinterpret_cast<float2 *>(w + L.partials);
    a.status = reinterpret_cast<uint32_t *>(w + L.finish);  // the status word is the workspace's first word
    a.wait_budget = wait_budget();
    // the cluster finish reads back only the selected rows and discards the rest from L2
    const bool cluster_finish = V % 4 == 0 && lm::fin_segs_per_cta(V) <= lm::kFinMaxSegs &&
                                (!sample || K == 0 || (reinterpret_cast<uintptr_t>(q) & 15u) == 0);
    a.spill_keep = (sample && cluster_finish) ? 1 : 0;
    // the copy through bulk tensor stores (rows of V floats must be 16-byte multiples)
    CUtensorMap tc = tb;
    a.spill_tma = (sample && V % 4 == 0 && lm::encode_f32_rows(&tc, a.spill, M, V)) ? 1 : 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    prof_begin(s);
    if (sample) lm::launch_gemm_bn<true>(bn, ta, tb, tc, a, grid, s);
    else lm::launch_gemm_bn<false>(bn, ta, tb, tc, a, grid, s);
    prof_end(s);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    if (cluster_finish) {
        // one cluster of kFinC CTAs per request over the spill and the partials
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(lm::kFinC, B);
        cfg.blockDim = dim3(lm::kFinThreads);
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = lm::kFinC;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        const float *spill = reinterpret_cast<const float *>(w + L.spill);
        const float2 *parts = a.partials;
        float *segs = reinterpret_cast<float *>(w + L.segs);
        const cudaError_t e =
            sample ? cudaLaunchKernelEx(&cfg, lm::verify_finish_kernel<true>, spill, parts, grid, q, K, V, a.c, draft,
                                        uniforms, out_tokens, accept_len, diag, a.status, segs, B)
                   : cudaLaunchKernelEx(&cfg, lm::verify_finish_kernel<false>, spill, parts, grid, q, K, V, a.c, draft,
                                        uniforms, out_tokens, accept_len, static_cast<float *>(nullptr), a.status,
                                        segs, B);
        set_launches(2);
        return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
    }
    int more = 0;
    const sv_status st = finish_from_partials(reinterpret_cast<const float *>(w + L.spill), a.partials, grid, q,
                                              B, K, V, sample ? temperature : 1.f, sample, draft, uniforms,
                                              out_tokens, accept_len, diag, w + L.finish, L.partials - L.finish, s,
                                              &more);
    set_launches(1 + more);
    return st;
}

// Workspace of spec_draft_sample: a status word, then one partial per row and
// GEMM CTA.
extern "C" size_t spec_draft_workspace_size(int M, int d, int V) {
    (void)d;
    (void)V;
    if (M <= 0) return 256;
    return 256 + lm::a256(sizeof(float2) * static_cast<size_t>(M) * lm::kMaxLmGrid);
}

extern "C" sv_status spec_draft_sample(const void *hidden, const void *w_vocab_t, int d, int M, int V,
                                       float temperature, uint64_t seed, uint64_t offset, float *q_out,
                                       int32_t *x_out, float *u_out, void *ws, size_t ws_bytes, void *stream) {
    if (M < 0 || M > lm::BM || V <= 0 || V % 4 != 0 || V > lm::kMaxDraftSegs * kSegElems || d < lm::BK ||
        d % lm::BK != 0 || !(temperature >= 0.f) || !std::isfinite(temperature))
        return SV_ERR_INVALID;
    if (M == 0) {
        set_launches(0);
        return SV_OK;
    }
    const bool sample = temperature > 0.f;
    if (!hidden || !w_vocab_t || !x_out || !ws || (sample && !q_out)) return SV_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(hidden) & 15u) || (reinterpret_cast<uintptr_t>(w_vocab_t) & 15u) ||
        (sample && (reinterpret_cast<uintptr_t>(q_out) & 15u)))
        return SV_ERR_INVALID;
    if (ws_bytes < spec_draft_workspace_size(M, d, V) || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return SV_ERR_WORKSPACE;
    const int bn = lm::choose_bn(V, sm_count());
    const int n_tiles = (V + bn - 1) / bn;
    int grid = n_tiles < sm_count() ? n_tiles : sm_count();
    if (grid > lm::kMaxLmGrid) grid = lm::kMaxLmGrid;
    CUtensorMap ta, tb;
    if (!lm::encode_bf16_kmajor(&ta, hidden, M, d, lm::BM) || !lm::encode_bf16_kmajor(&tb, w_vocab_t, V, d, bn))
        return SV_ERR_CUDA;
    char *w = static_cast<char *>(ws);
    lm::LmArgs a;
    a.M = M;
    a.d = d;
    a.V = V;
    a.n_tiles = n_tiles;
    a.c = sample ? static_cast<float>(1.4426950408889634 / static_cast<double>(temperature)) : 1.f;
    a.spill = sample ? q_out : nullptr;  // the logits land in q's buffer, turned into q in place
    a.spill_keep = 1;                    // read back and rewritten as q by the finish kernel, from L2
    CUtensorMap tc = tb;
    a.spill_tma = (sample && lm::encode_f32_rows(&tc, a.spill, M, V)) ? 1 : 0;  // V % 4 == 0 here
    a.partials = reinterpret_cast<float2 *>(w + 256);
    a.status = reinterpret_cast<uint32_t *>(w);
    a.wait_budget = wait_budget();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    prof_begin(s);
    if (sample) lm::launch_gemm_bn<true>(bn, ta, tb, tc, a, grid, s);
    else lm::launch_gemm_bn<false>(bn, ta, tb, tc, a, grid, s);
    prof_end(s);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(M);
    cfg.blockDim = dim3(lm::kDraftThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = sample ? cudaLaunchKernelEx(&cfg, lm::draft_finish_kernel<true>, q_out,
                                                      static_cast<const float2 *>(a.partials), grid, V, a.c, seed,
                                                      offset, x_out, u_out)
                                 : cudaLaunchKernelEx(&cfg, lm::draft_finish_kernel<false>, q_out,
                                                      static_cast<const float2 *>(a.partials), grid, V, a.c, seed,
                                                      offset, x_out, u_out);
    set_launches(2);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" sv_status spec_lmhead_logits(const void *hidden, const void *w_vocab_t, int d, int M, int V,
                                        float *logits, void *ws, size_t ws_bytes, void *stream) {
    if (M < 0 || M > lm::BM || V <= 0 || d < lm::BK || d % lm::BK != 0) return SV_ERR_INVALID;
    if (M == 0) {
        set_launches(0);
        return SV_OK;
    }
    if (!hidden || !w_vocab_t || !logits || !ws) return SV_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(hidden) & 15u) || (reinterpret_cast<uintptr_t>(w_vocab_t) & 15u) ||
        (reinterpret_cast<uintptr_t>(logits) & 15u))
        return SV_ERR_INVALID;
    if (ws_bytes < spec_draft_workspace_size(M, d, V) || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return SV_ERR_WORKSPACE;
    const int bn = lm::choose_bn(V, sm_count());
    const int n_tiles = (V + bn - 1) / bn;
    int grid = n_tiles < sm_count() ? n_tiles : sm_count();
    if (grid > lm::kMaxLmGrid) grid = lm::kMaxLmGrid;
    CUtensorMap ta, tb;
    if (!lm::encode_bf16_kmajor(&ta, hidden, M, d, lm::BM) || !lm::encode_bf16_kmajor(&tb, w_vocab_t, V, d, bn))
        return SV_ERR_CUDA;
    char *w = static_cast<char *>(ws);
    lm::LmArgs a;
    a.M = M;
    a.d = d;
    a.V = V;
    a.n_tiles = n_tiles;
    a.c = 1.4426950408889634f;  // the row partials it also writes are those of T = 1 (unused here)
    a.spill = logits;
    a.spill_keep = 0;
    CUtensorMap tc = tb;
    a.spill_tma = (V % 4 == 0 && lm::encode_f32_rows(&tc, logits, M, V)) ? 1 : 0;
    a.partials = reinterpret_cast<float2 *>(w + 256);
    a.status = reinterpret_cast<uint32_t *>(w);
    a.wait_budget = wait_budget();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    prof_begin(s);
    lm::launch_gemm_bn<true>(bn, ta, tb, tc, a, grid, s);
    prof_end(s);
    set_launches(1);
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
