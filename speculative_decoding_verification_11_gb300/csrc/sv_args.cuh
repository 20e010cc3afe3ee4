// Arguments of the verification kernels and the limits of the cluster path,
// shared by the translation units that launch them (verify.cu, cluster.cu).
#pragma once
#include <cstddef>
#include <cstdint>

#include "sv_device.cuh"  // kSegElems

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
    int B, K, V, rows, n_chunks, n_tiles, n_draft;
    float c;  // log2(e) / T
    // workspace
    uint32_t *status;
    const int *csr_ok;
    uint32_t *tickets1;
    uint32_t *sched;     // fused kernel: [0] next stats block, [1] CTAs done, [2] next residual block
    Decision *dec;
    float2 *partials;
    float *tile_mass;
    // fused kernel records (zero until written, zeroed again by their reader)
    uint64_t *fpart;     // per row: one partial per stats block and consumer warp (n_pe words)
    uint64_t *fdec;      // per request: the decision, two words
    uint32_t *fmass;     // per request: residual mass of each 256-token segment (n_seg words)
    int n_pe;            // partial records per row
    int n_seg;           // 256-token segments per row
    int n_rb;            // residual blocks per row
    int keep_rows;       // fused kernel: leading rows per request kept in L2 for the residual pass
    int n_st;            // fused kernel: residual stages per row
    int tail_b0;         // fused kernel: requests from here on take one-stage residual claims
    int early_res;       // fused kernel: residual claims may start during the stats stream
    float *cv_segs;      // cluster kernel: per request, one residual sum per 256-token segment
    long long wait_budget;  // SM cycles a wait on other warps' or CTAs' work may take
};

// Two kinds of bounded waits.  A wait on work that other warps or CTAs
// produce (a ring stage, a partial, a decision, a segment mass) gives up after
// Args::wait_budget SM cycles (spec_set_wait_budget; default kDefaultWaitBudget,
// ~2 s at 2 GHz), then flags SV_FLAG_TIMEOUT and leaves.  A wait on the CTA's
// own copies or MMAs, before it leaves or releases what they write, always
// allows kDrainBudget: those complete by themselves in microseconds, and a CTA
// may not leave while a copy into its shared memory is still landing, however
// short the other budget is set.
constexpr long long kDefaultWaitBudget = 4000000000ll;
constexpr long long kDrainBudget = 4000000000ll;

__device__ __forceinline__ void request_rows(const Args &a, int b, int &r0, int &nr) {
    if (a.row_offsets) {
        r0 = __ldg(a.row_offsets + b);
        nr = __ldg(a.row_offsets + b + 1) - r0;
    } else {
        r0 = b * (a.K + 1);
        nr = a.K + 1;
    }
}

namespace cv {

// One cluster of kC CTAs per request (cluster.cu).
constexpr int kC = 8;                          // CTAs per request
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRows = 16;                   // rows per request (K <= 15)
constexpr int kMaxSegs = 64;                   // segments per CTA: V <= kC x 64 x 256 = 131072
constexpr int kQBatch = 4;                     // segments whose q loads a warp holds in flight
constexpr size_t kSmemCap = 100 * 1024;        // row slices per CTA: two CTAs per SM
constexpr int kMaxB = 64;                      // batches the workspace keeps segment sums for

__host__ __device__ constexpr int segs_per_cta(int V) {
    return ((V + kSegElems - 1) / kSegElems + kC - 1) / kC;
}
__host__ __device__ constexpr size_t smem_bytes(int nr_cap, int V, int esize) {
    return static_cast<size_t>(nr_cap) * segs_per_cta(V) * kSegElems * esize;
}

}  // namespace cv

namespace sk {

// One CTA per request, the request's rows in shared memory (small.cu).
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr size_t kDefaultRowBytes = 48 * 1024;
constexpr size_t kMaxSmemBytes = 200 * 1024;  // largest dynamic shared memory a launch may ask for

__host__ __device__ constexpr size_t a16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

// Dynamic shared memory: rows (nr_cap x V elements) | row normalisers (8 B
// per row) | residual row (4 B per token) | per-thread sums (8 B per thread).
__host__ __device__ constexpr size_t smem_bytes(int nr_cap, int V, int esize) {
    return a16(static_cast<size_t>(nr_cap) * V * esize) + a16(static_cast<size_t>(nr_cap) * 8) +
           a16(static_cast<size_t>(V) * 4) + kThreads * 8;
}

}  // namespace sk

}  // namespace sv
