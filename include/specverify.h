/*
 * specverify: target-side verification step of speculative decoding on one
 * GB300 (sm_103a).  C ABI of libspecverify.so.
 *
 * The operation (every entry point computes some part of it):
 *   Given target logits z for B requests x (K+1) positions over a vocabulary
 *   of V tokens, draft probabilities q for the K drafted positions, the
 *   drafted ids x_0..x_{K-1} and uniforms u_0..u_K of each request:
 *     p_j = softmax(z_j / T)                       ("Speculative Decoding"
 *           glossary, "Mathematical Guarantee"; T = 0 selects greedy)
 *     accept x_j iff u_j <= min(1, p_j(x_j) / q_j(x_j)), evaluated as
 *           u_j * q_j(x_j) <= p_j(x_j)              ("Speculative Decoding in
 *           Large Language Models", section 2, "Modified Rejection Sampling")
 *     k* = the first rejected position, or K        ("Co-Designing AI Models
 *           Using Speculative Decoding", "What is speculative decoding?")
 *     emit x_0..x_{k*-1}, then one token drawn with the final uniform u_K from
 *           max(0, p_k* - q_k*) / sum max(0, p_k* - q_k*) when k* < K
 *           (section 2, residual p'(x)), or from p_K when every draft was
 *           accepted (the target always produces one more token, so the
 *           accepted length AL = k* + 1 lies in [1, 1 + K]).
 *   Greedy mode accepts while x_j == argmax_v z_j(v) (lowest index on ties)
 *   and emits argmax z_k* at the stop; its output equals plain argmax
 *   decoding ("Co-Designing...", "What is speculative decoding?").
 *   The draw from a distribution r is an inverse CDF in ascending token
 *   index: the smallest v with sum_{w<=v} r(w) > u_K * sum_w r(w); if rounding
 *   leaves none, the largest v with r(v) > 0.  If the residual is empty after
 *   a rejection (only possible through rounding) the draw uses p_k* instead
 *   and the device status word records it (SV_FLAG_ZERO_RESIDUAL).
 *
 * Conventions shared by every entry point:
 *   - Every data pointer is caller-owned DEVICE memory, row-major, densely
 *     packed.  The library never allocates device or host memory on these
 *     paths and keeps no per-call state outside the caller's workspace.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are stream-ordered and asynchronous; nothing
 *     synchronises the host except spec_verify_last_device_status().
 *   - Argument errors are detected on the host before any launch and return
 *     SV_ERR_INVALID (bad sizes, null pointers, T <= 0 in sampling mode,
 *     K > SV_MAX_K) or SV_ERR_WORKSPACE; nothing is launched then.
 *   - Input errors only the device can see (a drafted id outside [0, V),
 *     malformed CSR offsets) set bits of a status word kept in the workspace;
 *     the affected request gets AL = 0 and all its output slots -1, the others
 *     are unaffected (malformed CSR offsets invalidate every request of the
 *     call).  The word accumulates over calls until
 *     spec_verify_last_device_status() reads and clears it.
 *     No kernel traps.
 *   - Layout of a request b with K_b drafts and first logits row r_b:
 *       logits rows r_b .. r_b + K_b            (position j = row r_b + j)
 *       q rows / draft ids  r_b - b .. r_b - b + K_b - 1
 *       uniforms, out_tokens  r_b .. r_b + K_b  (u_j, j < K_b accept draws;
 *                                                u_{K_b} the final draw)
 *     Fixed-K calls use r_b = b (K+1).  Output slots past AL hold -1.
 *   - A workspace may not be shared by calls that overlap on the device.
 *     Zero-fill it once before its first use (cudaMemsetAsync).  After that
 *     it serves calls of any shape in turn: every call that completes leaves
 *     its per-request counters at zero (a call that reported SV_ERR_TIMEOUT
 *     may not: zero-fill the workspace again after one).
 *   - `diag` (may be NULL) receives per-token diagnostics in fp32:
 *       diag[i], i < Nq = rows - B : p_j(x_j) of draft slot i
 *       diag[Nq + 2b]              : mass R of the distribution the final
 *                                    token of request b was drawn from
 *       diag[Nq + 2b + 1]          : r(v*) / R, the probability of the token
 *                                    that was drawn
 *     In greedy mode diag is ignored.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sv_status {
    SV_OK = 0,
    SV_ERR_INVALID = 1,      /* bad argument, found on the host; nothing launched */
    SV_ERR_CUDA = 2,         /* a CUDA runtime call or launch failed */
    SV_ERR_DEVICE_INPUT = 3, /* device-detected input error (status word) */
    SV_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up */
    SV_ERR_WORKSPACE = 5     /* workspace too small or not 256-byte aligned */
} sv_status;

typedef enum sv_dtype { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* Bits of the device status word. */
#define SV_FLAG_BAD_TOKEN 0x1u      /* a drafted id outside [0, V) */
#define SV_FLAG_BAD_OFFSETS 0x2u    /* CSR offsets not increasing, or K_b > SV_MAX_K */
#define SV_FLAG_ZERO_RESIDUAL 0x4u  /* informational: a draw fell back to p */
#define SV_FLAG_TIMEOUT 0x8u        /* a bounded wait expired */
#define SV_FLAG_KV_OUT_OF_BLOCKS 0x10u  /* spec_kv_reserve: the free list is short */
#define SV_FLAG_KV_BAD_INPUT 0x20u      /* spec_kv_reserve / _rollback: an input breaks a rule */

/* Largest number of drafted tokens per request. */
#define SV_MAX_K 255

/*
 * Bytes of workspace a call over B requests, `rows` logits rows in total
 * (B (K+1) for fixed K) and vocabulary V needs.  Pure host function.
 */
size_t spec_verify_workspace_size(int B, int rows, int V);

/*
 * Greedy verification ("Co-Designing...", "What is speculative decoding?").
 *   logits     (B (K+1)) x V, dtype dt
 *   draft      B K int32 ids
 *   out_tokens B (K+1) int32;  accept_len  B int32 (AL per request)
 *   ws         spec_verify_workspace_size(B, B (K+1), V) bytes, 256-aligned
 * Bit-exact: argmax is taken on the logits as stored, ties to the lowest id.
 */
sv_status spec_verify_greedy(const void *logits, sv_dtype dt, int B, int K, int V,
                             const int32_t *draft, int32_t *out_tokens, int32_t *accept_len,
                             void *ws, size_t ws_bytes, void *stream);

/*
 * Sampling verification ("Speculative Decoding in Large Language Models",
 * section 2 "Modified Rejection Sampling"; the glossary's "Mathematical
 * Guarantee"; "Speculative Decoding in Production: Accelerating LLM
 * Inference via Custom Draft Models", "Speculative Decoding Mechanics", the
 * equations for alpha and P').
 *   logits      (B (K+1)) x V, dtype dt;   q  (B K) x V fp32 (already tempered)
 *   temperature T > 0;  draft B K int32;  uniforms B (K+1) fp32 in (0, 1)
 *   out_tokens  B (K+1) int32;  accept_len B int32;  diag see above
 */
sv_status spec_verify_sample(const void *logits, sv_dtype dt, const float *q, int B, int K,
                             int V, float temperature, const int32_t *draft,
                             const float *uniforms, int32_t *out_tokens, int32_t *accept_len,
                             float *diag, void *ws, size_t ws_bytes, void *stream);

/*
 * Per-request draft lengths K_b ("Hardware Aware Dynamic Speculative
 * Decoding": K chosen per batch at run time), given as CSR row offsets.
 *   row_offsets B+1 int32 on the device: row_offsets[0] = 0,
 *               row_offsets[b+1] - row_offsets[b] = K_b + 1 in [1, SV_MAX_K+1]
 *   rows        row_offsets[B] (the caller's host-side copy of it; the device
 *               checks that they agree)
 *   logits rows x V;  q (rows - B) x V fp32;  draft rows - B;  uniforms rows;
 *   out_tokens rows;  accept_len B.   temperature 0 = greedy (q, uniforms,
 *   diag then unused), else sampling.
 */
sv_status spec_verify_ragged(const void *logits, sv_dtype dt, const float *q,
                             const int32_t *row_offsets, int B, int rows, int V,
                             float temperature, const int32_t *draft, const float *uniforms,
                             int32_t *out_tokens, int32_t *accept_len, float *diag, void *ws,
                             size_t ws_bytes, void *stream);

/*
 * Bytes of workspace spec_lmhead_verify needs for M = B (K+1) rows, hidden
 * size d and vocabulary V (it includes an fp32 M x V spill of the tile
 * logits that only the selected rows are read back from).
 */
size_t spec_lmhead_workspace_size(int B, int K, int d, int V);

/*
 * Fused LM-head front end + verification.  The target logits are the
 * product z = hidden . W_vocab (bf16 operands, fp32 accumulation on the
 * tensor cores) and feed the verifier tile by tile; this is the GEMM whose M
 * grows from B to B (1 + D) under speculation ("Co-Designing...", Guideline 1).
 *   hidden     M x d bf16, row-major, 16-byte aligned; M = B (K+1) <= 128,
 *              d a multiple of 64
 *   w_vocab_t  V x d bf16, 16-byte aligned: W_vocab stored transposed (row
 *              v = the d weights of token v, the layout of a Linear layer's
 *              weight); any V >= 1
 *   q, draft, uniforms, out_tokens, accept_len, diag as in spec_verify_sample
 *   temperature 0 = greedy, else sampling
 *   ws         spec_lmhead_workspace_size(B, K, d, V) bytes, 256-byte aligned
 * Two launches when V is a multiple of 4, V <= 196608 and q (if used) is
 * 16-byte aligned: the GEMM, then one cluster of CTAs per request that
 * reads back only the selected rows of the spill.  Otherwise the GEMM is
 * followed by the finish of the unaligned verification path: decide, then
 * in sampling mode the residual draw (two or three launches in all).
 * Argument errors (M > 128, d not a multiple of 64, a misaligned operand,
 * T < 0 or not finite, K > SV_MAX_K) return SV_ERR_INVALID, and a short or
 * misaligned workspace SV_ERR_WORKSPACE, before any launch.
 */
sv_status spec_lmhead_verify(const void *hidden, const void *w_vocab_t, int d, const float *q,
                             int B, int K, int V, float temperature, const int32_t *draft,
                             const float *uniforms, int32_t *out_tokens, int32_t *accept_len,
                             float *diag, void *ws, size_t ws_bytes, void *stream);

/*
 * Draft side, the step before verification: q = softmax(h . W / T) over the
 * vocabulary and one drafted token x ~ q per row ("Speculative Decoding in
 * Large Language Models", section 2: the draft proposes x ~ q, which the
 * verification's law assumes; a draft head is read as one linear layer over
 * the vocabulary).  The logits come from the same tcgen05 GEMM as
 * spec_lmhead_verify and are written into q_out, which a second kernel turns
 * into q in place; x is the smallest v with sum_{w<=v} q(w) > u sum_w q(w),
 * else (rounding) the largest v with q(v) > 0.
 *   hidden     M x d bf16, row-major, 16-byte aligned; 1 <= M <= 128
 *   w_vocab_t  V x d bf16 (row v = the weights of token v), 16-byte aligned;
 *              d a multiple of 64; V a multiple of 4, V <= 1048576
 *   temperature > 0: sampling (q_out required, 16-byte aligned, M x V fp32);
 *              0: greedy drafting, x = argmax (lowest index on ties), q_out
 *              may be NULL and is not written
 *   seed, offset: row r draws the uniform of Philox4x32-10 (Salmon et al.,
 *              SC 2011) at counter (offset + r low word, 1, offset + r high
 *              word, 0) and key (seed low word, seed high word): u = ((w0 >>
 *              9) + 1/2) 2^-23, w0 its first output word; u_out (M, may be
 *              NULL) receives it
 *   x_out      M int32
 *   ws         spec_draft_workspace_size(M, d, V) bytes, 256-byte aligned
 * Two kernels on `stream`; argument errors return before any launch.
 */
size_t spec_draft_workspace_size(int M, int d, int V);
sv_status spec_draft_sample(const void *hidden, const void *w_vocab_t, int d, int M, int V,
                            float temperature, uint64_t seed, uint64_t offset, float *q_out,
                            int32_t *x_out, float *u_out, void *ws, size_t ws_bytes, void *stream);

/*
 * The LM-head projection alone: logits = hidden . W_vocab in fp32, from the
 * same tcgen05 GEMM (bf16 operands, fp32 accumulation in tensor memory over
 * the hidden size in ascending order, 16 products per step) that feeds
 * spec_lmhead_verify and spec_draft_sample ("Co-Designing AI Models Using
 * Speculative Decoding for Faster LLM Inference", Guideline 1: the target's
 * LM-head GEMM whose M grows from B to B (1 + D) under speculation).  For
 * callers that want the target's logits themselves, e.g. to verify through
 * spec_verify_sample, or to check the contraction on its own.
 *   hidden     M x d bf16, row-major, 16-byte aligned; 1 <= M <= 128,
 *              d a multiple of 64
 *   w_vocab_t  V x d bf16 (row v = the weights of token v), 16-byte aligned
 *   logits     M x V fp32, row-major, 16-byte aligned (written)
 *   ws         spec_draft_workspace_size(M, d, V) bytes, 256-byte aligned
 * One kernel on `stream`; argument errors return before any launch.
 */
sv_status spec_lmhead_logits(const void *hidden, const void *w_vocab_t, int d, int M, int V, float *logits,
                             void *ws, size_t ws_bytes, void *stream);

/*
 * Model-free n-gram (prompt lookup) drafter ("Co-Designing AI Models Using
 * Speculative Decoding for Faster LLM Inference", Table 1: suffix / n-gram
 * drafting matches strings over the token stream, no model, one lookup).
 * Request b's context is tokens[ctx_offsets[b] .. ctx_offsets[b+1]) (int32,
 * CSR, device; `tokens` 4-byte aligned, else SV_ERR_INVALID).  For n = n_max down to n_min, the context's last n tokens are
 * looked up among earlier windows that end before its last token; at the
 * first n with a match, the latest such window wins and the up to K tokens
 * that follow it are proposed (fewer when the context ends first).  Outputs:
 * draft_out [B x K] int32 (-1 past the proposal), k_out [B] (0..K: the draft
 * length each request proposes, e.g. the K_b of spec_verify_ragged).
 * 1 <= n_min <= n_max <= 32, 0 <= K <= SV_MAX_K.  One kernel on `stream`; a
 * request whose offsets decrease, or whose first offset is negative, proposes
 * nothing and reads no token.  Offsets past the end of `tokens` are not
 * detected (the buffer's length is not passed): the caller keeps them in range.
 */
sv_status spec_ngram_draft(const int32_t *tokens, const int32_t *ctx_offsets, int B, int K, int n_min,
                           int n_max, int32_t *draft_out, int32_t *k_out, void *stream);

/*
 * Dynamic draft length after verification ("Hardware Aware Dynamic
 * Speculative Decoding", section "Dynamic speculative decoding": K adapted to
 * acceptance and hardware, goodput = AL / ITL, a table extended with live
 * statistics; "Speculative Decoding in
 * Production: Accelerating LLM Inference via Custom Draft Models", "Production
 * Failure Modes and Mitigation Strategies", item 1: K from 5 down to 1 or 2
 * when the average accepted length over the last 10 falls below 1.5).
 * Per request b (device arrays owned by the caller, zero-filled before the
 * first call): hist [B x W x 2] int32 = a ring of its last W results
 * (AL, K used), count [B] = results pushed so far.  Each call pushes
 * (accept_len[b], k_used[b]) unless accept_len[b] = 0 (an invalid request),
 * then writes k_next[b]:
 *   SV_DYNK_WINDOW   k_low if the mean AL over the ring is below `threshold`,
 *                    else k_high (k_high while the ring is empty);
 *   SV_DYNK_GOODPUT  alpha = S / (S + F) over the ring, S = sum (AL - 1),
 *                    F = results with AL - 1 < K (alpha_prior when S + F = 0);
 *                    E(K) = 1 + alpha + ... + alpha^K; k_next = the K in
 *                    [k_low, k_high] maximising E(K) / itl[K] (smaller K on
 *                    ties), itl [k_high + 1] float = the caller's profiled
 *                    step time (draft + verify) with K drafts.
 * All decisions in fp32, round to nearest, in the order written.  If
 * row_offsets [B + 1] is not NULL it receives the CSR offsets of the next
 * ragged verification: row_offsets[b] = sum_{i<b} (k_next[i] + 1).
 * One kernel on `stream`.  0 <= k_low <= k_high <= SV_MAX_K, W >= 1.
 */
#define SV_DYNK_WINDOW 0
#define SV_DYNK_GOODPUT 1
sv_status spec_dynk_update(const int32_t *accept_len, const int32_t *k_used, int32_t *hist, int32_t *count,
                           int B, int W, int policy, float threshold, int k_low, int k_high,
                           const float *itl, float alpha_prior, int32_t *k_next, int32_t *row_offsets,
                           void *stream);

/*
 * spec_verify_sample for callers that cannot allocate device memory.  The
 * pages have no counterpart to this call; it exists for host programs with
 * no allocator to hand, e.g. a plugin inside an inference server whose
 * device memory is all held by the server's caching allocator, or a loop
 * that must not call cudaMalloc because it can synchronise the device.
 *   Arguments and results are those of spec_verify_sample without the
 *   workspace: the caller still passes inputs and outputs (device memory).
 *   Scratch is a fixed array of SV_NOALLOC_SCRATCH_BYTES inside this
 *   library, held on every GPU that loads it until the process exits.
 *   Returns SV_ERR_WORKSPACE when the call would need more than that
 *   (spec_verify_workspace_size(B, B (K+1), V) > SV_NOALLOC_SCRATCH_BYTES).
 *   The first call on each device looks up the array's device address with
 *   that device current; make that first call before any stream capture.
 *   Every call on a device shares the one array and clears the parts that
 *   must start at zero, so calls that overlap on the GPU race with each
 *   other: serialise them (one stream, or events).  Device-detected input
 *   errors show only as AL = 0 / -1 outputs; the status word cannot be read.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define SV_NOALLOC_SCRATCH_BYTES (2u << 20)
sv_status spec_verify_sample_noalloc(const void *logits, sv_dtype dt, const float *q, int B, int K, int V,
                                     float temperature, const int32_t *draft, const float *uniforms,
                                     int32_t *out_tokens, int32_t *accept_len, float *diag, void *stream);

/*
 * Synchronises `stream` and returns in *flags (SV_FLAG_* bits, may be NULL)
 * the device status word of workspace `ws` (the OR of every call since the
 * last read), then clears it.  Returns
 * SV_ERR_DEVICE_INPUT if an input-error bit was set, SV_ERR_TIMEOUT if the
 * timeout bit was set, SV_ERR_CUDA on a CUDA error, else SV_OK.
 */
sv_status spec_verify_last_device_status(void *ws, void *stream, uint32_t *flags);

/* Human-readable name of a status code (static storage). */
const char *spec_status_string(sv_status s);

/*
 * Profiling hook: when `begin` and `end` are non-NULL cudaEvent_t handles,
 * every later call records `begin` just before its dominant kernel (the
 * logits-streaming pass, or the LM-head GEMM) and `end` just after it, on the
 * call's stream.  Pass NULL, NULL to stop.  Process-wide; not thread-safe.
 */
sv_status spec_profile_set_events(void *begin, void *end);

/* Number of kernels the last call on this thread launched (for accounting). */
int spec_last_launch_count(void);

/*
 * Which verification kernel the last spec_verify_greedy / _sample / _ragged /
 * _sample_noalloc call on this thread chose: "small" (one CTA per request),
 * "cluster" (one cluster of CTAs per request), "stream" (the persistent
 * streaming kernel), "scalar" (rows not 16-byte aligned: element loads, two
 * passes), or "none" before any such call.  A static string; for accounting.
 */
const char *spec_last_kernel(void);

/*
 * Limit of the device-side waits, in SM clock cycles.  A kernel that waits on
 * work other warps or CTAs produce (a ring stage, a row partial, a decision, a
 * residual mass) gives up after `cycles` cycles from its start, sets
 * SV_FLAG_TIMEOUT in the call's status word (spec_verify_last_device_status
 * then returns SV_ERR_TIMEOUT), lets its own copies and MMAs in flight finish,
 * releases what it holds and returns; its outputs are then undefined, and the
 * workspace must be zero-filled again before its next use.  Waits on a CTA's
 * own copies and MMAs keep a fixed limit of the same default, whatever this
 * is set to.  cycles > 0 sets the limit, 0 restores the default (4e9 cycles,
 * about 2 s at 2 GHz); returns the previous value, or -1 (and changes
 * nothing) for cycles < 0.  Process-wide (an atomic), read by each call when
 * it launches.  For callers that bound their latency, and for tests of the
 * timeout path; the pages have no counterpart to it.
 */
long long spec_set_wait_budget(long long cycles);

/*
 * Kernel choice for small vocabularies.  A call of spec_verify_greedy,
 * spec_verify_sample, spec_verify_ragged or spec_verify_sample_noalloc whose
 * requests each hold at most `bytes` of logits ((rows per request) x V x
 * element size; for ragged calls the rows per request are bounded by
 * min(256, rows - B + 1)) runs one CTA per request with the request's rows in
 * shared memory; larger requests stream through one persistent kernel.  Both
 * compute the same step.  0 sends every call to the streaming kernel.
 * Default 49152.  Process-wide (an atomic); returns the previous value.  The
 * pages have no counterpart to it: it is a tuning knob of this library.
 */
size_t spec_set_small_kernel_limit(size_t bytes);

/*
 * Kernel choice for small batches of medium requests.  With `enable` non-zero
 * (the default), a call on 16-byte aligned rows (and q) that the small kernel
 * does not take runs one cluster of 8 CTAs per request when the request has
 * at most 16 rows, B <= 64, B x 8 CTAs fit twice over the GPU's SMs, V <=
 * 131072 and each CTA's slice of the request's rows fits in 100 KB of shared
 * memory; otherwise the call streams through the persistent kernel.  Both
 * compute the same step.  Process-wide (an atomic); returns the previous
 * setting (0 or 1).  A tuning knob of this library, like the one above.
 */
int spec_set_cluster_kernel(int enable);

/*
 * Paged KV-cache bookkeeping around verification ("Speculative Decoding in
 * Large Language Models", section 4, "Segmented Block Allocation
 * (PagedAttention)": fixed-size blocks, block pointers for the speculative
 * tokens, rejected positions return their pointers to the global free list
 * with no copy; "Speculative Decoding in Production: Accelerating LLM
 * Inference via Custom Draft Models", "Serving Architecture and KV Cache
 * Syncing": with M of K drafts accepted, K - M slots are evicted, in the
 * draft's cache and in the target's; call once per cache).
 *
 * A cache is, in device memory owned by the caller:
 *   block_table  int32 [B x max_blocks], row b = physical block ids of
 *                request b's logical blocks, -1 = no block;
 *   seq_len      int32 [B], tokens of request b with valid KV;
 *   free_ids     int32 [capacity], a stack of free block ids;
 *   free_count   int32 [1], entries of free_ids in use (its top).
 * Logical block i of a request holds positions [i bs, (i + 1) bs).
 * Both calls are one kernel on `stream`, stream-ordered and asynchronous,
 * touch block ids only (no KV data), and are deterministic.  A call whose
 * inputs break a rule changes nothing and ORs a flag into *status (a device
 * uint32 owned by the caller, zero until a flag is set); argument errors are
 * returned before any launch.
 */

/*
 * Blocks for the speculative slots: request b's table is extended to cover
 * positions [0, seq_len[b] + n_new[b]) (seq_len is not changed).  Blocks are
 * popped from the top of the stack; request 0 takes the lowest stack slots of
 * the popped range, each request its blocks in logical order.  If the stack
 * holds fewer blocks than the batch needs, nothing changes and
 * SV_FLAG_KV_OUT_OF_BLOCKS is set.  Rules: n_new >= 0, seq_len >= 0, the new
 * length fits the table, and the entries to fill hold no block (else
 * SV_FLAG_KV_BAD_INPUT).
 */
sv_status spec_kv_reserve(int32_t *block_table, const int32_t *seq_len, const int32_t *free_ids,
                          int32_t *free_count, const int32_t *n_new, int B, int max_blocks,
                          int block_size, uint32_t *status, void *stream);

/*
 * After verification: request b wrote n_spec[b] speculative slots after its
 * seq_len[b] valid ones; accept_len[b] (from a verification call: AL, or 0
 * for an invalid request) - 1 accepted drafts keep their KV, the final emitted
 * token gets its KV in the next step.  seq_len[b] += max(accept_len[b] - 1,
 * 0); the blocks wholly beyond the new length (logical blocks
 * ceil(new_len / bs) .. ceil((seq_len + n_spec) / bs) - 1) are pushed on the
 * stack in request order, each request's in logical order, and their table
 * entries set to -1.  Rules: counts >= 0, accept_len <= n_spec + 1, the
 * span fits the table, every entry to free holds a block, and the stack does
 * not overflow `capacity` (else SV_FLAG_KV_BAD_INPUT).
 */
sv_status spec_kv_rollback(int32_t *block_table, int32_t *seq_len, int32_t *free_ids,
                           int32_t *free_count, const int32_t *n_spec, const int32_t *accept_len,
                           int B, int max_blocks, int block_size, int capacity, uint32_t *status,
                           void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
