/*
 * Plain fp64 oracle of the speculative-decoding verification step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference that the
 * CUDA library is compared against.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it; the product path never does.
 * It shares no code, header or constant with the CUDA sources.
 *
 * Every step is written out in the order the pages give it, in fp64, one token
 * at a time, with no blocking or reordering:
 *
 *   p = softmax(z / T)          target probabilities (temperature divides the
 *                               logits; "Speculative Decoding" glossary,
 *                               "Mathematical Guarantee": T = 0 is greedy)
 *   accept x_j iff u_j <= min(1, p_j(x_j) / q_j(x_j)), evaluated as
 *   u_j * q_j(x_j) <= p_j(x_j)  ("Speculative Decoding in Large Language
 *                               Models", section 2 "Modified Rejection Sampling")
 *   stop at the first rejection ("Co-Designing AI Models Using Speculative
 *                               Decoding", "What is speculative decoding?")
 *   correction token ~ max(0, p - q) / sum max(0, p - q) at the rejected
 *                               position (same section 2, residual p'(x))
 *   bonus token ~ p at position K when every draft is accepted (the target
 *                               always yields one more token: AL in [1, 1+D])
 *   greedy: accept while x_j == argmax_j, then emit argmax at the stop.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - tokens are sampled by inverse CDF in ascending token index with one
 *     final uniform u_K per request: the smallest v with C(v) > u_K * R; if
 *     rounding leaves no such v, the largest v with r(v) > 0;
 *   - if R = 0 after a rejection (possible only through rounding), the token
 *     is drawn from p instead and the event is flagged;
 *   - greedy ties break to the lowest index;
 *   - a drafted id outside [0, V) invalidates its request: AL = 0, all -1.
 *
 * Near ties (decisions the parity rule lets differ) are flagged here in fp64:
 *   accept test: q > 0 and |u - p/q| < band + e_p p/q;
 *   final sample: a CDF boundary C(v)/R within band + 2 E / (R - E) of u
 *                 (every boundary is a near tie when E >= R);
 * band = 1e-6 unless the caller passes another.  e_p (per draft slot: a bound
 * on the relative error of p at the drafted token) and E (per logits row: a
 * bound on the absolute error of the row's probability masses, which bounds
 * the error of C and R alike) are zero unless the caller passes them: the
 * fused LM-head path does, from the error bound of its GEMM's fp32
 * accumulation.  Since the compared quantity p/q then carries a relative error
 * of at most e_p, and C and R an absolute one of at most E, the GPU's decision
 * can differ from the fp64 one only inside these bands.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_BF16 1
#define OR_F64 2

#define NEAR_TIE_DEFAULT 1e-6

/* Read element i of a logits buffer as fp64 (bf16 and fp32 decode exactly). */
static double logit_at(const void *base, int dtype, int64_t i)
{
    if (dtype == OR_F32)
        return (double)((const float *)base)[i];
    if (dtype == OR_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return ((const double *)base)[i];
}

/* Start of row j of a (rows x V) logits buffer. */
static const void *row_ptr(const void *z, int dtype, int64_t j, int64_t V)
{
    size_t esize = (dtype == OR_F32) ? 4 : (dtype == OR_BF16) ? 2 : 8;
    return (const char *)z + (size_t)j * (size_t)V * esize;
}

/* p(v) = exp(z(v)/T - m) / sum_w exp(z(w)/T - m), m = max_w z(w)/T. */
void oracle_softmax_row(const void *z, int dtype, int64_t V, double T, double *p)
{
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        double y = logit_at(z, dtype, v) / T;
        if (y > m)
            m = y;
    }
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        p[v] = exp(logit_at(z, dtype, v) / T - m);
        s += p[v];
    }
    for (int64_t v = 0; v < V; ++v)
        p[v] /= s;
}

/* Index of the largest logit; the first one on ties. */
int64_t oracle_argmax_row(const void *z, int dtype, int64_t V)
{
    int64_t best = 0;
    double bv = logit_at(z, dtype, 0);
    for (int64_t v = 1; v < V; ++v) {
        double y = logit_at(z, dtype, v);
        if (y > bv) {
            bv = y;
            best = v;
        }
    }
    return best;
}

/*
 * Verify one request with K drafted tokens.
 *   z     : (K+1) x V target logits of this request (row j = position j)
 *   q     : K x V draft probabilities (unused when greedy)
 *   x     : K drafted ids
 *   u     : K+1 uniforms: u[j] for the accept test at j < K, u[K] final draw
 *   out   : K+1 emitted ids, -1 past AL
 *   al    : accepted length AL = k* + 1 (0 for an invalid request)
 *   p_draft: K values p_j(x_j) (NAN where not evaluated)
 *   req   : 2 values: residual mass R of the sampled row, r(v*)/R
 *   flags : 3 values: near-tie accept count, near-tie final-sample flag,
 *           zero-residual flag
 *   work  : 2 V doubles of scratch
 *   p_rel_err  : K values (may be NULL = 0): bound on the relative error of
 *                the compared p_j(x_j)
 *   mass_err   : K+1 values (may be NULL = 0): bound on the absolute error of
 *                the probability masses of row j
 * Returns 0, or 1 when a drafted id is out of range.
 */
int oracle_verify_request(const void *z, int zdtype, const float *q, const int32_t *x,
                          const float *u, int K, int64_t V, double T, int greedy,
                          int32_t *out, int32_t *al, double *p_draft, double *req,
                          int32_t *flags, double *work, double tie_band,
                          const double *p_rel_err, const double *mass_err)
{
    for (int j = 0; j <= K; ++j)
        out[j] = -1;
    for (int j = 0; j < K; ++j)
        p_draft[j] = NAN;
    req[0] = NAN;
    req[1] = NAN;
    flags[0] = flags[1] = flags[2] = 0;
    for (int j = 0; j < K; ++j) {
        if (x[j] < 0 || (int64_t)x[j] >= V) {
            *al = 0;
            return 1;
        }
    }

    if (greedy) {
        int kstar = K;
        for (int j = 0; j < K; ++j) {
            if ((int64_t)x[j] != oracle_argmax_row(row_ptr(z, zdtype, j, V), zdtype, V)) {
                kstar = j;
                break;
            }
            out[j] = x[j];
        }
        out[kstar] = (int32_t)oracle_argmax_row(row_ptr(z, zdtype, kstar, V), zdtype, V);
        *al = kstar + 1;
        return 0;
    }

    double *p = work;
    double *r = work + V;
    int kstar = K;
    for (int j = 0; j < K; ++j) {
        oracle_softmax_row(row_ptr(z, zdtype, j, V), zdtype, V, T, p);
        double pj = p[x[j]];
        double qj = (double)q[(int64_t)j * V + x[j]];
        double uj = (double)u[j];
        p_draft[j] = pj;
        double ep = p_rel_err ? p_rel_err[j] : 0.0;
        if (qj > 0.0 && fabs(uj - pj / qj) < tie_band + ep * (pj / qj))
            flags[0] += 1;
        if (!(uj * qj <= pj)) {
            kstar = j;
            break;
        }
        out[j] = x[j];
    }

    if (kstar == K) {
        /* bonus: r = p at position K */
        oracle_softmax_row(row_ptr(z, zdtype, K, V), zdtype, V, T, p);
        for (int64_t v = 0; v < V; ++v)
            r[v] = p[v];
    } else {
        /* correction: r = max(0, p - q) at the rejected position; p still holds p_k* */
        const float *qk = q + (int64_t)kstar * V;
        for (int64_t v = 0; v < V; ++v) {
            double d = p[v] - (double)qk[v];
            r[v] = d > 0.0 ? d : 0.0;
        }
    }
    double R = 0.0;
    for (int64_t v = 0; v < V; ++v)
        R += r[v];
    if (R == 0.0) {
        for (int64_t v = 0; v < V; ++v)
            r[v] = p[v];
        R = 0.0;
        for (int64_t v = 0; v < V; ++v)
            R += r[v];
        flags[2] = 1;
    }

    double E = mass_err ? mass_err[kstar] : 0.0;
    double band = E < R ? tie_band + 2.0 * E / (R - E) : INFINITY;
    double ufin = (double)u[K];
    double t = ufin * R;
    double C = 0.0, Cprev = 0.0;
    int64_t vstar = -1;
    for (int64_t v = 0; v < V; ++v) {
        Cprev = C;
        C += r[v];
        if (C > t) {
            vstar = v;
            break;
        }
    }
    if (vstar < 0) {
        for (int64_t v = V - 1; v >= 0; --v) {
            if (r[v] > 0.0) {
                vstar = v;
                break;
            }
        }
        flags[1] = 1;
    } else if (ufin - Cprev / R < band || C / R - ufin < band) {
        flags[1] = 1;
    }
    out[kstar] = (int32_t)vstar;
    req[0] = R;
    req[1] = r[vstar] / R;
    *al = kstar + 1;
    return 0;
}

/*
 * Verify B requests laid out by CSR row offsets (fixed K is the special case
 * row_offsets[b] = b (K+1)).  Request b owns logits rows / uniforms / output
 * slots row_offsets[b] .. row_offsets[b+1]-1 and draft ids / q rows
 * row_offsets[b]-b .. row_offsets[b+1]-b-2.
 *   p_draft : (rows - B) values, req : 2 B values, flags : 3 B values.
 *   p_rel_err : (rows - B) values, mass_err : rows values (either may be NULL),
 *               the error bounds of oracle_verify_request laid out like the
 *               draft slots and the logits rows.
 * Returns -1 for malformed offsets, else the number of invalid requests.
 */
int oracle_verify_batch(const void *logits, int zdtype, const float *q,
                        const int32_t *row_offsets, int B, int64_t V, double T, int greedy,
                        const int32_t *draft, const float *uniforms, int32_t *out_tokens,
                        int32_t *accept_len, double *p_draft, double *req, int32_t *flags,
                        double tie_band, const double *p_rel_err, const double *mass_err)
{
    if (!(tie_band > 0.0))
        tie_band = NEAR_TIE_DEFAULT;
    if (row_offsets[0] != 0)
        return -1;
    for (int b = 0; b < B; ++b)
        if (row_offsets[b + 1] < row_offsets[b] + 1)
            return -1;
    double *work = (double *)malloc(sizeof(double) * 2 * (size_t)V);
    if (!work)
        return -1;
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        int64_t r0 = row_offsets[b];
        int K = (int)(row_offsets[b + 1] - r0 - 1);
        int64_t d0 = r0 - b;
        const void *z = row_ptr(logits, zdtype, r0, V);
        const float *qb = q ? q + d0 * V : NULL;
        const float *ub = uniforms ? uniforms + r0 : NULL;
        float dummy_u[1] = {0.5f};
        bad += oracle_verify_request(z, zdtype, qb, draft + d0, ub ? ub : dummy_u, K, V, T,
                                     greedy, out_tokens + r0, accept_len + b, p_draft + d0,
                                     req + 2 * b, flags + 3 * b, work, tie_band,
                                     p_rel_err ? p_rel_err + d0 : NULL, mass_err ? mass_err + r0 : NULL);
    }
    free(work);
    return bad;
}

/* ------------------------------------------------------------------------
 * Draft-side sampling (the step before verification: q and x for the drafted
 * positions; the proof of "Speculative Decoding in Large Language Models",
 * section 2, assumes x ~ q).  The uniforms are drawn, not passed in, so this
 * side has its own counter-based generator, written from its published
 * definition: Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3", SC 2011): ten rounds of two 32x32 -> 64-bit
 * products with multipliers 0xD2511F53 and 0xCD9E8D57, the key bumped by the
 * Weyl constants 0x9E3779B9 and 0xBB67AE85 between rounds.
 * ---------------------------------------------------------------------- */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/*
 * The uniform of draw `index` of stream `stream` under `seed` (the reading
 * used on both sides): counter (index low word, stream, index high word, 0),
 * key (seed low word, seed high word); u = ((w0 >> 9) + 1/2) 2^-23, in (0, 1).
 */
double oracle_philox_uniform(uint64_t seed, uint64_t index, uint32_t stream)
{
    uint32_t ctr[4] = {(uint32_t)index, stream, (uint32_t)(index >> 32), 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return ((double)(out[0] >> 9) + 0.5) * 0x1p-23;
}

/*
 * Inverse CDF in ascending index over weights r >= 0: the smallest v with
 * C(v) > u R (R = sum of r); if rounding leaves none, the largest v with
 * r(v) > 0.  *near_tie = 1 when a boundary C(v)/R lies within `band` of u.
 */
int64_t oracle_draw_inverse_cdf(const double *r, int64_t V, double u, double band, int *near_tie)
{
    double R = 0.0;
    for (int64_t v = 0; v < V; ++v)
        R += r[v];
    double t = u * R, C = 0.0, Cprev = 0.0;
    *near_tie = 0;
    for (int64_t v = 0; v < V; ++v) {
        Cprev = C;
        C += r[v];
        if (C > t) {
            if (u - Cprev / R < band || C / R - u < band)
                *near_tie = 1;
            return v;
        }
    }
    *near_tie = 1;
    for (int64_t v = V - 1; v >= 0; --v)
        if (r[v] > 0.0)
            return v;
    return -1;
}
