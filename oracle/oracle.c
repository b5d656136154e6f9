/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for the fused
 * MaxSim operator.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file; only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * Source: "FLASH-MAXSIM: IO-Aware Fused Kernels for Late-Interaction
 * Retrieval" (arXiv 2605.29517), abbreviated "Flash-MaxSim" below.
 *
 * Arithmetic: every floating-point dot product is a k-ascending sum of exact
 * double products (FP16/BF16 x FP16/BF16 products are exact in binary64);
 * maxima use a strict ">" scan in ascending token order, so the lowest token
 * index wins a tie; sums over query tokens run in ascending token order in
 * double.  INT8 work is done in int64.
 *
 * Readings of points the pages leave open (each repeated where it is used):
 *   R1  ties in the row maximum go to the lowest document-token index.
 *   R2  a document with zero tokens has row maximum -inf and argmax -1, so
 *       its score is -inf for a query with at least one token.
 *   R3  a query with zero valid tokens has score 0 (empty sum).
 *   R4  the argmax index is local to its document, in [0, Ld_b).
 *   R5  INT8 uses one symmetric scale per tensor (s_Q for Q, s_D for D); the
 *       score is fp32(raw * (s_Q * s_D)) evaluated in binary64 once at the
 *       end, where raw is the exact int64 sum of int32 row maxima.
 *   R6  INT8 with one scale per token (the per-token quantisation of
 *       Flash-MaxSim §4.3.1): the value ranked for query token i and document
 *       token t is the real product dot * s_D[t] of the exact integer dot
 *       product and the document token's scale, evaluated in binary64 (an
 *       integer below 2^24 times a binary32 scale is exact there); the row
 *       maximum and its lowest index are taken on those exact values, the
 *       query token's scale multiplies the maximum, and the sum over query
 *       tokens runs in binary64.
 *   R7  Chamfer distance (Flash-MaxSim §4.2 "Generalization to Chamfer
 *       Distance"): the squared Euclidean distance of a source point s and a
 *       target point t, evaluated in binary64 from the binary32 coordinates
 *       as (s.x - t.x)^2 + (s.y - t.y)^2 + (s.z - t.z)^2; the nearest target
 *       is the lowest index attaining the minimum; an empty target set gives
 *       +inf and index -1.  The means over points and the gradients are
 *       evaluated in binary64.  A mean over an empty set is 0.
 *
 * Parity status: every function here is pinned by CPU tests against closed
 * forms, invariants, brute force and finite differences (tests/test_oracle_*).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Storage decoding.  The kernels consume the stored 16-bit patterns; the     */
/* oracle evaluates the same patterns exactly in binary64.                    */
/* ------------------------------------------------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_binary16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                /* subnormal: f * 2^-24      */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25);  /* (1024 + f) * 2^(e-15-10) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32 pattern. */
static double decode_bfloat16(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* dtype: 0 = FP16, 1 = BF16.  Returns 0 on success, -1 on bad dtype. */
int oracle_decode(int dtype, const uint16_t *in, double *out, int64_t n)
{
    if (dtype != 0 && dtype != 1) return -1;
    for (int64_t k = 0; k < n; ++k)
        out[k] = dtype == 0 ? decode_binary16(in[k]) : decode_bfloat16(in[k]);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Forward: Flash-MaxSim §1 Eq. (1), score(Q,D) = sum_i max_j <Q_i, D_j>,     */
/* over the two regimes of §3.1 (one query vs B documents, or N_q x B).       */
/* Documents are packed token rows addressed by cu_seqlens (§4.3.2); queries  */
/* are padded to lq_max rows with q_lens valid.                               */
/* ------------------------------------------------------------------------- */

static double dot_f64(const double *a, const double *b, int dim)
{
    double s = 0.0;
    for (int k = 0; k < dim; ++k) s += a[k] * b[k];
    return s;
}

/*
 * One (query q, document b) pair.  Writes, for each query token i < lq_max:
 *   argmax_row[i] = lowest t attaining max_t <Q_qi, D_bt>   (R1, R4); -1 when
 *                   i >= q_lens[q] or the document is empty (R2);
 *   rowmax_row[i] = that maximum (NAN for an invalid row, -inf for R2);
 *   gap_row[i]    = maximum minus the largest value over the other tokens
 *                   (INFINITY when the document has fewer than two tokens,
 *                   or the row is invalid).
 * Returns the score (R2, R3).
 */
static double pair_forward(const double *Q, const int32_t *q_lens, int32_t lq_max,
                           const double *D, const int32_t *cu, int32_t dim,
                           int32_t q, int32_t b,
                           int32_t *argmax_row, double *rowmax_row, double *gap_row)
{
    int32_t lq = q_lens[q];
    int64_t t0 = cu[b];
    int64_t ld = (int64_t)cu[b + 1] - t0;
    double score = 0.0;
    for (int32_t i = 0; i < lq_max; ++i) {
        if (i >= lq) {
            if (argmax_row) argmax_row[i] = -1;
            if (rowmax_row) rowmax_row[i] = NAN;
            if (gap_row) gap_row[i] = INFINITY;
            continue;
        }
        const double *qi = Q + ((int64_t)q * lq_max + i) * dim;
        double best = -INFINITY, second = -INFINITY;
        int64_t arg = -1;
        for (int64_t t = 0; t < ld; ++t) {
            double v = dot_f64(qi, D + (t0 + t) * dim, dim);
            if (v > best) {          /* strict: the lowest t keeps a tie */
                second = best;
                best = v;
                arg = t;
            } else if (v > second) {
                second = v;
            }
        }
        score += best;               /* ascending i; -inf for an empty doc */
        if (argmax_row) argmax_row[i] = (int32_t)arg;
        if (rowmax_row) rowmax_row[i] = best;
        if (gap_row) gap_row[i] = ld >= 2 ? best - second : INFINITY;
    }
    return score;
}

/*
 * Forward over a list of (q, b) pairs, or over all pairs in row-major (q, b)
 * order when pair_q == NULL (then n_pairs is ignored and n_q * n_docs pairs
 * are produced).  Outputs are indexed by pair:
 *   score[p], argmax[p * lq_max + i], rowmax[p * lq_max + i], gap[...];
 * any of argmax/rowmax/gap may be NULL.
 * Returns 0, or -1 on a malformed argument.
 */
int oracle_forward_f64(const double *Q, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                       const double *D, const int32_t *cu_seqlens, int32_t n_docs, int32_t dim,
                       int64_t n_pairs, const int32_t *pair_q, const int32_t *pair_b,
                       double *score, int32_t *argmax, double *rowmax, double *gap)
{
    if (n_q < 0 || n_docs < 0 || lq_max < 0 || dim <= 0) return -1;
    if (pair_q == NULL) n_pairs = (int64_t)n_q * n_docs;
    for (int64_t p = 0; p < n_pairs; ++p) {
        int32_t q = pair_q ? pair_q[p] : (int32_t)(p / (n_docs ? n_docs : 1));
        int32_t b = pair_q ? pair_b[p] : (int32_t)(p % (n_docs ? n_docs : 1));
        if (q < 0 || q >= n_q || b < 0 || b >= n_docs) return -1;
        if (q_lens[q] < 0 || q_lens[q] > lq_max) return -1;
        score[p] = pair_forward(Q, q_lens, lq_max, D, cu_seqlens, dim, q, b,
                                argmax ? argmax + p * lq_max : NULL,
                                rowmax ? rowmax + p * lq_max : NULL,
                                gap ? gap + p * lq_max : NULL);
    }
    return 0;
}

/*
 * Same as oracle_forward_f64 but on stored FP16/BF16 patterns (dtype 0/1).
 * Q is decoded whole; each document is decoded when its pair is evaluated.
 */
int oracle_forward_bits(int dtype, const uint16_t *Qbits, const int32_t *q_lens,
                        int32_t n_q, int32_t lq_max,
                        const uint16_t *Dbits, const int32_t *cu_seqlens, int32_t n_docs,
                        int32_t dim, int64_t n_pairs, const int32_t *pair_q,
                        const int32_t *pair_b, double *score, int32_t *argmax,
                        double *rowmax, double *gap)
{
    if (dtype != 0 && dtype != 1) return -1;
    if (n_q < 0 || n_docs < 0 || lq_max < 0 || dim <= 0) return -1;
    int64_t nq_el = (int64_t)n_q * lq_max * dim;
    double *Q = (double *)malloc((size_t)(nq_el > 0 ? nq_el : 1) * sizeof(double));
    if (!Q) return -2;
    oracle_decode(dtype, Qbits, Q, nq_el);
    /* local cu for the single decoded document: {0, Ld} */
    int32_t cu_local[2];
    double *Dd = NULL;
    int64_t cap = 0;
    int rc = 0;
    if (pair_q == NULL) n_pairs = (int64_t)n_q * n_docs;
    for (int64_t p = 0; p < n_pairs && rc == 0; ++p) {
        int32_t q = pair_q ? pair_q[p] : (int32_t)(p / (n_docs ? n_docs : 1));
        int32_t b = pair_q ? pair_b[p] : (int32_t)(p % (n_docs ? n_docs : 1));
        if (q < 0 || q >= n_q || b < 0 || b >= n_docs || q_lens[q] < 0 || q_lens[q] > lq_max) {
            rc = -1;
            break;
        }
        int64_t ld = (int64_t)cu_seqlens[b + 1] - cu_seqlens[b];
        if (ld < 0) { rc = -1; break; }
        if (ld * dim > cap) {
            free(Dd);
            cap = ld * dim;
            Dd = (double *)malloc((size_t)cap * sizeof(double));
            if (!Dd) { rc = -2; break; }
        }
        oracle_decode(dtype, Dbits + (int64_t)cu_seqlens[b] * dim, Dd, ld * dim);
        cu_local[0] = 0;
        cu_local[1] = (int32_t)ld;
        /* pair_forward addresses the document as index 0 of cu_local */
        int32_t qlen_one = q_lens[q];
        score[p] = pair_forward(Q + (int64_t)q * lq_max * dim, &qlen_one, lq_max,
                                Dd ? Dd : Q, cu_local, dim, 0, 0,
                                argmax ? argmax + p * lq_max : NULL,
                                rowmax ? rowmax + p * lq_max : NULL,
                                gap ? gap + p * lq_max : NULL);
    }
    free(Dd);
    free(Q);
    return rc;
}

/*
 * Exact dot products <Q_{q,i}, D_{cu[b]+t}> of stored patterns for n given
 * (q, b, i, t) tuples -- used to judge an argmax reported by the kernel
 * against the true maximum (argmax acceptance on near-ties).
 */
int oracle_dot_bits(int dtype, const uint16_t *Qbits, int32_t lq_max,
                    const uint16_t *Dbits, const int32_t *cu_seqlens, int32_t dim,
                    int64_t n, const int32_t *q, const int32_t *b, const int32_t *i,
                    const int32_t *t, double *out)
{
    if (dtype != 0 && dtype != 1) return -1;
    double *qa = (double *)malloc((size_t)dim * sizeof(double));
    double *da = (double *)malloc((size_t)dim * sizeof(double));
    if (!qa || !da) { free(qa); free(da); return -2; }
    for (int64_t k = 0; k < n; ++k) {
        oracle_decode(dtype, Qbits + ((int64_t)q[k] * lq_max + i[k]) * dim, qa, dim);
        oracle_decode(dtype, Dbits + ((int64_t)cu_seqlens[b[k]] + t[k]) * dim, da, dim);
        out[k] = dot_f64(qa, da, dim);
    }
    free(qa);
    free(da);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* INT8 x INT8: Flash-MaxSim §4.3.1, read with one symmetric scale per tensor */
/* (R5): exact integer dots, integer maxima (lowest t on ties), int64 sum,    */
/* one scale at the end.                                                       */
/* ------------------------------------------------------------------------- */

/*
 * Outputs per pair p: raw[p] (int64; INT64_MIN for an empty document with a
 * non-empty query), score[p] (float; -inf for the same case), argmax as in
 * the floating-point forward.  Returns 0, -1 on a malformed argument, or -3
 * if an integer dot leaves the int32 range (it cannot for |x| <= 127, d=128).
 */
int oracle_forward_i8(const int8_t *Q, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                      const int8_t *D, const int32_t *cu_seqlens, int32_t n_docs, int32_t dim,
                      float q_scale, float d_scale,
                      int64_t n_pairs, const int32_t *pair_q, const int32_t *pair_b,
                      int64_t *raw, float *score, int32_t *argmax)
{
    if (n_q < 0 || n_docs < 0 || lq_max < 0 || dim <= 0) return -1;
    if (pair_q == NULL) n_pairs = (int64_t)n_q * n_docs;
    double scale = (double)q_scale * (double)d_scale;
    for (int64_t p = 0; p < n_pairs; ++p) {
        int32_t q = pair_q ? pair_q[p] : (int32_t)(p / (n_docs ? n_docs : 1));
        int32_t b = pair_q ? pair_b[p] : (int32_t)(p % (n_docs ? n_docs : 1));
        if (q < 0 || q >= n_q || b < 0 || b >= n_docs) return -1;
        int32_t lq = q_lens[q];
        if (lq < 0 || lq > lq_max) return -1;
        int64_t t0 = cu_seqlens[b];
        int64_t ld = (int64_t)cu_seqlens[b + 1] - t0;
        int64_t sum = 0;
        int empty = 0;
        for (int32_t i = 0; i < lq_max; ++i) {
            if (i >= lq) {
                if (argmax) argmax[p * lq_max + i] = -1;
                continue;
            }
            const int8_t *qi = Q + ((int64_t)q * lq_max + i) * dim;
            int64_t best = 0;
            int64_t arg = -1;
            for (int64_t t = 0; t < ld; ++t) {
                const int8_t *dt = D + (t0 + t) * dim;
                int64_t v = 0;
                for (int k = 0; k < dim; ++k) v += (int64_t)qi[k] * (int64_t)dt[k];
                if (v > INT32_MAX || v < INT32_MIN) return -3;
                if (arg < 0 || v > best) {   /* strict after the first: lowest t on ties */
                    best = v;
                    arg = t;
                }
            }
            if (arg < 0) empty = 1;
            else sum += best;
            if (argmax) argmax[p * lq_max + i] = (int32_t)arg;
        }
        if (empty) {
            raw[p] = INT64_MIN;
            score[p] = -INFINITY;
        } else {
            raw[p] = sum;
            score[p] = (float)((double)sum * scale);
        }
    }
    return 0;
}

/*
 * INT8 with one symmetric scale per token (R6).  q_scales [n_q, lq_max],
 * d_scales [total]; outputs per pair: score (binary64; -inf for an empty
 * document and a query with tokens), argmax [.., lq_max]; when rowmax / gap
 * are non-NULL, the binary64 row maxima and the gap from the maximum to the
 * largest value over the other tokens [.., lq_max] (-inf / +inf for padding
 * and empty documents, +inf for a document of one token).
 */
int oracle_forward_i8_token(const int8_t *Q, const float *q_scales, const int32_t *q_lens, int32_t n_q,
                            int32_t lq_max, const int8_t *D, const float *d_scales,
                            const int32_t *cu_seqlens, int32_t n_docs, int32_t dim,
                            int64_t n_pairs, const int32_t *pair_q, const int32_t *pair_b,
                            double *score, int32_t *argmax, double *rowmax, double *gap)
{
    if (n_q < 0 || n_docs < 0 || lq_max < 0 || dim <= 0) return -1;
    if (pair_q == NULL) n_pairs = (int64_t)n_q * n_docs;
    for (int64_t p = 0; p < n_pairs; ++p) {
        int32_t q = pair_q ? pair_q[p] : (int32_t)(p / (n_docs ? n_docs : 1));
        int32_t b = pair_q ? pair_b[p] : (int32_t)(p % (n_docs ? n_docs : 1));
        if (q < 0 || q >= n_q || b < 0 || b >= n_docs) return -1;
        int32_t lq = q_lens[q];
        if (lq < 0 || lq > lq_max) return -1;
        int64_t t0 = cu_seqlens[b];
        int64_t ld = (int64_t)cu_seqlens[b + 1] - t0;
        double sum = 0.0;
        int empty = 0;
        for (int32_t i = 0; i < lq_max; ++i) {
            int64_t o = p * lq_max + i;
            if (i >= lq) {
                if (argmax) argmax[o] = -1;
                if (rowmax) rowmax[o] = -INFINITY;
                if (gap) gap[o] = INFINITY;
                continue;
            }
            const int8_t *qi = Q + ((int64_t)q * lq_max + i) * dim;
            double best = -INFINITY, second = -INFINITY;
            int64_t arg = -1;
            for (int64_t t = 0; t < ld; ++t) {
                const int8_t *dt = D + (t0 + t) * dim;
                int64_t v = 0;
                for (int k = 0; k < dim; ++k) v += (int64_t)qi[k] * (int64_t)dt[k];
                if (v > 16777216 || v < -16777216) return -3;  /* < 2^24: the product below is exact */
                double scaled = (double)v * (double)d_scales[t0 + t];
                if (arg < 0 || scaled > best) {                  /* lowest t on ties */
                    second = best;
                    best = scaled;
                    arg = t;
                } else if (scaled > second) {
                    second = scaled;
                }
            }
            if (arg < 0) empty = 1;
            else sum += (double)q_scales[(int64_t)q * lq_max + i] * best;
            if (argmax) argmax[o] = (int32_t)arg;
            if (rowmax) rowmax[o] = best;
            if (gap) gap[o] = ld >= 2 ? best - second : INFINITY;
        }
        score[p] = empty ? -INFINITY : sum;
    }
    return 0;
}

/*
 * Exact ranked values dot(Q_{q,i}, D_{cu[b]+t}) * s_D[cu[b]+t] (R6) for n
 * given (q, b, i, t) tuples -- used to judge an argmax reported by the
 * kernel against the true maximum.
 */
int oracle_dot_i8_token(const int8_t *Q, int32_t lq_max, const int8_t *D, const float *d_scales,
                        const int32_t *cu_seqlens, int32_t dim, int64_t n, const int32_t *q,
                        const int32_t *b, const int32_t *i, const int32_t *t, double *out)
{
    for (int64_t k = 0; k < n; ++k) {
        const int8_t *qi = Q + ((int64_t)q[k] * lq_max + i[k]) * dim;
        int64_t row = (int64_t)cu_seqlens[b[k]] + t[k];
        const int8_t *dt = D + row * dim;
        int64_t v = 0;
        for (int c = 0; c < dim; ++c) v += (int64_t)qi[c] * (int64_t)dt[c];
        out[k] = (double)v * (double)d_scales[row];
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Chamfer distance (R7).  Point sets are packed: item b owns source points  */
/* cu_s[b] .. cu_s[b+1]-1 and target points cu_t[b] .. cu_t[b+1]-1, each a   */
/* row of three binary32 coordinates.                                        */
/* ------------------------------------------------------------------------- */

static double chamfer_d2(const float *s, const float *t)
{
    double dx = (double)s[0] - (double)t[0];
    double dy = (double)s[1] - (double)t[1];
    double dz = (double)s[2] - (double)t[2];
    return dx * dx + dy * dy + dz * dz;
}

/* Nearest target of every source point: dist [total_s] (binary64), arg
 * [total_s] (index local to the item's target set, -1 when it is empty) and,
 * when gap is non-NULL, the second-smallest distance minus the smallest
 * (+inf with fewer than two targets). */
int oracle_chamfer_nn(const float *S, const int32_t *cu_s, const float *T, const int32_t *cu_t,
                      int32_t n_items, double *dist, int32_t *arg, double *gap)
{
    if (n_items < 0) return -1;
    for (int32_t b = 0; b < n_items; ++b) {
        int64_t t0 = cu_t[b], m = (int64_t)cu_t[b + 1] - t0;
        for (int64_t s = cu_s[b]; s < cu_s[b + 1]; ++s) {
            double best = INFINITY, second = INFINITY;
            int64_t a = -1;
            for (int64_t t = 0; t < m; ++t) {
                double d = chamfer_d2(S + 3 * s, T + 3 * (t0 + t));
                if (a < 0 || d < best) {     /* strict after the first: lowest t on ties */
                    second = best;
                    best = d;
                    a = t;
                } else if (d < second) {
                    second = d;
                }
            }
            dist[s] = best;
            arg[s] = (int32_t)a;
            if (gap) gap[s] = m >= 2 ? second - best : INFINITY;
        }
    }
    return 0;
}

/* Squared distances (R7) of n given (source, target) index pairs of the
 * packed point arrays. */
int oracle_chamfer_pair_dist(const float *S, const float *T, int64_t n, const int32_t *si, const int32_t *ti,
                             double *out)
{
    for (int64_t k = 0; k < n; ++k) out[k] = chamfer_d2(S + 3 * (int64_t)si[k], T + 3 * (int64_t)ti[k]);
    return 0;
}

/* cd[b] = mean over P of its nearest-target distance + mean over Q of its
 * nearest-source distance, in binary64. */
int oracle_chamfer_reduce(const double *dist_pq, const int32_t *cu_p, const double *dist_qp, const int32_t *cu_q,
                          int32_t n_items, double *cd)
{
    for (int32_t b = 0; b < n_items; ++b) {
        double a = 0.0, c = 0.0;
        int64_t n = (int64_t)cu_p[b + 1] - cu_p[b], m = (int64_t)cu_q[b + 1] - cu_q[b];
        for (int64_t i = cu_p[b]; i < cu_p[b + 1]; ++i) a += dist_pq[i];
        for (int64_t j = cu_q[b]; j < cu_q[b + 1]; ++j) c += dist_qp[j];
        cd[b] = (n ? a / (double)n : 0.0) + (m ? c / (double)m : 0.0);
    }
    return 0;
}

/* Gradient of sum_b grad[b] * cd[b] for the given nearest-neighbour indices,
 * scattered straight from the chain rule in binary64: the term of point p
 * with nearest target q contributes 2 g (p - q) / N to dP[p] and its negative
 * to dQ[q] (and symmetrically for the Q -> P term with 1 / M). */
int oracle_chamfer_backward(const float *P, const int32_t *cu_p, const float *Q, const int32_t *cu_q,
                            int32_t n_items, const int32_t *arg_pq, const int32_t *arg_qp,
                            const double *grad, double *dP, double *dQ)
{
    memset(dP, 0, sizeof(double) * 3 * (size_t)cu_p[n_items]);
    memset(dQ, 0, sizeof(double) * 3 * (size_t)cu_q[n_items]);
    for (int32_t b = 0; b < n_items; ++b) {
        int64_t p0 = cu_p[b], n = (int64_t)cu_p[b + 1] - p0;
        int64_t q0 = cu_q[b], m = (int64_t)cu_q[b + 1] - q0;
        for (int64_t i = 0; i < n; ++i) {
            int32_t a = arg_pq[p0 + i];
            if (a < 0) continue;
            if (a >= m) return -2;
            double w = 2.0 * grad[b] / (double)n;
            for (int k = 0; k < 3; ++k) {
                double diff = (double)P[3 * (p0 + i) + k] - (double)Q[3 * (q0 + a) + k];
                dP[3 * (p0 + i) + k] += w * diff;
                dQ[3 * (q0 + a) + k] -= w * diff;
            }
        }
        for (int64_t j = 0; j < m; ++j) {
            int32_t a = arg_qp[q0 + j];
            if (a < 0) continue;
            if (a >= n) return -2;
            double w = 2.0 * grad[b] / (double)m;
            for (int k = 0; k < 3; ++k) {
                double diff = (double)Q[3 * (q0 + j) + k] - (double)P[3 * (p0 + a) + k];
                dQ[3 * (q0 + j) + k] += w * diff;
                dP[3 * (p0 + a) + k] -= w * diff;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Backward: Flash-MaxSim §4.2.1 Eq. (2) and Eq. (3), written here in scatter */
/* form straight from the chain rule -- each selected (q, b, i) adds          */
/* g[q,b] * D_{b,t*} into dQ_{q,i} and g[q,b] * Q_{q,i} into dD_{b,t*}.       */
/* It consumes a given argmax (the forward's winners t*).                     */
/* ------------------------------------------------------------------------- */

/*
 * grad: [n_q, n_docs] (double);  argmax: [n_q, n_docs, lq_max], -1 = none;
 * dQ: [n_q, lq_max, dim] and dD: [total_tokens, dim] are overwritten.
 * Returns 0, or -1 when an argmax entry of a valid row lies outside its
 * document.
 */
int oracle_backward_f64(const double *grad, const int32_t *argmax,
                        const double *Q, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                        const double *D, const int32_t *cu_seqlens, int32_t n_docs, int32_t dim,
                        double *dQ, double *dD)
{
    int64_t total = n_docs > 0 ? cu_seqlens[n_docs] : 0;
    memset(dQ, 0, (size_t)n_q * lq_max * dim * sizeof(double));
    memset(dD, 0, (size_t)total * dim * sizeof(double));
    for (int32_t q = 0; q < n_q; ++q) {
        for (int32_t b = 0; b < n_docs; ++b) {
            double g = grad[(int64_t)q * n_docs + b];
            int64_t ld = (int64_t)cu_seqlens[b + 1] - cu_seqlens[b];
            for (int32_t i = 0; i < q_lens[q]; ++i) {
                int32_t t = argmax[((int64_t)q * n_docs + b) * lq_max + i];
                if (t < 0) continue;
                if (t >= ld) return -1;
                double *dq = dQ + ((int64_t)q * lq_max + i) * dim;
                double *dd = dD + ((int64_t)cu_seqlens[b] + t) * dim;
                const double *qi = Q + ((int64_t)q * lq_max + i) * dim;
                const double *dt = D + ((int64_t)cu_seqlens[b] + t) * dim;
                for (int k = 0; k < dim; ++k) {
                    dq[k] += g * dt[k];
                    dd[k] += g * qi[k];
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Inverse-grid CSR: Flash-MaxSim §4.2.2 and Alg. 3 step 1.  Each selected    */
/* source -- flat position s = (q * n_docs + b) * lq_max + i of the argmax    */
/* array -- points at destination row dst = cu[b] + A[s] of the packed D.     */
/* row_ptr = exclusive cumulative sum of bincount(dst) over all rows;         */
/* col_idx = the sources ordered by a stable sort on dst (so ascending s      */
/* within a row).  The sort step here is the C library's qsort on the         */
/* (dst, s) pair, which orders exactly like a stable sort on dst.             */
/* ------------------------------------------------------------------------- */

typedef struct { int64_t dst; int64_t src; } csr_pair_t;

static int cmp_pair(const void *a, const void *b)
{
    const csr_pair_t *x = (const csr_pair_t *)a, *y = (const csr_pair_t *)b;
    if (x->dst != y->dst) return x->dst < y->dst ? -1 : 1;
    if (x->src != y->src) return x->src < y->src ? -1 : 1;
    return 0;
}

/*
 * row_ptr: [total_tokens + 1];  col_idx: room for every valid source.
 * Sources are rows i < q_lens[q] whose argmax is >= 0.  Returns the number of
 * sources (nnz), or -1 when an argmax entry lies outside its document.
 */
int64_t oracle_build_csr(const int32_t *argmax, const int32_t *q_lens, int32_t n_q,
                         int32_t lq_max, const int32_t *cu_seqlens, int32_t n_docs,
                         int64_t *row_ptr, int64_t *col_idx)
{
    int64_t total = n_docs > 0 ? cu_seqlens[n_docs] : 0;
    int64_t cap = (int64_t)n_q * n_docs * lq_max;
    csr_pair_t *pairs = (csr_pair_t *)malloc((size_t)(cap > 0 ? cap : 1) * sizeof(csr_pair_t));
    int64_t *count = (int64_t *)calloc((size_t)(total + 1), sizeof(int64_t));
    if (!pairs || !count) { free(pairs); free(count); return -2; }
    int64_t nnz = 0;
    for (int32_t q = 0; q < n_q; ++q)
        for (int32_t b = 0; b < n_docs; ++b) {
            int64_t ld = (int64_t)cu_seqlens[b + 1] - cu_seqlens[b];
            for (int32_t i = 0; i < q_lens[q]; ++i) {
                int64_t s = ((int64_t)q * n_docs + b) * lq_max + i;
                int32_t a = argmax[s];
                if (a < 0) continue;
                if (a >= ld) { free(pairs); free(count); return -1; }
                pairs[nnz].dst = (int64_t)cu_seqlens[b] + a;
                pairs[nnz].src = s;
                ++nnz;
            }
        }
    /* bincount -> cumsum */
    for (int64_t k = 0; k < nnz; ++k) count[pairs[k].dst] += 1;
    row_ptr[0] = 0;
    for (int64_t r = 0; r < total; ++r) row_ptr[r + 1] = row_ptr[r] + count[r];
    /* stable argsort of dst */
    qsort(pairs, (size_t)nnz, sizeof(csr_pair_t), cmp_pair);
    for (int64_t k = 0; k < nnz; ++k) col_idx[k] = pairs[k].src;
    free(pairs);
    free(count);
    return nnz;
}
