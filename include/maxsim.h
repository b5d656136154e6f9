/*
 * maxsim.h -- C ABI of the GB300 (sm_103a) fused MaxSim library.
 *
 * The operator is late-interaction scoring as defined in "FLASH-MAXSIM:
 * IO-Aware Fused Kernels for Late-Interaction Retrieval" (arXiv 2605.29517):
 *
 *     score(q, b) = sum_{i < q_lens[q]}  max_{t < Ld_b}  <Q[q, i, :], D_b[t, :]>
 *
 * (§1 Eq. (1)), computed without materialising the [B, Lq, Ld] similarity
 * tensor (§4.1, Alg. 2), together with its training backward (§4.2, Eqs. (2)
 * and (3), Alg. 3), INT8 x INT8 scoring (§4.3.1) and padding-free
 * variable-length documents (§4.3.2).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All array pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates or frees memory; scratch space is passed in as a
 *    caller-owned workspace whose size the matching *_workspace_size() call
 *    reports (maxsim_forward_noalloc instead uses a fixed array the library
 *    owns, see there).
 *  - Calls are stream-ordered and asynchronous: they enqueue work on
 *    `stream` (a cudaStream_t; NULL = the legacy default stream) and return.
 *    Outputs are valid once the stream has been synchronised.
 *  - Layouts.  Q: [n_q, lq_max, dim] row-major, query q's valid tokens are
 *    rows 0 .. q_lens[q]-1 (the rest is padding and is never read as data).
 *    D: the packed token rows of all documents, [total_d_tokens, dim]
 *    row-major; document b owns rows cu_seqlens[b] .. cu_seqlens[b+1]-1.
 *    cu_seqlens: int32 [n_docs + 1], cu_seqlens[0] = 0, non-decreasing,
 *    cu_seqlens[n_docs] = total_d_tokens.  A dense batch of equal-length
 *    documents passes cu_seqlens[b] = b * Ld.
 *  - Q and D must start on a 16-byte boundary.  dim must be 128 (the pages'
 *    d; other widths return MAXSIM_ERR_UNSUPPORTED).
 *  - Synchronous return codes report argument errors before anything is
 *    enqueued.  A device-side failure (a pipeline wait that timed out, an
 *    out-of-range argmax handed to the backward) sets a device status word
 *    that maxsim_device_status() reads; the affected outputs are then
 *    unspecified.
 *  - Every result is deterministic: the same inputs give the same bits on
 *    every run (no floating-point atomics anywhere).
 */
#ifndef MAXSIM_H_
#define MAXSIM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MAXSIM_ABI_VERSION 1

typedef enum {
    MAXSIM_FP16 = 0, /* IEEE binary16 inputs, FP32 accumulation              */
    MAXSIM_BF16 = 1, /* bfloat16 inputs, FP32 accumulation                   */
    MAXSIM_INT8 = 2  /* int8 inputs in [-127, 127], exact integer arithmetic */
} maxsim_dtype_t;

typedef enum {
    MAXSIM_OK = 0,
    MAXSIM_ERR_INVALID_ARGUMENT = 1, /* null/misaligned pointer, bad size      */
    MAXSIM_ERR_UNSUPPORTED = 2,      /* dim != 128, dtype not supported here   */
    MAXSIM_ERR_WORKSPACE = 3,        /* workspace missing or too small         */
    MAXSIM_ERR_CUDA = 4,             /* a CUDA runtime/driver call failed      */
    MAXSIM_ERR_DEVICE = 5            /* the device status word reports a fault */
} maxsim_status_t;

/* MAXSIM_ABI_VERSION of the loaded library. */
int32_t maxsim_abi_version(void);

/* Static text for a status code. */
const char *maxsim_status_string(maxsim_status_t status);

/*
 * Bytes of workspace maxsim_forward needs for these sizes (0 when none).
 * Queries longer than 32 tokens keep one partial sum per 32-token chunk
 * (FP32, or int64 for INT8); INT8 inputs also keep an FP16 copy of Q.
 */
size_t maxsim_forward_workspace_size(int32_t n_q, int32_t lq_max, int32_t n_docs,
                                     int32_t dim, maxsim_dtype_t dtype);

/*
 * Fused forward: Flash-MaxSim §4.1 (Alg. 2, the online-max recurrence of
 * §4.1.1, the query-chunk decomposition of §4.1) over packed documents
 * (§4.3.2), for N_q queries against B documents (the all-pairs regime of
 * §3.1).  Each document row is read from HBM once for all queries.
 *
 *   Q, D        FP16/BF16/INT8 per `dtype`, layouts above.
 *   q_lens      int32 [n_q], 0 <= q_lens[q] <= lq_max (device).
 *   cu_seqlens  int32 [n_docs + 1] (device).
 *   q_scale, d_scale   INT8 only: one symmetric scale per tensor (§4.3.1,
 *               read per tensor); ignored for FP16/BF16.
 *   scores      FP32 [n_q, n_docs], written in full.  FP16/BF16: FP32
 *               tensor-core dot products, FP32 row maxima, a fixed-order
 *               FP32 sum over query tokens.  INT8: fp32(raw * (s_Q * s_D))
 *               with the product evaluated in binary64 once.
 *   raw_scores  INT8 only, optional (may be NULL): int64 [n_q, n_docs], the
 *               exact sum of the int32 row maxima.
 *   argmax      optional (may be NULL): int32 [n_q, n_docs, lq_max].  For a
 *               valid row, the lowest document-local token index attaining
 *               the row maximum; -1 for padding rows (i >= q_lens[q]) and
 *               for empty documents.  This is the saved winner map the
 *               backward consumes (§4.2.2).
 *   workspace   device scratch of at least maxsim_forward_workspace_size()
 *               bytes (may be NULL when that size is 0).
 * Edge cases: a document with no tokens scores -inf (and raw INT64_MIN) for
 * a query with at least one valid token; a query with q_lens[q] = 0 scores 0.
 * Returns MAXSIM_OK or an argument error; nothing is enqueued on error.
 */
maxsim_status_t maxsim_forward(const void *Q, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                               const void *D, const int32_t *cu_seqlens, int32_t n_docs,
                               int64_t total_d_tokens, int32_t dim, maxsim_dtype_t dtype,
                               float q_scale, float d_scale,
                               float *scores, int64_t *raw_scores, int32_t *argmax,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * maxsim_forward for callers that cannot allocate device memory.
 *
 * The pages have no counterpart: this is a deployment convenience.  Some
 * callers cannot call cudaMalloc where they score -- a plugin inside a host
 * framework that owns every device allocation and gives its plugins no
 * allocator, or a serving loop that must never allocate because cudaMalloc
 * and cudaFree can synchronise the device and stall all of its streams.
 * This entry point takes the same arguments as maxsim_forward minus the
 * workspace and allocates nothing: the forward's scratch lives in one
 * fixed 4 MiB array in device memory owned by the library (each GPU that
 * loads the library holds it until the process exits).
 *   - Sizes whose maxsim_forward_workspace_size() exceeds 4 MiB return
 *     MAXSIM_ERR_WORKSPACE before anything is enqueued (4 MiB holds about
 *     one million FP32 partial sums: e.g. a 1024-token query against
 *     32,000 documents).
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it with the device's context; make
 *     that first call before any stream capture.  A call that finds another
 *     context current on the device (after cudaDeviceReset, say) looks the
 *     address up again.
 *   - Every call shares the one array and leaves its contents behind; calls
 *     whose work overlaps on the GPU (other streams, other threads) race on
 *     it and must be serialised by the caller.
 */
maxsim_status_t maxsim_forward_noalloc(const void *Q, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                                       const void *D, const int32_t *cu_seqlens, int32_t n_docs,
                                       int64_t total_d_tokens, int32_t dim, maxsim_dtype_t dtype,
                                       float q_scale, float d_scale,
                                       float *scores, int64_t *raw_scores, int32_t *argmax,
                                       void *stream);

/*
 * INT8 x INT8 forward with one symmetric scale per TOKEN: Flash-MaxSim
 * §4.3.1 "INT8xINT8 Quantization" (per-token quantisation of both Q and D,
 * dequantisation fused into the kernel).  For each valid query row i and
 * document token t the kernel forms the exact integer dot product
 * dot(i, t) = <Q[q, i, :], D[cu[b] + t, :]> and ranks
 *     v(i, t) = fp32( (float)dot(i, t) * d_scales[cu[b] + t] )
 * (one IEEE single-precision product: dot is an integer below 2^24, so
 * (float)dot is exact); the row maximum m_i = max_t v(i, t) and its lowest
 * attaining t (the argmax) are taken on these FP32 values, then
 *     scores[q, b] = sum_{i < q_lens[q]} fp32(q_scales[q, i] * m_i)
 * in FP32 in a fixed order (a document with no tokens gives -inf).  The
 * query scale multiplies after the maximum, which selects the same token as
 * scaling before it when the scale is positive.
 *   Q           int8 [n_q, lq_max, dim], values in [-127, 127] (device).
 *   q_scales    FP32 [n_q, lq_max], finite and >= 0 (device).
 *   D           int8 [total_d_tokens, dim] packed (device).
 *   d_scales    FP32 [total_d_tokens], finite and >= 0 (device).
 *   scores, argmax   as maxsim_forward (argmax optional).
 *   workspace   maxsim_forward_workspace_size(n_q, lq_max, n_docs, dim,
 *               MAXSIM_INT8) bytes.
 * Unlike the per-tensor INT8 path the result is not an exact integer: the
 * page's own description calls the per-token path approximate.
 */
maxsim_status_t maxsim_forward_int8_per_token(const int8_t *Q, const float *q_scales, const int32_t *q_lens,
                                              int32_t n_q, int32_t lq_max, const int8_t *D,
                                              const float *d_scales, const int32_t *cu_seqlens,
                                              int32_t n_docs, int64_t total_d_tokens, int32_t dim,
                                              float *scores, int32_t *argmax,
                                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Row-wise top-K selection, the selection step of the two-stage scan below.
 * For each of n_rows rows of `values` (FP32, row stride ld >= n_cols), the
 * k largest entries in descending order; equal values are ordered by
 * ascending column, so the result is unique.  out_ids / out_values: [n_rows,
 * k]; positions past n_cols (k > n_cols) get id -1 and value -inf.  -inf
 * ranks below every finite value; NaN inputs give unspecified results.
 * k <= 4096 (larger: MAXSIM_ERR_UNSUPPORTED).  One CTA per row.
 */
maxsim_status_t maxsim_topk(const float *values, int32_t n_rows, int32_t n_cols, int64_t ld, int32_t k,
                            int32_t *out_ids, float *out_values, void *stream);

/* Bytes of workspace maxsim_rerank_two_stage needs. */
size_t maxsim_rerank_workspace_size(int32_t n_q, int32_t lq_max, int32_t n_docs, int32_t k_candidates,
                                    int32_t max_doc_len, int32_t dim, maxsim_dtype_t dtype16);

/*
 * Two-stage INT8 -> FP16 top-K scan: Flash-MaxSim §4.1 "Kernel Family" lists
 * it among the forward variants without further detail; the reading taken:
 *   1. every document is scored against every query with the INT8 MaxSim
 *      (maxsim_forward with MAXSIM_INT8 and one scale per tensor, or
 *      maxsim_forward_int8_per_token when q_tok_scales and d_tok_scales are
 *      both given);
 *   2. each query keeps its k_candidates best documents (maxsim_topk order:
 *      ties to the lower document index);
 *   3. those candidates' rows are gathered from the FP16/BF16 copy of the
 *      corpus and rescored against the query's FP16/BF16 tokens with the
 *      fused forward (FP32 accumulation);
 *   4. each query returns its k best candidates by the stage-3 score
 *      (ties to the earlier candidate).
 *   Q8, D8, q_lens, cu_seqlens   the INT8 query/corpus (device), layouts as
 *               maxsim_forward; q_scale, d_scale the per-tensor scales
 *               (ignored in per-token mode).
 *   Q16         FP16/BF16 [n_q, lq_max, dim] (device), the same queries.
 *   D16         FP16/BF16 [total_d_tokens, dim], the same corpus: device
 *               memory, or page-locked host memory (cudaHostAlloc /
 *               cudaHostRegister) that the gather reads over the host link;
 *               pageable memory is an argument error.  Only candidates'
 *               rows are read.
 *   max_doc_len the longest document (sizes the gather buffer); a longer
 *               candidate is cut to max_doc_len rows and sets the device
 *               status word (code 0x202).
 *   top_ids, top_scores   [n_q, k] (device): document ids and their stage-3
 *               FP32 scores; -1 / -inf past the number of documents.
 *   candidate_ids  optional [n_q, k_candidates] (device): stage-2 ids.
 *   workspace   maxsim_rerank_workspace_size() bytes (device): holds the
 *               stage-1 scores [n_q, n_docs] and n_q * k_candidates *
 *               max_doc_len gathered rows.
 * 1 <= k_candidates <= 4096, 0 <= k <= k_candidates.
 */
maxsim_status_t maxsim_rerank_two_stage(const int8_t *Q8, const float *q_tok_scales, float q_scale,
                                        const int8_t *D8, const float *d_tok_scales, float d_scale,
                                        const void *Q16, const void *D16, maxsim_dtype_t dtype16,
                                        const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                                        const int32_t *cu_seqlens, int32_t n_docs, int64_t total_d_tokens,
                                        int32_t max_doc_len, int32_t dim, int32_t k_candidates, int32_t k,
                                        int32_t *top_ids, float *top_scores, int32_t *candidate_ids,
                                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * Bytes of workspace maxsim_forward_host needs: two staging blocks of
 * block_tokens document rows (double buffer), a device copy of the n_docs + 1
 * offsets and the current block's rebased offsets, plus the forward's own
 * scratch for block_docs documents.  Returns 0 for invalid sizes.
 */
size_t maxsim_forward_host_workspace_size(int32_t n_q, int32_t lq_max, int32_t n_docs, int32_t block_docs,
                                          int64_t block_tokens, int32_t dim, maxsim_dtype_t dtype);

/*
 * Forward over a HOST-resident corpus: Flash-MaxSim §5 "Out-of-Core Corpus
 * Scaling" (Table "Out-of-core scoring").  The fused forward's device
 * footprint is one streamed block of documents, so a corpus larger than
 * device memory is scored by keeping it in host memory and copying
 * consecutive blocks of documents to the device, each block scored by the
 * same kernels as maxsim_forward while the next block is copied.
 *
 *   Q, q_lens   DEVICE, as for maxsim_forward.
 *   D_host      HOST [total_d_tokens, dim] packed rows.  For copy/compute
 *               overlap it must be page-locked (cudaHostAlloc /
 *               cudaHostRegister); pageable memory is accepted but its
 *               copies stage through the driver and do not overlap.
 *   cu_seqlens_host  HOST int32 [n_docs + 1] (cu[0] = 0, non-decreasing,
 *               cu[n_docs] = total_d_tokens).  The call plans the blocks
 *               from it and copies it to the workspace once, on `stream`.
 *   scores, raw_scores, argmax   DEVICE, the same layouts and values as
 *               maxsim_forward with the whole corpus resident; argmax and
 *               raw_scores optional.
 *   block_docs, block_tokens   Blocks are consecutive documents, greedily
 *               as many as fit both limits; no document is split, so a
 *               document longer than block_tokens is an argument error.
 *   workspace   DEVICE, at least maxsim_forward_host_workspace_size() bytes.
 *   stream      the stream every kernel runs on; the call's results are
 *               complete when it has synchronised.
 *   copy_stream a second stream for the host-to-device copies (NULL: the
 *               copies go on `stream` and nothing overlaps).  It first waits
 *               for the work already queued on `stream`.
 * Scores are bit-identical to maxsim_forward's over the same corpus (a
 * document's score does not depend on which other documents share a
 * launch).  The call only enqueues; D_host and cu_seqlens_host must stay
 * valid and unchanged until `stream` has synchronised.  Returns MAXSIM_OK, an argument error
 * (nothing enqueued), or MAXSIM_ERR_CUDA (blocks before the failing one
 * may have been enqueued).
 */
maxsim_status_t maxsim_forward_host(const void *Q, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                                    const void *D_host, const int32_t *cu_seqlens_host, int32_t n_docs,
                                    int64_t total_d_tokens, int32_t dim, maxsim_dtype_t dtype,
                                    float q_scale, float d_scale,
                                    float *scores, int64_t *raw_scores, int32_t *argmax,
                                    int32_t block_docs, int64_t block_tokens,
                                    void *workspace, size_t workspace_bytes, void *stream,
                                    void *copy_stream);

/* Bytes of workspace maxsim_backward / maxsim_build_csr need. */
size_t maxsim_backward_workspace_size(int32_t n_q, int32_t lq_max, int32_t n_docs,
                                      int64_t total_d_tokens);

/*
 * Inverse-grid CSR: Flash-MaxSim §4.2.2 (Alg. 3 step 1).  A source is a
 * flat position s = (q * n_docs + b) * lq_max + i of `argmax` with
 * i < q_lens[q] and argmax[s] >= 0; it points at destination row
 * r = cu_seqlens[b] + argmax[s] of the packed D.
 *   row_ptr  int32 [total_d_tokens + 1]: row_ptr[r] = number of sources whose
 *            destination is < r (exclusive cumulative bincount).
 *   col_idx  int32 [number of sources] (at most n_q * n_docs * lq_max):
 *            sources ordered by destination, ascending s within a row -- the
 *            order of a stable argsort of the destinations.
 * Built per document with an atomic-free, deterministic counting sort.
 * An argmax entry outside [-1, Ld_b) sets the device status word and the
 * entry is skipped.  Requires n_q * n_docs * lq_max < 2^31.
 */
maxsim_status_t maxsim_build_csr(const int32_t *argmax, const int32_t *q_lens, int32_t n_q,
                                 int32_t lq_max, const int32_t *cu_seqlens, int32_t n_docs,
                                 int64_t total_d_tokens, int32_t *row_ptr, int32_t *col_idx,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * Training backward: Flash-MaxSim §4.2.1 Eqs. (2)-(3) via Alg. 3 -- the
 * argmax is inverted into per-document lists of sources ordered as in the
 * CSR above (each document's sources sorted by token in shared memory, in
 * chunks of about 2,048 candidates, ascending source order within a token),
 * then
 *   dD[r, :]    = sum over the sources s = (q, b, i) of row r of
 *                 grad_scores[q, b] * Q[q, i, :]      (destination-owned,
 *                 one writer per row, no atomics; §4.2.3)
 *   dQ[q, i, :] = sum over b of
 *                 grad_scores[q, b] * D[cu_seqlens[b] + argmax[q, b, i], :]
 * both accumulated in FP32 in a fixed order that depends only on the
 * shapes and the argmax: each row's list is visited from a position derived
 * from the row's index, wrapping around (rows that run together then read
 * different parts of Q / D), its even and odd visits summed separately and
 * the two sums added -- so the result is the same bit for bit on every run.
 * dQ runs on a non-blocking stream the library keeps per device (created on
 * the first backward on that device), forked from and joined back into
 * `stream` with events, so it overlaps dD; the call is stream-ordered like
 * every other.
 *   grad_scores FP32 [n_q, n_docs];  argmax as produced by maxsim_forward.
 *   dQ          FP32 [n_q, lq_max, dim], written in full (padding rows 0).
 *   dD          FP32 [total_d_tokens, dim], written in full (rows nobody
 *               selected are 0).
 *   Q, D, dQ and dD must start on a 16-byte boundary.
 * An argmax entry outside [-1, Ld_b) (of a valid query row) sets the device
 * status word and contributes to neither gradient.
 * dtype: FP16 or BF16 (INT8 returns MAXSIM_ERR_UNSUPPORTED).  At most
 * 491,520 candidates per document (n_q * lq_max), else
 * MAXSIM_ERR_UNSUPPORTED.
 */
maxsim_status_t maxsim_backward(const float *grad_scores, const int32_t *argmax,
                                const void *Q, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                                const void *D, const int32_t *cu_seqlens, int32_t n_docs,
                                int64_t total_d_tokens, int32_t dim, maxsim_dtype_t dtype,
                                float *dQ, float *dD,
                                void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------ */
/* Chamfer distance: Flash-MaxSim §4.2 "Generalization to Chamfer Distance".  */
/* The MaxSim skeleton with a minimum over squared Euclidean distances:       */
/*   CD(P, Q) = 1/N sum_p min_q |p - q|^2 + 1/M sum_q min_p |q - p|^2         */
/* for a batch of point-set pairs packed like documents: item b owns points  */
/* cu_p[b] .. cu_p[b+1]-1 of P and cu_q[b] .. cu_q[b+1]-1 of Q, each point a */
/* row of three FP32 coordinates ([total, 3] row-major, device).              */
/* ------------------------------------------------------------------------ */

/* Bytes of workspace maxsim_chamfer_forward needs (0: none). */
size_t maxsim_chamfer_forward_workspace_size(int32_t n_items, int64_t total_p, int64_t total_q, int32_t max_p,
                                             int32_t max_q);

/*
 * Forward: for every point its nearest neighbour in the item's other set,
 * ranked on the FP32 value fma(dz, dz, fma(dy, dy, dx * dx)) with
 * dx = p.x - q.x (each step rounded to nearest even), the lowest index on
 * ties; an empty other set gives +inf and index -1.
 *   max_p, max_q   the largest |P_b| and |Q_b| (size the launch; a larger set
 *               sets the device status word, code 0x203).
 *   cd          FP32 [n_items]: the two means of the FP32 distances, summed
 *               in binary64 in a fixed order (a mean over an empty set is 0).
 *   dist_pq, arg_pq   FP32 / int32 [total_p]: nearest distance and the
 *               index of the nearest point of Q_b (local to the item).
 *   dist_qp, arg_qp   the same for Q against P_b.
 * Coordinates must be finite with finite squared differences.
 */
maxsim_status_t maxsim_chamfer_forward(const float *P, const int32_t *cu_p, const float *Q, const int32_t *cu_q,
                                       int32_t n_items, int64_t total_p, int64_t total_q, int32_t max_p,
                                       int32_t max_q, float *cd, float *dist_pq, int32_t *arg_pq,
                                       float *dist_qp, int32_t *arg_qp,
                                       void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace maxsim_chamfer_build_csr needs. */
size_t maxsim_chamfer_csr_workspace_size(int64_t total_src, int64_t total_dst);

/*
 * Inverse-grid CSR of a nearest-neighbour map (Flash-MaxSim §4.2.2 applied
 * to Chamfer): source point i of item b (cu_src[b] <= i < cu_src[b+1])
 * points at destination r = cu_dst[b] + arg[i]; sources with arg -1 are
 * left out.
 *   row_ptr  int32 [total_dst + 1]: sources with destination < r.
 *   col_idx  int32 [total_src]: the first row_ptr[total_dst] entries are the
 *            sources ordered by destination, ascending source index within
 *            one (a stable argsort); the rest is scratch.
 * Built with a stable LSD radix sort (8-bit digits), no floating point and
 * no order-dependent atomics.  An arg outside [-1, |dst_b|) sets the status
 * word (code 0x201) and the source is left out.
 */
maxsim_status_t maxsim_chamfer_build_csr(const int32_t *arg, const int32_t *cu_src, const int32_t *cu_dst,
                                         int32_t n_items, int64_t total_src, int64_t total_dst,
                                         int32_t *row_ptr, int32_t *col_idx,
                                         void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace maxsim_chamfer_backward needs. */
size_t maxsim_chamfer_backward_workspace_size(int64_t total_p, int64_t total_q);

/*
 * Backward of sum_b grad_cd[b] * CD_b through the saved nearest-neighbour
 * indices: both CSRs are built, then each point's gradient is written once
 * by its owner (no atomics):
 *   dP[p] = 2 g / N_b (p - Q[arg_pq[p]])  +  2 g / M_b  sum_{q : arg_qp[q] = p} (p - q)
 * and symmetrically for dQ; FP32, own term first, then the CSR sources in
 * ascending order.
 *   grad_cd  FP32 [n_items];  dP [total_p, 3], dQ [total_q, 3] FP32,
 *   written in full.
 */
maxsim_status_t maxsim_chamfer_backward(const float *grad_cd, const float *P, const int32_t *cu_p,
                                        const float *Q, const int32_t *cu_q, int32_t n_items,
                                        int64_t total_p, int64_t total_q,
                                        const int32_t *arg_pq, const int32_t *arg_qp, float *dP, float *dQ,
                                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * Training forward: maxsim_forward (FP16/BF16, argmax required) that also
 * counts, in its epilogue, the sources of the backward's inverse-grid CSR.
 * Flash-MaxSim §4.2.2 derives that CSR from the saved argmax during the
 * training step; counting while the argmax is produced saves the backward
 * one pass over it.  The counts go into `backward_workspace` (at least
 * maxsim_backward_workspace_size() bytes), which must then be handed,
 * unchanged, to maxsim_backward_with_counts together with this call's
 * argmax.  `workspace` is the forward's own scratch, as for maxsim_forward.
 * Scores and argmax are identical to maxsim_forward's.  The backward now
 * sorts each document's sources itself in shared memory (see
 * maxsim_backward) and needs no counts, so nothing is counted: this pair is
 * maxsim_forward / maxsim_backward under the names of the training pair.
 */
maxsim_status_t maxsim_forward_with_counts(const void *Q, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                                           const void *D, const int32_t *cu_seqlens, int32_t n_docs,
                                           int64_t total_d_tokens, int32_t dim, maxsim_dtype_t dtype,
                                           float *scores, int32_t *argmax,
                                           void *workspace, size_t workspace_bytes,
                                           void *backward_workspace, size_t backward_workspace_bytes,
                                           void *stream);

/*
 * maxsim_backward after maxsim_forward_with_counts: the same arguments and
 * results, with `workspace` the forward's `backward_workspace` (identical to
 * maxsim_backward: see maxsim_forward_with_counts).
 */
maxsim_status_t maxsim_backward_with_counts(const float *grad_scores, const int32_t *argmax,
                                            const void *Q, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                                            const void *D, const int32_t *cu_seqlens, int32_t n_docs,
                                            int64_t total_d_tokens, int32_t dim, maxsim_dtype_t dtype,
                                            float *dQ, float *dD,
                                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * Synchronises `stream`, then reads the device status word of the current
 * device (0 = no fault); `*code` receives the raw word when non-NULL.
 * When `clear` is non-zero the word is reset to 0.  Returns MAXSIM_OK,
 * MAXSIM_ERR_DEVICE when the word is non-zero, or MAXSIM_ERR_CUDA.
 */
maxsim_status_t maxsim_device_status(void *stream, int32_t clear, int32_t *code);

/*
 * The launch layout maxsim_forward (and maxsim_forward_int8_per_token, with
 * dtype MAXSIM_INT8) would use for these sizes, computed on the host without
 * touching a device; `sm_count` is the device's SM count (152 on a GB300).
 * Writes five int32 into `layout`: M-tiles of 128 padded query rows per CTA
 * (1, 2 or 4), CTAs per SM, row groups, CTAs (token-balanced document parts)
 * per row group, and 1 when the single document stage streams as two K-block
 * halves.  All five are 0 when no forward kernel would launch (no query, no
 * document, lq_max 0 or no document token).  Returns MAXSIM_ERR_UNSUPPORTED
 * for an unknown dtype, MAXSIM_ERR_INVALID_ARGUMENT for a null `layout`,
 * negative sizes, sm_count <= 0 or sizes beyond the forward's limits.
 */
maxsim_status_t maxsim_forward_plan(int32_t n_q, int32_t lq_max, int32_t n_docs, int64_t total_d_tokens,
                                    maxsim_dtype_t dtype, int32_t with_argmax, int32_t sm_count,
                                    int32_t *layout);

/*
 * A plain read of an L2-resident buffer, to measure the rate at which the
 * SMs can read from L2 -- the bound of the backward's row gathers (each
 * gradient row is a sum of 256-byte rows gathered from an L2-resident Q or
 * D).  The pages have no counterpart; it is a measuring stick for the
 * roofline of those kernels.  Enqueues one kernel of 2 CTAs per SM (at most
 * 1024) that streams the `bytes` of `buf` `passes` times with 16-byte loads
 * cached in L2 only, folding every word into sink[cta] (so the loads cannot be
 * elided).  Time it with events on `stream`: rate = passes * bytes / time.
 * For the rate to be L2's, `bytes` must fit in L2 with room to spare (on a
 * GB300, 126 MB of L2: 32-64 MB) and a first pass should warm it.
 *   buf     device, 16-byte aligned; bytes a multiple of 16, >= 16.
 *   sink    device uint64 [1024], caller-owned, XOR-accumulated (any
 *           initial contents).
 * Returns MAXSIM_ERR_INVALID_ARGUMENT for a bad argument, MAXSIM_ERR_CUDA on a
 * launch failure, else MAXSIM_OK.
 */
maxsim_status_t maxsim_probe_l2_read(const void *buf, size_t bytes, int32_t passes, uint64_t *sink,
                                     void *stream);

/*
 * Self-test of the kernels' failure path (no fault is involved): enqueues on
 * `stream` one CTA that holds tensor memory and waits on a barrier nothing
 * completes.  Its bounded wait gives up after `limit_us` microseconds
 * (1 .. 1,000,000), raises the CTA's abort flag (a second waiter returns on
 * it), records 0x105 in the device status word, releases the tensor memory
 * and exits.  Afterwards maxsim_device_status reports 0x105 and every entry
 * point works as before.  Returns MAXSIM_ERR_INVALID_ARGUMENT for a limit
 * out of range, MAXSIM_ERR_CUDA on a launch failure, else MAXSIM_OK.
 */
maxsim_status_t maxsim_selftest_bounded_wait(uint32_t limit_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MAXSIM_H_ */
