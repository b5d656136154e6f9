// internal.cuh -- declarations shared between the host layer and the kernel
// translation units of the MaxSim library (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace maxsim {

// Query rows of all queries are laid out "padded": query q, token i sits at
// padded row rho = q * lq_pad + i, where lq_pad is lq_max rounded up to a
// power of two (lq_max <= 32) or to a multiple of 32 (lq_max > 32), so a
// 32-row warp slice never mixes a query's tokens with another query's
// unless whole queries share it.
struct FwdParams {
    const int32_t *q_lens;
    const int32_t *cu_seqlens;
    float *scores;       // [n_q, ld_out], columns [0, n_docs) written
    float *partials;     // [lq_pad / 32, n_q, n_docs] when lq_pad > 32
    int64_t *ipartials;  // INT8: [lq_pad / 32, n_q, n_docs] int64 when lq_pad > 32
    int64_t *raw_scores; // INT8 only, may be null; [n_q, ld_out]
    int32_t *argmax;     // [n_q, ld_out, lq_max] or null
    const float *q_tok_scale;  // INT8 per-token mode: [n_q, lq_max] query-token scales
    const float *d_tok_scale;  // INT8 per-token mode: [total_tokens] document-token scales
    int32_t *status;     // device status word
    int32_t n_q, lq_max, lq_pad, n_docs;
    int32_t total_tokens;
    int64_t ld_out;         // documents per output row (>= n_docs)
    int32_t groups, parts;  // grid = groups * parts CTAs
    int32_t ksplit;         // two-M-tile 16-bit launch: stream K-blocks as half-stages
    uint32_t idesc;         // tcgen05 instruction descriptor
    double int8_scale;      // (double)q_scale * (double)d_scale
};

// Number of 128-row M-tiles one CTA holds (1, 2 or 4) for R padded rows.
// 16-bit: two CTAs of two M-tiles per SM, except for 257-384 rows, where one
// CTA of four M-tiles (one of them empty) finishes sooner than two groups of
// two.  With several row groups every group gets the same share of the SMs,
// so a part-filled last group of four saves no time.  INT8 keeps four above
// 256 rows (its two-M-tile form runs one CTA per SM).
inline int forward_mtiles(int64_t rows, bool int8) {
    if (rows <= 128) return 1;
    if (rows <= 256) return 2;
    return (int8 || rows <= 384) ? 4 : 2;
}

// Half-stage (K-block) streaming at two M-tiles: it hides part of the load
// latency of the single document stage, which pays where loads set the pace:
// without argmax, or with long documents (few boundaries, rare argmax
// searches: 1024-token pages 2.19 -> 2.11 ms).  Where the argmax epilogue sets
// the pace (documents of a few hundred tokens) it gains nothing and costs up
// to 2% (256 x 32 queries vs 180-token documents).
inline bool forward_ksplit(bool with_argmax, int64_t total_tokens, int64_t n_docs) {
    return !with_argmax || total_tokens >= 512 * n_docs;
}

// fwd_tc.cu
int forward_smem_bytes(int nmt, bool int8);
int forward_threads(int nmt, bool int8);
bool forward_stage_split(int nmt, bool int8);  // the configuration can stream K-block halves
int forward_ctas_per_sm(int nmt, bool int8);   // CTAs one SM runs at once
// Forward arithmetic: FP16/BF16 MMA on the inputs; INT8 with one scale per
// tensor (exact integer maxima, int64 sums); INT8 with one scale per token
// (exact integer dots scaled per document token in FP32 before the maximum,
// per query token after it, FP32 sums).
enum class FwdMode { kF16 = 0, kInt8Tensor = 1, kInt8Token = 2 };
cudaError_t launch_forward(const CUtensorMap &tmQ, const CUtensorMap &tmD, const FwdParams &p,
                           int nmt, bool with_argmax, FwdMode mode, cudaStream_t stream);
cudaError_t launch_finalize_partials(const FwdParams &p, bool int8, cudaStream_t stream);
cudaError_t launch_fill_empty(const FwdParams &p, bool int8, cudaStream_t stream);
cudaError_t launch_int8_to_f16(const int8_t *src, uint16_t *dst, int64_t n, cudaStream_t stream);
cudaError_t launch_rebase_offsets(const int32_t *src, int32_t *dst, int32_t n, cudaStream_t stream);
// One CTA holding TMEM waits on an mbarrier that nothing completes: the
// bounded wait must give up after limit_ns and record kStatusSelfTestExpired.
cudaError_t launch_wait_selftest(int32_t *status, uint64_t limit_ns, cudaStream_t stream);

// topk.cu
constexpr int kTopkMax = 4096;  // largest k a row-wise top-K selection takes
cudaError_t launch_topk(const float *values, int64_t ld, int32_t n_rows, int32_t n_cols, int32_t k,
                        const int32_t *col_ids, int64_t ld_ids, int32_t *out_ids, float *out_values,
                        cudaStream_t stream);
cudaError_t launch_candidate_offsets(const int32_t *cand, int32_t n_q, int32_t n_cand, const int32_t *cu,
                                     int32_t max_len, int32_t *cand_cu, int32_t *status, cudaStream_t stream);
cudaError_t launch_gather_candidates(const int32_t *cand, int32_t n_q, int32_t n_cand, const int32_t *cu,
                                     const int32_t *cand_cu, const void *src, int64_t row_bytes, void *dst,
                                     int64_t slice_rows, int sm_count, cudaStream_t stream);

// chamfer.cu
int chamfer_slices(int32_t n_items, int32_t max_s, int32_t max_t, int sm_count);
cudaError_t launch_chamfer_nn(const float *S, const int32_t *cu_s, const float *T, const int32_t *cu_t,
                              int32_t n_items, int32_t max_s, int32_t max_t, int64_t total_s, int slices,
                              float *dist, int32_t *arg, float *part_d, int32_t *part_a, int32_t *status,
                              cudaStream_t stream);
cudaError_t launch_chamfer_reduce(const float *dist_pq, const int32_t *cu_p, const float *dist_qp,
                                  const int32_t *cu_q, int32_t n_items, float *cd, cudaStream_t stream);
size_t chamfer_csr_scratch_bytes(int64_t total_src, int32_t total_dst);
cudaError_t launch_chamfer_csr(const int32_t *arg, const int32_t *cu_src, const int32_t *cu_dst, int32_t n_items,
                               int64_t total_src, int32_t total_dst, int32_t *row_ptr, int32_t *col_idx,
                               void *scratch, int32_t *status, cudaStream_t stream);
cudaError_t launch_chamfer_grad(const float *grad, const float *A, const int32_t *cu_a, const float *B,
                                const int32_t *cu_b, int32_t n_items, const int32_t *arg_ab,
                                const int32_t *row_ptr_ba, const int32_t *col_ba, int64_t total_a, float *dA,
                                cudaStream_t stream);

// bwd.cu
struct BwdParams {
    const float *grad;       // [n_q, n_docs]
    const int32_t *argmax;   // [n_q, n_docs, lq_max]
    const void *Q;           // [n_q, lq_max, 128] fp16/bf16
    const void *D;           // [total, 128]
    const int32_t *q_lens;
    const int32_t *cu_seqlens;
    float *dQ;               // [n_q, lq_max, 128]
    float *dD;               // [total, 128]
    int32_t *row_ptr;        // [total + 1]
    int32_t *col_idx;        // [n_q * n_docs * lq_max]
    int32_t *doc_count;      // [n_docs + 1] scratch: sources per document, then offsets
    int32_t *chunk_cnt;      // [chunks * total] scratch: per-chunk token counts, then first slots
    int32_t *row_start;      // first col_idx slot of (chunk, token)'s sources, at run_bound_index
    int32_t *row_end;        // one past the last
    float *col_w;            // [n_docs * n_q * lq_max]: the backward's sorted sources' g[q, b]
    int32_t sort_chunks, sort_chunk_len;   // candidate chunks per document of the backward's sort
    int32_t *status;
    int32_t n_q, lq_max, n_docs, total_tokens;
    int32_t chunks;          // candidate chunks per document (csr_chunks)
    int32_t bf16;
    uint32_t lq_magic, lq_shift;  // k / lq_max == (k * lq_magic) >> (31 + lq_shift) for 0 <= k < 2^31
};

// Division by a fixed divisor d >= 1 for numerators below 2^31 (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994):
// s = ceil(log2 d), m = ceil(2^(31+s) / d); then m * d - 2^(31+s) < d <= 2^s,
// which makes floor(n * m / 2^(31+s)) == floor(n / d) for 0 <= n < 2^31.
inline void make_divisor(int32_t d, uint32_t &m, uint32_t &s) {
    s = 0;
    while ((int64_t{1} << s) < d) ++s;
    m = static_cast<uint32_t>(((uint64_t{1} << (31 + s)) + static_cast<uint64_t>(d) - 1) / static_cast<uint64_t>(d));
}
int csr_chunks(int32_t n_q, int32_t lq_max, int32_t n_docs);
// Longest document the CSR build handles (its shared-memory histograms);
// longer ones get empty rows and a status code.
constexpr int kCsrMaxDocTokens = 24 * 1024;
// The exact CSR (maxsim_build_csr): chunked per-document counting sort.
cudaError_t launch_build_csr(const BwdParams &p, cudaStream_t stream);
// dQ: one warp per dQ row, reading its argmax entries directly.
cudaError_t launch_grad_q(const BwdParams &p, cudaStream_t stream);
// The backward's inverse map and dD: each document's n_q * lq_max candidates
// in C = sort_chunks() chunks (about kSortChunkTarget each, at most
// kSortMaxChunks chunks of at most kSortMaxChunkLen), sorted per (document,
// chunk) in shared memory into fixed slots of col_idx (their g[q, b] in the
// same slots of col_w), with per-(chunk, token) run bounds in row_start /
// row_end; then one warp per dD row, kRunBlock rows per CTA.
constexpr int kSortChunkTarget = 2048;
// Run bounds of token t in chunk c (of C) sit at run_bound_index: blocks of
// kRunBlock consecutive tokens per chunk, chunk after chunk, so a sorting CTA
// (one chunk) writes whole 32-byte sectors and a dD CTA (kRunBlock
// consecutive rows) finds its rows' bounds of every chunk in one contiguous
// range.  Arrays hold C * round_up(total, kRunBlock) words.
constexpr int kRunBlock = 8;
__host__ __device__ inline int64_t run_bound_index(int64_t t, int c, int C) {
    return ((t / kRunBlock) * C + c) * kRunBlock + (t % kRunBlock);
}
constexpr int kSortMaxChunks = 32;
constexpr int kSortMaxChunkLen = 15360;   // tokens and staged output: 120 KB of shared memory
constexpr int64_t kBackwardMaxCandidates = int64_t{kSortMaxChunks} * kSortMaxChunkLen;
// The sort's window: 1024 tokens when documents average more than 256, else 256.
inline bool sort_long_docs(int64_t total_tokens, int32_t n_docs) {
    return total_tokens > 256 * static_cast<int64_t>(n_docs);
}
int sort_chunks(int32_t n_q, int32_t lq_max);
cudaError_t launch_sort_and_grad_d(const BwdParams &p, cudaStream_t stream);
// Streams `bytes` of `buf` (16-byte aligned, a multiple of 16) `passes` times
// with `ctas` CTAs of 512 threads, folding the words into sink[0 .. ctas).
cudaError_t launch_l2_read_probe(const void *buf, size_t bytes, int passes, unsigned long long *sink, int ctas,
                                 cudaStream_t stream);

}  // namespace maxsim
