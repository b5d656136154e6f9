// maxsim_api.cu -- the C ABI declared in include/maxsim.h: argument checks,
// TMA descriptor encoding, shape-based configuration and launches.  The
// library allocates nothing; all scratch comes from caller workspaces.
#include "maxsim.h"

#include "internal.cuh"
#include "sm103.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <unordered_map>
#include <vector>

namespace maxsim {

// Device status word: 0 = healthy; kernels record a code here on a pipeline
// timeout or an out-of-range argmax (see sm103.cuh for the codes).
__device__ int32_t g_status_word = 0;

namespace {

constexpr int kDim = 128;
constexpr size_t kAlign = 256;
constexpr int kProbeSinkWords = 1024;   // the L2 probe's sink: one word per CTA

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct DeviceInfo {
    int sm_count = 0;
    int32_t *status = nullptr;
};

std::mutex g_mu;
std::unordered_map<int, DeviceInfo> g_devices;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

maxsim_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MAXSIM_OK : MAXSIM_ERR_CUDA; }

maxsim_status_t device_info(DeviceInfo *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MAXSIM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_devices.find(dev);
    if (it == g_devices.end()) {
        DeviceInfo di;
        if (cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&di.status), g_status_word) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        it = g_devices.emplace(dev, di).first;
    }
    if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return MAXSIM_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = it->second;
    return MAXSIM_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A non-blocking stream per device (and the two events that fork work onto
// it from a caller's stream and join it back), created on first use with the
// device current and kept for the life of the process.  g_side_mu serialises
// the fork / launch / join sequences of concurrent callers.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;
std::unordered_map<int, SideStream> g_side;

maxsim_status_t side_stream(SideStream *out) {   // caller holds g_side_mu
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MAXSIM_ERR_CUDA;
    auto it = g_side.find(dev);
    if (it == g_side.end()) {
        SideStream s;
        if (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess) return MAXSIM_ERR_CUDA;
        if (cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        it = g_side.emplace(dev, s).first;
    }
    *out = it->second;
    return MAXSIM_OK;
}

int lq_padded(int lq_max) {
    if (lq_max <= 32) {
        int v = 1;
        while (v < lq_max) v <<= 1;
        return v;
    }
    return (lq_max + 31) / 32 * 32;
}

// Rank-3 map over Q [n_q][lq_max][128] (16-bit elements): a box is one
// 64-column K-block of 32 padded query rows -- 32 tokens of one query, or
// 32 / lq_pad whole queries of lq_pad tokens; rows past lq_max or n_q read 0.
maxsim_status_t encode_q(CUtensorMap *map, const void *Q, int n_q, int lq_max, int lq_pad, bool bf16) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(lq_max),
                          static_cast<cuuint64_t>(n_q)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDim) * 2,
                             static_cast<cuuint64_t>(lq_max) * kDim * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(std::min(32, lq_pad)),
                         static_cast<cuuint32_t>(std::max(1, 32 / lq_pad))};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                          const_cast<void *>(Q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

// Rank-2 map over the packed D [total][128]: 16-bit -> boxes of 64 columns x
// box_rows tokens; int8 -> boxes of 128 columns x box_rows tokens.  Rows past
// the end read 0 and are masked by the kernel.
maxsim_status_t encode_d(CUtensorMap *map, const void *D, int64_t total, maxsim_dtype_t dtype,
                         uint32_t box_rows) {
    const bool i8 = dtype == MAXSIM_INT8;
    const cuuint64_t esize = i8 ? 1 : 2;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(total)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDim) * esize};
    cuuint32_t box[2] = {i8 ? 128u : 64u, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUtensorMapDataType t = i8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                               : (dtype == MAXSIM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    CUresult r = g_encode(map, t, 2, const_cast<void *>(D), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MAXSIM_OK : MAXSIM_ERR_CUDA;
}

struct FwdLayout {
    size_t partials = 0;   // bytes of per-chunk partial sums
    size_t q16 = 0;        // bytes of the FP16 copy of an INT8 Q
    size_t total = 0;
};

FwdLayout forward_layout(int32_t n_q, int32_t lq_max, int32_t n_docs, maxsim_dtype_t dtype) {
    FwdLayout l;
    if (n_q <= 0 || n_docs <= 0 || lq_max <= 0) return l;
    const int lq_pad = lq_padded(lq_max);
    if (lq_pad > 32)
        l.partials = align_up(static_cast<size_t>(lq_pad / 32) * n_q * n_docs *
                              (dtype == MAXSIM_INT8 ? sizeof(int64_t) : sizeof(float)));
    if (dtype == MAXSIM_INT8) l.q16 = align_up(static_cast<size_t>(n_q) * lq_max * kDim * 2);
    l.total = l.partials + l.q16;
    return l;
}

// Backward / CSR scratch: the CSR (row_ptr, col_idx) and its per-document
// and per-chunk counts; the backward's own sort fills col_idx in
// per-(document, chunk) slots instead, with the sources' weights in a second
// array of the same size and the runs' bounds.
struct BwdLayout {
    size_t row_ptr = 0, col_idx = 0, doc_count = 0, chunk_cnt = 0, row_bounds = 0, total = 0;
};

BwdLayout backward_layout(int32_t n_q, int32_t lq_max, int32_t n_docs, int64_t total) {
    BwdLayout l;
    l.row_ptr = align_up(static_cast<size_t>(total + 1) * 4);
    l.col_idx = align_up(static_cast<size_t>(std::max<int64_t>(1, int64_t(n_q) * n_docs * lq_max)) * 4);
    l.doc_count = align_up(static_cast<size_t>(n_docs + 1) * 4);
    l.chunk_cnt = align_up(static_cast<size_t>(csr_chunks(n_q, lq_max, n_docs)) * std::max<int64_t>(total, 1) * 4);
    // run bounds in blocks of kRunBlock tokens per chunk (run_bound_index)
    l.row_bounds = align_up(static_cast<size_t>(sort_chunks(n_q, lq_max)) *
                            ((std::max<int64_t>(total, 1) + kRunBlock - 1) / kRunBlock * kRunBlock) * 4);
    l.total = l.row_ptr + 2 * l.col_idx + l.doc_count + l.chunk_cnt + 2 * l.row_bounds;
    return l;
}

// Staging layout of maxsim_forward_host: two D blocks (double buffer), the
// corpus's offsets copied once, the current block's rebased offsets, one
// set of per-chunk partials (the forwards run in order on one stream) and
// the FP16 copy of an INT8 Q.
struct HostLayout {
    size_t stage_off[2] = {0, 0};
    size_t cu_all_off = 0, cu_block_off = 0, partials_off = 0, q16_off = 0, total = 0;
};

HostLayout host_layout(int32_t n_q, int32_t lq_max, int32_t n_docs, int32_t block_docs, int64_t block_tokens,
                       maxsim_dtype_t dtype) {
    HostLayout h;
    const size_t stage = align_up(static_cast<size_t>(block_tokens) * kDim * (dtype == MAXSIM_INT8 ? 1 : 2));
    const FwdLayout f = forward_layout(n_q, std::max(lq_max, 1), block_docs, dtype);
    size_t off = 0;
    h.stage_off[0] = off;
    off += stage;
    h.stage_off[1] = off;
    off += stage;
    h.cu_all_off = off;
    off += align_up(static_cast<size_t>(n_docs + 1) * sizeof(int32_t));
    h.cu_block_off = off;
    off += align_up(static_cast<size_t>(block_docs + 1) * sizeof(int32_t));
    h.partials_off = off;
    off += f.partials;
    h.q16_off = off;
    off += f.q16;
    h.total = off;
    return h;
}

// Greedy split of documents [0, n_docs) into consecutive blocks; starts gets
// the first document of each block followed by n_docs.
maxsim_status_t plan_host_blocks(const int32_t *cu, int32_t n_docs, int64_t total, int32_t block_docs,
                                 int64_t block_tokens, std::vector<int32_t> &starts) {
    if (cu[0] != 0 || cu[n_docs] != total) return MAXSIM_ERR_INVALID_ARGUMENT;
    starts.clear();
    starts.push_back(0);
    int32_t b0 = 0;
    for (int32_t b = 0; b < n_docs; ++b) {
        const int64_t len = static_cast<int64_t>(cu[b + 1]) - cu[b];
        if (len < 0 || len > block_tokens) return MAXSIM_ERR_INVALID_ARGUMENT;
        if (b - b0 == block_docs || static_cast<int64_t>(cu[b + 1]) - cu[b0] > block_tokens) {
            starts.push_back(b);
            b0 = b;
        }
    }
    starts.push_back(n_docs);
    return MAXSIM_OK;
}

// Events of one maxsim_forward_host call; destroyed when the call returns
// (the runtime releases an event still pending once the device reaches it).
struct EventSet {
    cudaEvent_t start = nullptr, copied[2] = {nullptr, nullptr}, computed[2] = {nullptr, nullptr};
    cudaError_t create(bool needed) {
        if (!needed) return cudaSuccess;
        for (cudaEvent_t *e : {&start, &copied[0], &copied[1], &computed[0], &computed[1]}) {
            cudaError_t r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
            if (r != cudaSuccess) return r;
        }
        return cudaSuccess;
    }
    ~EventSet() {
        for (cudaEvent_t e : {start, copied[0], copied[1], computed[0], computed[1]})
            if (e) cudaEventDestroy(e);
    }
};

// The size limits of every forward: non-negative sizes, a token count the
// kernels' 32-bit row indices cover, padded query rows within int32 and the
// argmax element count within int64 bytes.
maxsim_status_t check_forward_sizes(int32_t n_q, int32_t lq_max, int32_t n_docs, int64_t total_d_tokens) {
    if (n_q < 0 || n_docs < 0 || lq_max < 0 || total_d_tokens < 0) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (total_d_tokens > INT32_MAX - 256) return MAXSIM_ERR_INVALID_ARGUMENT;
    const int64_t rows = static_cast<int64_t>(n_q) * (lq_max > 0 ? lq_padded(lq_max) : 1);
    if (rows > INT32_MAX / 2 || static_cast<int64_t>(n_q) * n_docs * std::max(1, lq_max) > INT64_MAX / 8)
        return MAXSIM_ERR_INVALID_ARGUMENT;
    return MAXSIM_OK;
}

maxsim_status_t check_forward_args(const void *Q, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                                   int32_t n_docs, int64_t total_d_tokens, int32_t dim, maxsim_dtype_t dtype,
                                   float q_scale, float d_scale) {
    if (dtype != MAXSIM_FP16 && dtype != MAXSIM_BF16 && dtype != MAXSIM_INT8) return MAXSIM_ERR_UNSUPPORTED;
    if (dim != kDim) return MAXSIM_ERR_UNSUPPORTED;
    const maxsim_status_t st = check_forward_sizes(n_q, lq_max, n_docs, total_d_tokens);
    if (st != MAXSIM_OK) return st;
    if (n_q == 0 || n_docs == 0) return MAXSIM_OK;
    if (!q_lens) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (lq_max > 0 && (!Q || !aligned16(Q))) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (dtype == MAXSIM_INT8 && !(q_scale > 0.0f && d_scale > 0.0f)) return MAXSIM_ERR_INVALID_ARGUMENT;
    return MAXSIM_OK;
}

// Grid of one forward launch: row groups of nmt * 128 padded rows, each
// group's documents split into token-balanced parts (one CTA per group and
// part, enough parts to fill ctas_per_sm CTAs on every SM), and whether the
// single document stage streams as K-block halves.
struct LaunchLayout {
    int nmt = 0, ctas_per_sm = 0;
    int64_t groups = 0, parts = 0;
    bool ksplit = false;
};

LaunchLayout launch_layout(int64_t rows, int nmt, bool int8, int sm_count, bool with_argmax, int64_t total,
                           int64_t n_docs) {
    LaunchLayout l;
    l.nmt = nmt;
    l.ctas_per_sm = forward_ctas_per_sm(nmt, int8);
    l.groups = (rows + nmt * 128 - 1) / (nmt * 128);
    l.parts = std::max<int64_t>(1, static_cast<int64_t>(l.ctas_per_sm) * sm_count / l.groups);
    l.ksplit = forward_stage_split(nmt, int8) && forward_ksplit(with_argmax, total, n_docs);
    return l;
}

// What a forward over any set of documents shares: the query side (its
// tensor map, the FP16 widening of an INT8 Q), the tile configuration and
// the partial-sum scratch.
struct ForwardPlan {
    FwdParams p{};
    alignas(64) CUtensorMap tmQ;
    int nmt = 1;
    int sm_count = 0;
    bool int8 = false, empty_q = false;
    FwdMode mode = FwdMode::kF16;
    maxsim_dtype_t dtype = MAXSIM_FP16;
};

maxsim_status_t forward_prepare(ForwardPlan &plan, const void *Q, const int32_t *q_lens, int32_t n_q,
                                int32_t lq_max, maxsim_dtype_t dtype, float q_scale, float d_scale,
                                uint8_t *partials, uint8_t *q16_scratch, cudaStream_t stream,
                                const float *q_tok_scale = nullptr) {
    DeviceInfo di;
    maxsim_status_t st = device_info(&di);
    if (st != MAXSIM_OK) return st;
    const bool int8 = dtype == MAXSIM_INT8;
    const int lq_pad = lq_max > 0 ? lq_padded(lq_max) : 1;
    FwdParams &p = plan.p;
    p.q_lens = q_lens;
    p.status = di.status;
    p.n_q = n_q;
    p.lq_max = lq_max;
    p.lq_pad = lq_pad;
    p.int8_scale = int8 ? static_cast<double>(q_scale) * static_cast<double>(d_scale) : 0.0;
    plan.mode = !int8 ? FwdMode::kF16 : q_tok_scale ? FwdMode::kInt8Token : FwdMode::kInt8Tensor;
    p.q_tok_scale = q_tok_scale;
    if (lq_pad > 32) {
        if (plan.mode == FwdMode::kInt8Tensor) p.ipartials = reinterpret_cast<int64_t *>(partials);
        else p.partials = reinterpret_cast<float *>(partials);
    }
    p.idesc = ptx::idesc_f16(dtype == MAXSIM_BF16, 128, 128);
    plan.int8 = int8;
    plan.dtype = dtype;
    plan.sm_count = di.sm_count;
    plan.empty_q = lq_max == 0;
    plan.nmt = forward_mtiles(static_cast<int64_t>(n_q) * lq_pad, int8);
    if (plan.empty_q) return MAXSIM_OK;
    const void *q_src = Q;
    if (int8) {
        uint16_t *q16 = reinterpret_cast<uint16_t *>(q16_scratch);
        if (launch_int8_to_f16(static_cast<const int8_t *>(Q), q16, static_cast<int64_t>(n_q) * lq_max * kDim,
                               stream) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        q_src = q16;
    }
    return encode_q(&plan.tmQ, q_src, n_q, lq_max, lq_pad, dtype == MAXSIM_BF16);
}

// One forward over documents [0, n_docs) of (D, cu_seqlens) whose outputs
// land in columns [0, n_docs) of rows of ld_out documents.  `total` sizes the
// tensor map over D and may exceed cu_seqlens[n_docs] (the kernels balance
// work by the offsets themselves).
maxsim_status_t forward_block(ForwardPlan &plan, const void *D, const int32_t *cu_seqlens, int32_t n_docs,
                              int64_t total, float *scores, int64_t *raw_scores, int32_t *argmax,
                              int64_t ld_out, cudaStream_t stream, const float *d_tok_scale = nullptr) {
    const bool int64_sums = plan.mode == FwdMode::kInt8Tensor;
    FwdParams p = plan.p;
    p.cu_seqlens = cu_seqlens;
    p.d_tok_scale = d_tok_scale;
    p.scores = scores;
    p.raw_scores = int64_sums ? raw_scores : nullptr;
    p.argmax = argmax;
    p.n_docs = n_docs;
    p.total_tokens = static_cast<int32_t>(total);
    p.ld_out = ld_out;
    if (n_docs == 0) return MAXSIM_OK;
    if (total == 0 || plan.empty_q) return cuda_status(launch_fill_empty(p, int64_sums, stream));

    alignas(64) CUtensorMap tmD;
    maxsim_status_t st = encode_d(&tmD, D, total, plan.dtype, 128u);
    if (st != MAXSIM_OK) return st;
    const LaunchLayout l = launch_layout(static_cast<int64_t>(p.n_q) * p.lq_pad, plan.nmt, plan.int8,
                                         plan.sm_count, argmax != nullptr, total, n_docs);
    if (l.groups * l.parts > INT32_MAX) return MAXSIM_ERR_INVALID_ARGUMENT;
    p.groups = static_cast<int32_t>(l.groups);
    p.parts = static_cast<int32_t>(l.parts);
    p.ksplit = l.ksplit ? 1 : 0;
    cudaError_t e = launch_forward(plan.tmQ, tmD, p, plan.nmt, argmax != nullptr, plan.mode, stream);
    if (e != cudaSuccess) return MAXSIM_ERR_CUDA;
    if (p.lq_pad > 32) return cuda_status(launch_finalize_partials(p, int64_sums, stream));
    return MAXSIM_OK;
}

// Workspace of maxsim_rerank_two_stage: stage-1 scores and forward scratch,
// candidate ids / stage-1 values / gathered offsets, the gather buffer (one
// slice of k_candidates * max_doc_len rows per query), stage-2 scores and the
// stage-2 forward's scratch (one query at a time).
struct RerankLayout {
    size_t s1 = 0, fwd8 = 0, cand = 0, cand_val = 0, cand_cu = 0, gather = 0, s2 = 0, fwd16 = 0, total = 0;
    int64_t slice_rows = 0;
};

RerankLayout rerank_layout(int32_t n_q, int32_t lq_max, int32_t n_docs, int32_t k_cand, int32_t max_doc_len,
                           maxsim_dtype_t dtype16) {
    RerankLayout l;
    l.slice_rows = static_cast<int64_t>(k_cand) * max_doc_len;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += align_up(bytes);
        return at;
    };
    l.s1 = take(static_cast<size_t>(n_q) * n_docs * sizeof(float));
    l.fwd8 = take(forward_layout(n_q, lq_max, n_docs, MAXSIM_INT8).total);
    l.cand = take(static_cast<size_t>(n_q) * k_cand * sizeof(int32_t));
    l.cand_val = take(static_cast<size_t>(n_q) * k_cand * sizeof(float));
    l.cand_cu = take(static_cast<size_t>(n_q) * (k_cand + 1) * sizeof(int32_t));
    l.gather = take(static_cast<size_t>(n_q) * l.slice_rows * kDim * 2);
    l.s2 = take(static_cast<size_t>(n_q) * k_cand * sizeof(float));
    l.fwd16 = take(forward_layout(1, lq_max, k_cand, dtype16).total);
    l.total = off;
    return l;
}

maxsim_status_t check_chamfer_sets(int32_t n_items, int64_t total_p, int64_t total_q, int32_t max_p,
                                   int32_t max_q) {
    if (n_items < 0 || total_p < 0 || total_q < 0 || max_p < 0 || max_q < 0) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (total_p > INT32_MAX - 1 || total_q > INT32_MAX - 1) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (max_p > total_p || max_q > total_q) return MAXSIM_ERR_INVALID_ARGUMENT;
    return MAXSIM_OK;
}

struct ChamferFwdLayout {
    int slices_pq = 1, slices_qp = 1;
    size_t part_d = 0, part_a = 0, total = 0;
};

ChamferFwdLayout chamfer_fwd_layout(int32_t n_items, int64_t total_p, int64_t total_q, int32_t max_p,
                                    int32_t max_q, int sm_count) {
    ChamferFwdLayout l;
    l.slices_pq = chamfer_slices(n_items, max_p, max_q, sm_count);
    l.slices_qp = chamfer_slices(n_items, max_q, max_p, sm_count);
    const int64_t elems = std::max<int64_t>(l.slices_pq > 1 ? l.slices_pq * total_p : 0,
                                            l.slices_qp > 1 ? l.slices_qp * total_q : 0);
    l.part_d = 0;
    l.part_a = align_up(static_cast<size_t>(elems) * sizeof(float));
    l.total = l.part_a + align_up(static_cast<size_t>(elems) * sizeof(int32_t));
    return l;
}

struct ChamferBwdLayout {
    size_t row_qp = 0, col_qp = 0, row_pq = 0, col_pq = 0, scratch = 0, total = 0;
};

ChamferBwdLayout chamfer_bwd_layout(int64_t total_p, int64_t total_q) {
    ChamferBwdLayout l;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += align_up(bytes);
        return at;
    };
    l.row_qp = take(static_cast<size_t>(total_p + 1) * 4);
    l.col_qp = take(static_cast<size_t>(std::max<int64_t>(total_q, 1)) * 4);
    l.row_pq = take(static_cast<size_t>(total_q + 1) * 4);
    l.col_pq = take(static_cast<size_t>(std::max<int64_t>(total_p, 1)) * 4);
    l.scratch = take(std::max(chamfer_csr_scratch_bytes(total_q, static_cast<int32_t>(total_p)),
                              chamfer_csr_scratch_bytes(total_p, static_cast<int32_t>(total_q))));
    l.total = off;
    return l;
}

}  // namespace
}  // namespace maxsim

using namespace maxsim;

extern "C" {

int32_t maxsim_abi_version(void) { return MAXSIM_ABI_VERSION; }

const char *maxsim_status_string(maxsim_status_t s) {
    switch (s) {
        case MAXSIM_OK: return "ok";
        case MAXSIM_ERR_INVALID_ARGUMENT: return "invalid argument";
        case MAXSIM_ERR_UNSUPPORTED: return "unsupported configuration";
        case MAXSIM_ERR_WORKSPACE: return "workspace missing or too small";
        case MAXSIM_ERR_CUDA: return "CUDA runtime or driver error";
        case MAXSIM_ERR_DEVICE: return "device status word reports a fault";
    }
    return "unknown status";
}

size_t maxsim_forward_workspace_size(int32_t n_q, int32_t lq_max, int32_t n_docs, int32_t dim,
                                     maxsim_dtype_t dtype) {
    (void)dim;
    return forward_layout(n_q, lq_max, n_docs, dtype).total;
}

maxsim_status_t maxsim_forward(const void *Q, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                               const void *D, const int32_t *cu_seqlens, int32_t n_docs,
                               int64_t total_d_tokens, int32_t dim, maxsim_dtype_t dtype,
                               float q_scale, float d_scale, float *scores, int64_t *raw_scores,
                               int32_t *argmax, void *workspace, size_t workspace_bytes,
                               void *stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    maxsim_status_t st = check_forward_args(Q, q_lens, n_q, lq_max, n_docs, total_d_tokens, dim, dtype,
                                            q_scale, d_scale);
    if (st != MAXSIM_OK) return st;
    if (n_q == 0 || n_docs == 0) return MAXSIM_OK;
    if (!cu_seqlens || !scores) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (total_d_tokens > 0 && (!D || !aligned16(D))) return MAXSIM_ERR_INVALID_ARGUMENT;
    const FwdLayout wl = forward_layout(n_q, lq_max, n_docs, dtype);
    if (wl.total > 0 && (workspace == nullptr || workspace_bytes < wl.total)) return MAXSIM_ERR_WORKSPACE;

    ForwardPlan plan;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    st = forward_prepare(plan, Q, q_lens, n_q, lq_max, dtype, q_scale, d_scale, ws, ws + wl.partials,
                         stream);
    if (st != MAXSIM_OK) return st;
    return forward_block(plan, D, cu_seqlens, n_docs, total_d_tokens, scores, raw_scores, argmax, n_docs,
                         stream);
}

maxsim_status_t maxsim_forward_int8_per_token(const int8_t *Q, const float *q_scales, const int32_t *q_lens,
                                              int32_t n_q, int32_t lq_max, const int8_t *D, const float *d_scales,
                                              const int32_t *cu_seqlens, int32_t n_docs, int64_t total_d_tokens,
                                              int32_t dim, float *scores, int32_t *argmax, void *workspace,
                                              size_t workspace_bytes, void *stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    maxsim_status_t st = check_forward_args(Q, q_lens, n_q, lq_max, n_docs, total_d_tokens, dim, MAXSIM_INT8,
                                            1.0f, 1.0f);
    if (st != MAXSIM_OK) return st;
    if (n_q == 0 || n_docs == 0) return MAXSIM_OK;
    if (!cu_seqlens || !scores || (lq_max > 0 && !q_scales)) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (total_d_tokens > 0 && (!D || !aligned16(D) || !d_scales)) return MAXSIM_ERR_INVALID_ARGUMENT;
    const FwdLayout wl = forward_layout(n_q, lq_max, n_docs, MAXSIM_INT8);
    if (wl.total > 0 && (workspace == nullptr || workspace_bytes < wl.total)) return MAXSIM_ERR_WORKSPACE;
    ForwardPlan plan;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    st = forward_prepare(plan, Q, q_lens, n_q, lq_max, MAXSIM_INT8, 1.0f, 1.0f, ws, ws + wl.partials, stream,
                         q_scales);
    if (st != MAXSIM_OK) return st;
    return forward_block(plan, D, cu_seqlens, n_docs, total_d_tokens, scores, nullptr, argmax, n_docs, stream,
                         d_scales);
}

size_t maxsim_forward_host_workspace_size(int32_t n_q, int32_t lq_max, int32_t n_docs, int32_t block_docs,
                                          int64_t block_tokens, int32_t dim, maxsim_dtype_t dtype) {
    (void)dim;
    if (n_q <= 0 || lq_max < 0 || n_docs < 0 || block_docs <= 0 || block_tokens <= 0) return 0;
    return host_layout(n_q, lq_max, n_docs, block_docs, block_tokens, dtype).total;
}

maxsim_status_t maxsim_forward_host(const void *Q, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                                    const void *D_host, const int32_t *cu_seqlens_host, int32_t n_docs,
                                    int64_t total_d_tokens, int32_t dim, maxsim_dtype_t dtype,
                                    float q_scale, float d_scale, float *scores, int64_t *raw_scores,
                                    int32_t *argmax, int32_t block_docs, int64_t block_tokens,
                                    void *workspace, size_t workspace_bytes, void *stream_,
                                    void *copy_stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    cudaStream_t copy_stream = copy_stream_ ? static_cast<cudaStream_t>(copy_stream_) : stream;
    maxsim_status_t st = check_forward_args(Q, q_lens, n_q, lq_max, n_docs, total_d_tokens, dim, dtype,
                                            q_scale, d_scale);
    if (st != MAXSIM_OK) return st;
    if (block_docs <= 0 || block_tokens <= 0 || block_tokens > INT32_MAX - 256)
        return MAXSIM_ERR_INVALID_ARGUMENT;
    if (n_q == 0 || n_docs == 0) return MAXSIM_OK;
    if (!cu_seqlens_host || !scores) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (total_d_tokens > 0 && !D_host) return MAXSIM_ERR_INVALID_ARGUMENT;

    // Plan on the host: consecutive documents, at most block_docs documents
    // and block_tokens tokens per block; a document never straddles blocks.
    std::vector<int32_t> starts;
    st = plan_host_blocks(cu_seqlens_host, n_docs, total_d_tokens, block_docs, block_tokens, starts);
    if (st != MAXSIM_OK) return st;

    const HostLayout hl = host_layout(n_q, lq_max, n_docs, block_docs, block_tokens, dtype);
    if (workspace == nullptr || workspace_bytes < hl.total) return MAXSIM_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);

    ForwardPlan plan;
    st = forward_prepare(plan, Q, q_lens, n_q, lq_max, dtype, q_scale, d_scale, ws + hl.partials_off,
                         ws + hl.q16_off, stream);
    if (st != MAXSIM_OK) return st;

    // The offsets go to the device once, ordered before every block on the
    // compute stream; each block's rebased slice is made there by a kernel.
    int32_t *cu_all = reinterpret_cast<int32_t *>(ws + hl.cu_all_off);
    int32_t *cu_block = reinterpret_cast<int32_t *>(ws + hl.cu_block_off);
    cudaError_t e = cudaMemcpyAsync(cu_all, cu_seqlens_host, static_cast<size_t>(n_docs + 1) * sizeof(int32_t),
                                    cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return MAXSIM_ERR_CUDA;

    const size_t row_bytes = static_cast<size_t>(kDim) * (dtype == MAXSIM_INT8 ? 1 : 2);
    const char *d_host = static_cast<const char *>(D_host);
    EventSet ev;
    if (ev.create(copy_stream != stream) != cudaSuccess) return MAXSIM_ERR_CUDA;
    if (copy_stream != stream) {
        // The copies may overwrite staging buffers only after whatever the
        // compute stream had queued before this call.
        if ((e = cudaEventRecord(ev.start, stream)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(copy_stream, ev.start, 0)) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
    }
    const int n_blocks = static_cast<int>(starts.size()) - 1;
    for (int k = 0; k < n_blocks; ++k) {
        const int slot = k & 1;
        const int32_t b0 = starts[k], b1 = starts[k + 1];
        const int32_t nb = b1 - b0;
        const int64_t t0 = cu_seqlens_host[b0], t1 = cu_seqlens_host[b1];
        uint8_t *d_stage = ws + hl.stage_off[slot];
        // Staging slot k & 1 is free once block k - 2's forward has run.
        if (copy_stream != stream && k >= 2 &&
            (e = cudaStreamWaitEvent(copy_stream, ev.computed[slot], 0)) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        if (t1 > t0 && (e = cudaMemcpyAsync(d_stage, d_host + static_cast<size_t>(t0) * row_bytes,
                                            static_cast<size_t>(t1 - t0) * row_bytes,
                                            cudaMemcpyHostToDevice, copy_stream)) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
        if (copy_stream != stream) {
            if ((e = cudaEventRecord(ev.copied[slot], copy_stream)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(stream, ev.copied[slot], 0)) != cudaSuccess)
                return MAXSIM_ERR_CUDA;
        }
        if ((e = launch_rebase_offsets(cu_all + b0, cu_block, nb, stream)) != cudaSuccess) return MAXSIM_ERR_CUDA;
        st = forward_block(plan, d_stage, cu_block, nb, t1 - t0, scores + b0,
                           raw_scores ? raw_scores + b0 : nullptr,
                           argmax ? argmax + static_cast<int64_t>(b0) * lq_max : nullptr, n_docs, stream);
        if (st != MAXSIM_OK) return st;
        if (copy_stream != stream && (e = cudaEventRecord(ev.computed[slot], stream)) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
    }
    return MAXSIM_OK;
}

maxsim_status_t maxsim_topk(const float *values, int32_t n_rows, int32_t n_cols, int64_t ld, int32_t k,
                            int32_t *out_ids, float *out_values, void *stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (n_rows < 0 || n_cols < 0 || k < 0 || ld < n_cols) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (k > kTopkMax) return MAXSIM_ERR_UNSUPPORTED;
    if (n_rows == 0 || k == 0) return MAXSIM_OK;
    if (!out_ids || !out_values || (n_cols > 0 && !values)) return MAXSIM_ERR_INVALID_ARGUMENT;
    return cuda_status(launch_topk(values, ld, n_rows, n_cols, k, nullptr, 0, out_ids, out_values, stream));
}

size_t maxsim_rerank_workspace_size(int32_t n_q, int32_t lq_max, int32_t n_docs, int32_t k_candidates,
                                    int32_t max_doc_len, int32_t dim, maxsim_dtype_t dtype16) {
    (void)dim;
    if (n_q < 0 || lq_max < 0 || n_docs < 0 || k_candidates <= 0 || max_doc_len < 0) return 0;
    return rerank_layout(n_q, lq_max, n_docs, k_candidates, max_doc_len, dtype16).total;
}

maxsim_status_t maxsim_rerank_two_stage(const int8_t *Q8, const float *q_tok_scales, float q_scale,
                                        const int8_t *D8, const float *d_tok_scales, float d_scale,
                                        const void *Q16, const void *D16, maxsim_dtype_t dtype16,
                                        const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                                        const int32_t *cu_seqlens, int32_t n_docs, int64_t total_d_tokens,
                                        int32_t max_doc_len, int32_t dim, int32_t k_candidates, int32_t k,
                                        int32_t *top_ids, float *top_scores, int32_t *candidate_ids,
                                        void *workspace, size_t workspace_bytes, void *stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (dtype16 != MAXSIM_FP16 && dtype16 != MAXSIM_BF16) return MAXSIM_ERR_UNSUPPORTED;
    const bool per_token = q_tok_scales != nullptr || d_tok_scales != nullptr;
    if (per_token && (q_tok_scales == nullptr || (total_d_tokens > 0 && d_tok_scales == nullptr)))
        return MAXSIM_ERR_INVALID_ARGUMENT;
    maxsim_status_t st = check_forward_args(Q8, q_lens, n_q, lq_max, n_docs, total_d_tokens, dim, MAXSIM_INT8,
                                            per_token ? 1.0f : q_scale, per_token ? 1.0f : d_scale);
    if (st != MAXSIM_OK) return st;
    if (k_candidates <= 0 || k < 0 || k > k_candidates || max_doc_len < 0) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (k_candidates > kTopkMax) return MAXSIM_ERR_UNSUPPORTED;
    if (n_q == 0) return MAXSIM_OK;
    if (!cu_seqlens || !top_ids || !top_scores) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (lq_max > 0 && (!Q16 || !aligned16(Q16))) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (total_d_tokens > 0 && (!D8 || !aligned16(D8) || !D16 || !aligned16(D16)))
        return MAXSIM_ERR_INVALID_ARGUMENT;
    const RerankLayout l = rerank_layout(n_q, lq_max, n_docs, k_candidates, max_doc_len, dtype16);
    if (l.slice_rows > INT32_MAX - 256) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (workspace == nullptr || workspace_bytes < l.total) return MAXSIM_ERR_WORKSPACE;

    // The FP16/BF16 corpus is read only by the gather: device memory, or
    // page-locked host memory through its device mapping (zero-copy).
    const void *d16 = D16;
    if (total_d_tokens > 0) {
        cudaPointerAttributes attr;
        if (cudaPointerGetAttributes(&attr, D16) != cudaSuccess) return MAXSIM_ERR_INVALID_ARGUMENT;
        if (attr.type == cudaMemoryTypeUnregistered || attr.devicePointer == nullptr)
            return MAXSIM_ERR_INVALID_ARGUMENT;
        d16 = attr.devicePointer;
    }

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *s1 = reinterpret_cast<float *>(ws + l.s1);
    int32_t *cand = candidate_ids ? candidate_ids : reinterpret_cast<int32_t *>(ws + l.cand);
    float *cand_val = reinterpret_cast<float *>(ws + l.cand_val);
    int32_t *cand_cu = reinterpret_cast<int32_t *>(ws + l.cand_cu);
    uint8_t *gather = ws + l.gather;
    float *s2 = reinterpret_cast<float *>(ws + l.s2);

    // stage 1: every document, INT8
    ForwardPlan p8;
    const FwdLayout f8 = forward_layout(n_q, lq_max, n_docs, MAXSIM_INT8);
    st = forward_prepare(p8, Q8, q_lens, n_q, lq_max, MAXSIM_INT8, q_scale, d_scale, ws + l.fwd8,
                         ws + l.fwd8 + f8.partials, stream, per_token ? q_tok_scales : nullptr);
    if (st != MAXSIM_OK) return st;
    st = forward_block(p8, D8, cu_seqlens, n_docs, total_d_tokens, s1, nullptr, nullptr, n_docs, stream,
                       per_token ? d_tok_scales : nullptr);
    if (st != MAXSIM_OK) return st;
    cudaError_t e = launch_topk(s1, n_docs, n_q, n_docs, k_candidates, nullptr, 0, cand, cand_val, stream);
    if (e != cudaSuccess) return MAXSIM_ERR_CUDA;

    // stage 2: each query's candidates, gathered and rescored in FP16/BF16
    e = launch_candidate_offsets(cand, n_q, k_candidates, cu_seqlens, max_doc_len, cand_cu, p8.p.status, stream);
    if (e == cudaSuccess && total_d_tokens > 0)
        e = launch_gather_candidates(cand, n_q, k_candidates, cu_seqlens, cand_cu, d16, kDim * 2, gather,
                                     l.slice_rows, p8.sm_count, stream);
    if (e != cudaSuccess) return MAXSIM_ERR_CUDA;
    const size_t q_stride = static_cast<size_t>(lq_max) * kDim * 2;
    for (int32_t q = 0; q < n_q; ++q) {
        ForwardPlan p16;
        st = forward_prepare(p16, static_cast<const uint8_t *>(Q16) + q * q_stride, q_lens + q, 1, lq_max,
                             dtype16, 1.0f, 1.0f, ws + l.fwd16, ws + l.fwd16, stream);
        if (st != MAXSIM_OK) return st;
        st = forward_block(p16, gather + static_cast<size_t>(q) * l.slice_rows * kDim * 2,
                           cand_cu + static_cast<int64_t>(q) * (k_candidates + 1), k_candidates,
                           std::max<int64_t>(l.slice_rows, 1), s2 + static_cast<int64_t>(q) * k_candidates,
                           nullptr, nullptr, k_candidates, stream);
        if (st != MAXSIM_OK) return st;
    }
    return cuda_status(launch_topk(s2, k_candidates, n_q, k_candidates, k, cand, k_candidates, top_ids, top_scores,
                                   stream));
}

size_t maxsim_chamfer_forward_workspace_size(int32_t n_items, int64_t total_p, int64_t total_q, int32_t max_p,
                                             int32_t max_q) {
    if (check_chamfer_sets(n_items, total_p, total_q, max_p, max_q) != MAXSIM_OK) return 0;
    DeviceInfo di;
    if (device_info(&di) != MAXSIM_OK) return 0;
    return chamfer_fwd_layout(n_items, total_p, total_q, max_p, max_q, di.sm_count).total;
}

maxsim_status_t maxsim_chamfer_forward(const float *P, const int32_t *cu_p, const float *Q, const int32_t *cu_q,
                                       int32_t n_items, int64_t total_p, int64_t total_q, int32_t max_p,
                                       int32_t max_q, float *cd, float *dist_pq, int32_t *arg_pq, float *dist_qp,
                                       int32_t *arg_qp, void *workspace, size_t workspace_bytes, void *stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    maxsim_status_t st = check_chamfer_sets(n_items, total_p, total_q, max_p, max_q);
    if (st != MAXSIM_OK) return st;
    if (n_items == 0) return MAXSIM_OK;
    if (!cu_p || !cu_q || !cd || (total_p > 0 && (!P || !dist_pq || !arg_pq)) ||
        (total_q > 0 && (!Q || !dist_qp || !arg_qp)))
        return MAXSIM_ERR_INVALID_ARGUMENT;
    DeviceInfo di;
    if ((st = device_info(&di)) != MAXSIM_OK) return st;
    const ChamferFwdLayout l = chamfer_fwd_layout(n_items, total_p, total_q, max_p, max_q, di.sm_count);
    if (l.total > 0 && (workspace == nullptr || workspace_bytes < l.total)) return MAXSIM_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *part_d = reinterpret_cast<float *>(ws + l.part_d);
    int32_t *part_a = reinterpret_cast<int32_t *>(ws + l.part_a);
    cudaError_t e = launch_chamfer_nn(P, cu_p, Q, cu_q, n_items, max_p, max_q, total_p, l.slices_pq, dist_pq,
                                      arg_pq, part_d, part_a, di.status, stream);
    if (e == cudaSuccess)
        e = launch_chamfer_nn(Q, cu_q, P, cu_p, n_items, max_q, max_p, total_q, l.slices_qp, dist_qp, arg_qp,
                              part_d, part_a, di.status, stream);
    if (e == cudaSuccess) e = launch_chamfer_reduce(dist_pq, cu_p, dist_qp, cu_q, n_items, cd, stream);
    return cuda_status(e);
}

size_t maxsim_chamfer_csr_workspace_size(int64_t total_src, int64_t total_dst) {
    if (total_src < 0 || total_dst < 0 || total_dst > INT32_MAX - 1) return 0;
    return chamfer_csr_scratch_bytes(total_src, static_cast<int32_t>(total_dst));
}

maxsim_status_t maxsim_chamfer_build_csr(const int32_t *arg, const int32_t *cu_src, const int32_t *cu_dst,
                                         int32_t n_items, int64_t total_src, int64_t total_dst, int32_t *row_ptr,
                                         int32_t *col_idx, void *workspace, size_t workspace_bytes,
                                         void *stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (n_items < 0 || total_src < 0 || total_dst < 0 || total_src > INT32_MAX - 1 || total_dst > INT32_MAX - 1)
        return MAXSIM_ERR_INVALID_ARGUMENT;
    if (n_items == 0 && (total_src > 0 || total_dst > 0)) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (!row_ptr || (n_items > 0 && (!cu_src || !cu_dst)) || (total_src > 0 && (!arg || !col_idx)))
        return MAXSIM_ERR_INVALID_ARGUMENT;
    const size_t need = chamfer_csr_scratch_bytes(total_src, static_cast<int32_t>(total_dst));
    if (workspace == nullptr || workspace_bytes < need) return MAXSIM_ERR_WORKSPACE;
    DeviceInfo di;
    maxsim_status_t st = device_info(&di);
    if (st != MAXSIM_OK) return st;
    return cuda_status(launch_chamfer_csr(arg, cu_src, cu_dst, n_items, total_src, static_cast<int32_t>(total_dst),
                                          row_ptr, col_idx, workspace, di.status, stream));
}

size_t maxsim_chamfer_backward_workspace_size(int64_t total_p, int64_t total_q) {
    if (total_p < 0 || total_q < 0 || total_p > INT32_MAX - 1 || total_q > INT32_MAX - 1) return 0;
    return chamfer_bwd_layout(total_p, total_q).total;
}

maxsim_status_t maxsim_chamfer_backward(const float *grad_cd, const float *P, const int32_t *cu_p, const float *Q,
                                        const int32_t *cu_q, int32_t n_items, int64_t total_p, int64_t total_q,
                                        const int32_t *arg_pq, const int32_t *arg_qp, float *dP, float *dQ,
                                        void *workspace, size_t workspace_bytes, void *stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    maxsim_status_t st = check_chamfer_sets(n_items, total_p, total_q, 0, 0);
    if (st != MAXSIM_OK) return st;
    if (n_items == 0) return MAXSIM_OK;
    if (!grad_cd || !cu_p || !cu_q || (total_p > 0 && (!P || !arg_pq || !dP)) ||
        (total_q > 0 && (!Q || !arg_qp || !dQ)))
        return MAXSIM_ERR_INVALID_ARGUMENT;
    const ChamferBwdLayout l = chamfer_bwd_layout(total_p, total_q);
    if (workspace == nullptr || workspace_bytes < l.total) return MAXSIM_ERR_WORKSPACE;
    DeviceInfo di;
    if ((st = device_info(&di)) != MAXSIM_OK) return st;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *row_qp = reinterpret_cast<int32_t *>(ws + l.row_qp);
    int32_t *col_qp = reinterpret_cast<int32_t *>(ws + l.col_qp);
    int32_t *row_pq = reinterpret_cast<int32_t *>(ws + l.row_pq);
    int32_t *col_pq = reinterpret_cast<int32_t *>(ws + l.col_pq);
    // inverse of Q -> P (destinations in P) and of P -> Q (destinations in Q)
    cudaError_t e = launch_chamfer_csr(arg_qp, cu_q, cu_p, n_items, total_q, static_cast<int32_t>(total_p), row_qp,
                                       col_qp, ws + l.scratch, di.status, stream);
    if (e == cudaSuccess)
        e = launch_chamfer_csr(arg_pq, cu_p, cu_q, n_items, total_p, static_cast<int32_t>(total_q), row_pq, col_pq,
                               ws + l.scratch, di.status, stream);
    if (e == cudaSuccess)
        e = launch_chamfer_grad(grad_cd, P, cu_p, Q, cu_q, n_items, arg_pq, row_qp, col_qp, total_p, dP, stream);
    if (e == cudaSuccess)
        e = launch_chamfer_grad(grad_cd, Q, cu_q, P, cu_p, n_items, arg_qp, row_pq, col_pq, total_q, dQ, stream);
    return cuda_status(e);
}

size_t maxsim_backward_workspace_size(int32_t n_q, int32_t lq_max, int32_t n_docs, int64_t total_d_tokens) {
    if (n_q < 0 || lq_max < 0 || n_docs < 0 || total_d_tokens < 0) return 0;
    return backward_layout(n_q, lq_max, n_docs, total_d_tokens).total;
}

static maxsim_status_t check_csr_args(const int32_t *argmax, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                                      const int32_t *cu_seqlens, int32_t n_docs, int64_t total) {
    if (n_q < 0 || lq_max < 0 || n_docs < 0 || total < 0 || total > INT32_MAX - 256)
        return MAXSIM_ERR_INVALID_ARGUMENT;
    if (static_cast<int64_t>(n_q) * n_docs * lq_max >= INT32_MAX) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (n_q > 0 && n_docs > 0 && lq_max > 0 && (!argmax || !q_lens)) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (n_docs > 0 && !cu_seqlens) return MAXSIM_ERR_INVALID_ARGUMENT;
    return MAXSIM_OK;
}

static void fill_bwd_params(BwdParams &p, const int32_t *argmax, const int32_t *q_lens, int32_t n_q,
                            int32_t lq_max, const int32_t *cu_seqlens, int32_t n_docs, int64_t total,
                            void *workspace, const DeviceInfo &di) {
    const BwdLayout l = backward_layout(n_q, lq_max, n_docs, total);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.argmax = argmax;
    p.q_lens = q_lens;
    p.cu_seqlens = cu_seqlens;
    p.n_q = n_q;
    p.lq_max = lq_max;
    p.n_docs = n_docs;
    p.total_tokens = static_cast<int32_t>(total);
    p.row_ptr = reinterpret_cast<int32_t *>(ws);
    p.col_idx = reinterpret_cast<int32_t *>(ws + l.row_ptr);
    p.doc_count = reinterpret_cast<int32_t *>(ws + l.row_ptr + l.col_idx);
    p.chunk_cnt = reinterpret_cast<int32_t *>(ws + l.row_ptr + l.col_idx + l.doc_count);
    p.row_start = reinterpret_cast<int32_t *>(ws + l.row_ptr + l.col_idx + l.doc_count + l.chunk_cnt);
    p.row_end = reinterpret_cast<int32_t *>(ws + l.row_ptr + l.col_idx + l.doc_count + l.chunk_cnt + l.row_bounds);
    p.col_w = reinterpret_cast<float *>(ws + l.row_ptr + l.col_idx + l.doc_count + l.chunk_cnt + 2 * l.row_bounds);
    p.chunks = csr_chunks(n_q, lq_max, n_docs);
    p.sort_chunks = sort_chunks(n_q, lq_max);
    p.sort_chunk_len = static_cast<int32_t>(
        std::max<int64_t>(1, (static_cast<int64_t>(n_q) * lq_max + p.sort_chunks - 1) / p.sort_chunks));
    make_divisor(std::max(1, lq_max), p.lq_magic, p.lq_shift);
    p.status = di.status;
}

maxsim_status_t maxsim_build_csr(const int32_t *argmax, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                                 const int32_t *cu_seqlens, int32_t n_docs, int64_t total_d_tokens,
                                 int32_t *row_ptr, int32_t *col_idx, void *workspace,
                                 size_t workspace_bytes, void *stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    maxsim_status_t st = check_csr_args(argmax, q_lens, n_q, lq_max, cu_seqlens, n_docs, total_d_tokens);
    if (st != MAXSIM_OK) return st;
    if (!row_ptr || !col_idx) return MAXSIM_ERR_INVALID_ARGUMENT;
    const BwdLayout l = backward_layout(n_q, lq_max, n_docs, total_d_tokens);
    if (!workspace || workspace_bytes < l.total) return MAXSIM_ERR_WORKSPACE;
    DeviceInfo di;
    if ((st = device_info(&di)) != MAXSIM_OK) return st;
    BwdParams p{};
    fill_bwd_params(p, argmax, q_lens, n_q, lq_max, cu_seqlens, n_docs, total_d_tokens, workspace, di);
    p.row_ptr = row_ptr;
    p.col_idx = col_idx;
    return cuda_status(launch_build_csr(p, stream));
}

static maxsim_status_t backward_impl(const float *grad_scores, const int32_t *argmax, const void *Q,
                                     const int32_t *q_lens, int32_t n_q, int32_t lq_max, const void *D,
                                     const int32_t *cu_seqlens, int32_t n_docs, int64_t total_d_tokens,
                                     int32_t dim, maxsim_dtype_t dtype, float *dQ, float *dD, void *workspace,
                                     size_t workspace_bytes, cudaStream_t stream) {
    if (dtype == MAXSIM_INT8) return MAXSIM_ERR_UNSUPPORTED;
    if (dtype != MAXSIM_FP16 && dtype != MAXSIM_BF16) return MAXSIM_ERR_UNSUPPORTED;
    if (dim != kDim) return MAXSIM_ERR_UNSUPPORTED;
    maxsim_status_t st = check_csr_args(argmax, q_lens, n_q, lq_max, cu_seqlens, n_docs, total_d_tokens);
    if (st != MAXSIM_OK) return st;
    if ((n_q > 0 && lq_max > 0 && (!dQ || !Q)) || (total_d_tokens > 0 && (!dD || !D)))
        return MAXSIM_ERR_INVALID_ARGUMENT;
    // rows are read with vector loads and gradient rows written with 16-byte stores
    if ((n_q > 0 && lq_max > 0 && (!aligned16(Q) || !aligned16(dQ))) ||
        (total_d_tokens > 0 && (!aligned16(D) || !aligned16(dD))))
        return MAXSIM_ERR_INVALID_ARGUMENT;
    if (n_q > 0 && n_docs > 0 && !grad_scores) return MAXSIM_ERR_INVALID_ARGUMENT;
    // a document's candidates must fit the backward's shared-memory sort
    if (static_cast<int64_t>(n_q) * lq_max > kBackwardMaxCandidates) return MAXSIM_ERR_UNSUPPORTED;
    const BwdLayout l = backward_layout(n_q, lq_max, n_docs, total_d_tokens);
    if (!workspace || workspace_bytes < l.total) return MAXSIM_ERR_WORKSPACE;
    DeviceInfo di;
    if ((st = device_info(&di)) != MAXSIM_OK) return st;
    BwdParams p{};
    fill_bwd_params(p, argmax, q_lens, n_q, lq_max, cu_seqlens, n_docs, total_d_tokens, workspace, di);
    p.grad = grad_scores;
    p.Q = Q;
    p.D = D;
    p.dQ = dQ;
    p.dD = dD;
    p.bf16 = dtype == MAXSIM_BF16;
    // dQ needs only the argmax: it runs on the device's side stream, forked
    // from and joined back into `stream`, while dD's (latency-bound) sort and
    // its reduction run here
    std::lock_guard<std::mutex> lock(g_side_mu);
    SideStream side;
    if ((st = side_stream(&side)) != MAXSIM_OK) return st;
    cudaError_t e = cudaEventRecord(side.fork, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side.stream, side.fork, 0);
    if (e == cudaSuccess) e = launch_grad_q(p, side.stream);
    if (e == cudaSuccess) e = cudaEventRecord(side.join, side.stream);
    if (e != cudaSuccess) return MAXSIM_ERR_CUDA;
    e = launch_sort_and_grad_d(p, stream);
    const cudaError_t j = cudaStreamWaitEvent(stream, side.join, 0);   // joined even if a launch failed
    return cuda_status(e != cudaSuccess ? e : j);
}

maxsim_status_t maxsim_backward(const float *grad_scores, const int32_t *argmax, const void *Q,
                                const int32_t *q_lens, int32_t n_q, int32_t lq_max, const void *D,
                                const int32_t *cu_seqlens, int32_t n_docs, int64_t total_d_tokens,
                                int32_t dim, maxsim_dtype_t dtype, float *dQ, float *dD, void *workspace,
                                size_t workspace_bytes, void *stream_) {
    return backward_impl(grad_scores, argmax, Q, q_lens, n_q, lq_max, D, cu_seqlens, n_docs, total_d_tokens, dim,
                         dtype, dQ, dD, workspace, workspace_bytes, static_cast<cudaStream_t>(stream_));
}

maxsim_status_t maxsim_forward_with_counts(const void *Q, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                                           const void *D, const int32_t *cu_seqlens, int32_t n_docs,
                                           int64_t total_d_tokens, int32_t dim, maxsim_dtype_t dtype,
                                           float *scores, int32_t *argmax, void *workspace,
                                           size_t workspace_bytes, void *backward_workspace,
                                           size_t backward_workspace_bytes, void *stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (dtype != MAXSIM_FP16 && dtype != MAXSIM_BF16) return MAXSIM_ERR_UNSUPPORTED;
    maxsim_status_t st = check_forward_args(Q, q_lens, n_q, lq_max, n_docs, total_d_tokens, dim, dtype, 1.0f,
                                            1.0f);
    if (st != MAXSIM_OK) return st;
    if ((st = check_csr_args(argmax, q_lens, n_q, lq_max, cu_seqlens, n_docs, total_d_tokens)) != MAXSIM_OK)
        return st;
    if (n_q == 0 || n_docs == 0) return MAXSIM_OK;
    if (!cu_seqlens || !scores || !argmax) return MAXSIM_ERR_INVALID_ARGUMENT;
    if (total_d_tokens > 0 && (!D || !aligned16(D))) return MAXSIM_ERR_INVALID_ARGUMENT;
    const FwdLayout wl = forward_layout(n_q, lq_max, n_docs, dtype);
    if (wl.total > 0 && (workspace == nullptr || workspace_bytes < wl.total)) return MAXSIM_ERR_WORKSPACE;
    const BwdLayout bl = backward_layout(n_q, lq_max, n_docs, total_d_tokens);
    if (backward_workspace == nullptr || backward_workspace_bytes < bl.total) return MAXSIM_ERR_WORKSPACE;

    ForwardPlan plan;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    st = forward_prepare(plan, Q, q_lens, n_q, lq_max, dtype, 1.0f, 1.0f, ws, ws + wl.partials, stream);
    if (st != MAXSIM_OK) return st;
    // the backward sorts each document's sources itself: nothing to count
    return forward_block(plan, D, cu_seqlens, n_docs, total_d_tokens, scores, nullptr, argmax, n_docs, stream);
}

maxsim_status_t maxsim_backward_with_counts(const float *grad_scores, const int32_t *argmax, const void *Q,
                                            const int32_t *q_lens, int32_t n_q, int32_t lq_max, const void *D,
                                            const int32_t *cu_seqlens, int32_t n_docs, int64_t total_d_tokens,
                                            int32_t dim, maxsim_dtype_t dtype, float *dQ, float *dD,
                                            void *workspace, size_t workspace_bytes, void *stream_) {
    return backward_impl(grad_scores, argmax, Q, q_lens, n_q, lq_max, D, cu_seqlens, n_docs, total_d_tokens, dim,
                         dtype, dQ, dD, workspace, workspace_bytes, static_cast<cudaStream_t>(stream_));
}

maxsim_status_t maxsim_forward_plan(int32_t n_q, int32_t lq_max, int32_t n_docs, int64_t total_d_tokens,
                                    maxsim_dtype_t dtype, int32_t with_argmax, int32_t sm_count,
                                    int32_t *layout) {
    if (dtype != MAXSIM_FP16 && dtype != MAXSIM_BF16 && dtype != MAXSIM_INT8) return MAXSIM_ERR_UNSUPPORTED;
    if (!layout || sm_count <= 0) return MAXSIM_ERR_INVALID_ARGUMENT;
    const maxsim_status_t st = check_forward_sizes(n_q, lq_max, n_docs, total_d_tokens);
    if (st != MAXSIM_OK) return st;
    for (int k = 0; k < 5; ++k) layout[k] = 0;
    if (n_q == 0 || n_docs == 0 || lq_max == 0 || total_d_tokens == 0) return MAXSIM_OK;   // no forward kernel
    const bool int8 = dtype == MAXSIM_INT8;
    const int64_t rows = static_cast<int64_t>(n_q) * lq_padded(lq_max);
    const LaunchLayout l =
        launch_layout(rows, forward_mtiles(rows, int8), int8, sm_count, with_argmax != 0, total_d_tokens, n_docs);
    if (l.groups * l.parts > INT32_MAX) return MAXSIM_ERR_INVALID_ARGUMENT;
    layout[0] = l.nmt;
    layout[1] = l.ctas_per_sm;
    layout[2] = static_cast<int32_t>(l.groups);
    layout[3] = static_cast<int32_t>(l.parts);
    layout[4] = l.ksplit ? 1 : 0;
    return MAXSIM_OK;
}

maxsim_status_t maxsim_probe_l2_read(const void *buf, size_t bytes, int32_t passes, uint64_t *sink,
                                     void *stream_) {
    if (!buf || !sink || bytes < 16 || bytes % 16 != 0 || !aligned16(buf) || passes <= 0)
        return MAXSIM_ERR_INVALID_ARGUMENT;
    DeviceInfo di;
    maxsim_status_t st = device_info(&di);
    if (st != MAXSIM_OK) return st;
    const int ctas = std::min(kProbeSinkWords, 2 * di.sm_count);
    return cuda_status(launch_l2_read_probe(buf, bytes, passes, reinterpret_cast<unsigned long long *>(sink), ctas,
                                            static_cast<cudaStream_t>(stream_)));
}

maxsim_status_t maxsim_selftest_bounded_wait(uint32_t limit_us, void *stream_) {
    if (limit_us == 0 || limit_us > 1000000u) return MAXSIM_ERR_INVALID_ARGUMENT;
    DeviceInfo di;
    maxsim_status_t st = device_info(&di);
    if (st != MAXSIM_OK) return st;
    return cuda_status(launch_wait_selftest(di.status, static_cast<uint64_t>(limit_us) * 1000u,
                                            static_cast<cudaStream_t>(stream_)));
}

maxsim_status_t maxsim_device_status(void *stream_, int32_t clear, int32_t *code) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    int32_t v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status_word, sizeof v, 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return MAXSIM_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MAXSIM_ERR_CUDA;
    if (clear && v != 0) {
        const int32_t zero = 0;
        if (cudaMemcpyToSymbolAsync(g_status_word, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream) !=
                cudaSuccess ||
            cudaStreamSynchronize(stream) != cudaSuccess)
            return MAXSIM_ERR_CUDA;
    }
    if (code) *code = v;
    return v == 0 ? MAXSIM_OK : MAXSIM_ERR_DEVICE;
}

}  // extern "C"
