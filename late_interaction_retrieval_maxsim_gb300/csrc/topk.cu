// topk.cu -- row-wise top-K selection and the candidate gather of the
// two-stage INT8 -> FP16 top-K scan ("FLASH-MAXSIM: IO-Aware Fused Kernels
// for Late-Interaction Retrieval", arXiv 2605.29517, §4.1 "Kernel Family").
//
// Top-K: one CTA per row.  Scores map to order-preserving 32-bit keys; four
// 8-bit radix passes over the row find the key T of the k-th largest entry
// (shared-memory histograms of integer counts), one pass collects every
// entry above T and the lowest-indexed entries equal to T (an ordered,
// CTA-wide ballot scan), and a bitonic sort on (key descending, column
// ascending) orders the k survivors.  The result is unique: ties go to the
// lower column.
#include "internal.cuh"
#include "sm103.cuh"

#include <algorithm>
#include <cstdint>

namespace maxsim {
namespace {

using namespace ptx;

constexpr int kTopkThreads = 1024;

// Larger float -> larger key (IEEE order; -inf is the smallest finite key).
__device__ __forceinline__ uint32_t order_key(float x) {
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__global__ void __launch_bounds__(kTopkThreads)
topk_rows_kernel(const float *__restrict__ values, int64_t ld, int32_t n_cols, int32_t k,
                 const int32_t *__restrict__ col_ids, int64_t ld_ids, int32_t *__restrict__ out_ids,
                 float *__restrict__ out_values) {
    __shared__ uint32_t hist[256];
    __shared__ uint64_t cand[kTopkMax];
    __shared__ uint32_t s_prefix, s_krem;
    __shared__ int32_t s_ngt;
    __shared__ int32_t warp_eq[kTopkThreads / 32];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t row = blockIdx.x;
    const float *x = values + row * ld;
    const int32_t *ids = col_ids ? col_ids + row * ld_ids : nullptr;
    const int kk = min(k, n_cols);
    const uint32_t neg_inf_key = order_key(-INFINITY);
    // columns mapped to no id (-1) rank as -inf
    auto key_at = [&](int c) -> uint32_t {
        if (ids && ids[c] < 0) return neg_inf_key;
        return order_key(x[c]);
    };

    uint32_t prefix = 0, mask = 0, krem = static_cast<uint32_t>(kk);
    if (kk > 0) {
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
            __syncthreads();
            for (int c = tid; c < n_cols; c += kTopkThreads) {
                const uint32_t key = key_at(c);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (warp == 0) {
                // lane l owns digits 255 - 8l down to 248 - 8l
                uint32_t cnt[8], sum = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    cnt[j] = hist[255 - 8 * lane - j];
                    sum += cnt[j];
                }
                uint32_t incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                uint32_t acc = incl - sum;  // entries whose digit lies above this lane's digits
                if (acc < krem && krem <= incl) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (krem <= acc + cnt[j]) {
                            s_prefix = prefix | (static_cast<uint32_t>(255 - 8 * lane - j) << shift);
                            s_krem = krem - acc;
                            break;
                        }
                        acc += cnt[j];
                    }
                }
            }
            __syncthreads();
            prefix = s_prefix;
            krem = s_krem;
            mask |= 255u << shift;
            __syncthreads();
        }
        // prefix = T, the k-th largest key; krem entries equal to T are needed
        const int n_gt = kk - static_cast<int>(krem);
        if (tid == 0) s_ngt = 0;
        __syncthreads();
        int eq_base = 0;
        for (int base = 0; base < n_cols; base += kTopkThreads) {
            const int c = base + tid;
            const uint32_t key = c < n_cols ? key_at(c) : 0u;
            const bool gt = c < n_cols && key > prefix;
            const bool eq = c < n_cols && key == prefix;
            if (gt) cand[atomicAdd(&s_ngt, 1)] = (static_cast<uint64_t>(~key) << 32) | static_cast<uint32_t>(c);
            const uint32_t bal = __ballot_sync(0xffffffffu, eq);
            if (lane == 0) warp_eq[warp] = __popc(bal);
            __syncthreads();
            int before = 0, total = 0;
            for (int w = 0; w < kTopkThreads / 32; ++w) {
                const int v = warp_eq[w];
                before += w < warp ? v : 0;
                total += v;
            }
            const int rank = eq_base + before + __popc(bal & ((1u << lane) - 1u));
            if (eq && rank < static_cast<int>(krem))
                cand[n_gt + rank] = (static_cast<uint64_t>(~key) << 32) | static_cast<uint32_t>(c);
            eq_base += total;
            __syncthreads();
        }
        // bitonic sort of the kk survivors (ascending composite = key
        // descending, column ascending), padded to a power of two
        int P = 1;
        while (P < kk) P <<= 1;
        for (int i = kk + tid; i < P; i += kTopkThreads) cand[i] = ~0ull;
        __syncthreads();
        for (int size = 2; size <= P; size <<= 1)
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = tid; i < P; i += kTopkThreads) {
                    const int j = i ^ stride;
                    if (j > i) {
                        const uint64_t a = cand[i], b = cand[j];
                        const bool ascending = (i & size) == 0;
                        if ((a > b) == ascending) {
                            cand[i] = b;
                            cand[j] = a;
                        }
                    }
                }
                __syncthreads();
            }
    }
    for (int j = tid; j < k; j += kTopkThreads) {
        int32_t id = -1;
        float v = -INFINITY;
        if (j < kk) {
            const uint64_t e = cand[j];
            const int c = static_cast<int>(static_cast<uint32_t>(e));
            id = ids ? ids[c] : c;
            v = id < 0 ? -INFINITY : key_value(~static_cast<uint32_t>(e >> 32));
        }
        out_ids[row * k + j] = id;
        out_values[row * k + j] = v;
    }
}

// Offsets of each query's gathered candidates: cand_cu[q][j] = sum of the
// lengths of candidates 0 .. j-1 (a candidate id of -1 has length 0).  A
// document longer than max_len is cut to max_len and recorded in the status
// word.  One CTA per query.
__global__ void __launch_bounds__(kTopkThreads)
candidate_offsets_kernel(const int32_t *__restrict__ cand, int32_t n_cand, const int32_t *__restrict__ cu,
                         int32_t max_len, int32_t *__restrict__ cand_cu, int32_t *status) {
    __shared__ int32_t warp_sum[kTopkThreads / 32];
    __shared__ int32_t s_carry;
    const int q = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t *c = cand + static_cast<int64_t>(q) * n_cand;
    int32_t *out = cand_cu + static_cast<int64_t>(q) * (n_cand + 1);
    if (tid == 0) s_carry = 0;
    __syncthreads();
    for (int base = 0; base < n_cand; base += kTopkThreads) {
        const int j = base + tid;
        int len = 0;
        if (j < n_cand && c[j] >= 0) {
            len = cu[c[j] + 1] - cu[c[j]];
            if (len > max_len) {
                atomicCAS(status, 0, kStatusDocTooLong);
                len = max_len;
            }
        }
        int incl = len;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) warp_sum[warp] = incl;
        __syncthreads();
        int before = s_carry;
        for (int w = 0; w < warp; ++w) before += warp_sum[w];
        if (j < n_cand) out[j] = before + incl - len;
        __syncthreads();
        if (tid == kTopkThreads - 1) s_carry = before + incl;
        __syncthreads();
    }
    if (tid == 0) out[n_cand] = s_carry;
}

// Copy each candidate's rows (row_bytes each) into its query's slice of the
// gather buffer: slice q starts at q * slice_rows rows.  One warp per
// candidate, 16-byte copies.  src may be device memory or page-locked host
// memory mapped into the device's address space.
__global__ void gather_candidates_kernel(const int32_t *__restrict__ cand, int32_t n_q, int32_t n_cand,
                                         const int32_t *__restrict__ cu, const int32_t *__restrict__ cand_cu,
                                         const uint8_t *__restrict__ src, int64_t row_bytes,
                                         uint8_t *__restrict__ dst, int64_t slice_rows) {
    const int lane = threadIdx.x & 31;
    const int64_t n_items = static_cast<int64_t>(n_q) * n_cand;
    for (int64_t item = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; item < n_items;
         item += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
        const int q = static_cast<int>(item / n_cand);
        const int j = static_cast<int>(item - static_cast<int64_t>(q) * n_cand);
        const int32_t id = cand[item];
        if (id < 0) continue;
        const int32_t *qcu = cand_cu + static_cast<int64_t>(q) * (n_cand + 1);
        const int64_t rows = qcu[j + 1] - qcu[j];  // already cut to the slice's limit
        const uint4 *s = reinterpret_cast<const uint4 *>(src + static_cast<int64_t>(cu[id]) * row_bytes);
        uint4 *d = reinterpret_cast<uint4 *>(dst + (static_cast<int64_t>(q) * slice_rows + qcu[j]) * row_bytes);
        const int64_t n16 = rows * row_bytes / 16;
        for (int64_t v = lane; v < n16; v += 32) d[v] = s[v];
    }
}

}  // namespace

cudaError_t launch_topk(const float *values, int64_t ld, int32_t n_rows, int32_t n_cols, int32_t k,
                        const int32_t *col_ids, int64_t ld_ids, int32_t *out_ids, float *out_values,
                        cudaStream_t stream) {
    if (n_rows == 0 || k == 0) return cudaSuccess;
    topk_rows_kernel<<<n_rows, kTopkThreads, 0, stream>>>(values, ld, n_cols, k, col_ids, ld_ids, out_ids,
                                                         out_values);
    return cudaGetLastError();
}

cudaError_t launch_candidate_offsets(const int32_t *cand, int32_t n_q, int32_t n_cand, const int32_t *cu,
                                     int32_t max_len, int32_t *cand_cu, int32_t *status, cudaStream_t stream) {
    if (n_q == 0) return cudaSuccess;
    candidate_offsets_kernel<<<n_q, kTopkThreads, 0, stream>>>(cand, n_cand, cu, max_len, cand_cu, status);
    return cudaGetLastError();
}

cudaError_t launch_gather_candidates(const int32_t *cand, int32_t n_q, int32_t n_cand, const int32_t *cu,
                                     const int32_t *cand_cu, const void *src, int64_t row_bytes, void *dst,
                                     int64_t slice_rows, int sm_count, cudaStream_t stream) {
    const int64_t items = static_cast<int64_t>(n_q) * n_cand;
    if (items == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((items * 32 + 255) / 256, static_cast<int64_t>(sm_count) * 8);
    gather_candidates_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(
        cand, n_q, n_cand, cu, cand_cu, static_cast<const uint8_t *>(src), row_bytes,
        static_cast<uint8_t *>(dst), slice_rows);
    return cudaGetLastError();
}

}  // namespace maxsim
