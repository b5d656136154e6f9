// bwd.cu -- training backward of the fused MaxSim operator.
//
// "FLASH-MAXSIM: IO-Aware Fused Kernels for Late-Interaction Retrieval"
// (arXiv 2605.29517) §4.2: with the forward winners t*(q, b, i) saved as
// the argmax, Eq. (2) is a gather and Eq. (3) a scatter; Alg. 3 inverts the
// argmax into a CSR map (bincount -> cumsum -> stable argsort) so that the
// scatter becomes a destination-owned, atomic-free reduction (§4.2.3).
//
// GB300 reading of Alg. 3 step 1: every source pointing into document b lies
// in argmax[:, b, :], so one CTA per document runs a stable counting sort of
// those sources in shared memory (per-warp histograms, a prefix over
// (token, warp) order, then in-order placement ranked with __match_any_sync).
// It produces exactly the global bincount/cumsum/stable-argsort CSR, with no
// global sort and no atomics outside a CTA's own shared memory.
#include "internal.cuh"
#include "sm103.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace maxsim {
namespace {

constexpr int kCsrWarps = 8;
constexpr int kCsrThreads = 32 * kCsrWarps;
constexpr int kCsrSmemBytes = 96 * 1024;   // per-warp histograms of one document

__device__ __forceinline__ bool valid_row(const BwdParams &p, int q, int i) {
    return i < p.q_lens[q];
}

// Sources per document (argmax entries of valid rows that name a token of
// the document).  An entry outside [-1, Ld_b) is reported and skipped.
__global__ void __launch_bounds__(256) csr_count_kernel(BwdParams p) {
    const int b = blockIdx.x;
    const int ld = p.cu_seqlens[b + 1] - p.cu_seqlens[b];
    const int n_cand = p.n_q * p.lq_max;
    int count = 0;
    for (int k = threadIdx.x; k < n_cand; k += blockDim.x) {
        const int q = k / p.lq_max;
        const int i = k - q * p.lq_max;
        if (!valid_row(p, q, i)) continue;
        const int a = p.argmax[(static_cast<int64_t>(q) * p.n_docs + b) * p.lq_max + i];
        if (a >= 0 && a < ld) ++count;
        else if (a < -1 || a >= ld) atomicCAS(p.status, 0, ptx::kStatusBadArgmax);
    }
    // fixed-shape block reduction (integer: order does not matter)
    __shared__ int red[256 / 32];
    for (int off = 16; off > 0; off >>= 1) count += __shfl_xor_sync(0xffffffffu, count, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = count;
    __syncthreads();
    if (threadIdx.x == 0) {
        int s = 0;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) s += red[w];
        p.doc_count[b] = s;
    }
}

// Exclusive prefix over documents (one CTA): doc_count[b] becomes the offset
// of document b's first source; doc_count[n_docs] and row_ptr[total] the
// number of sources.
__global__ void __launch_bounds__(1024) csr_doc_scan_kernel(BwdParams p) {
    __shared__ int warp_tot[32];
    __shared__ int carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int base = 0; base < p.n_docs; base += blockDim.x) {
        const int b = base + threadIdx.x;
        const int v = b < p.n_docs ? p.doc_count[b] : 0;
        int x = v;
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int t = lane < static_cast<int>(blockDim.x >> 5) ? warp_tot[lane] : 0;
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, t, off);
                if (lane >= off) t += y;
            }
            warp_tot[lane] = t;   // inclusive prefix of warp totals
        }
        __syncthreads();
        const int excl = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
        if (b < p.n_docs) p.doc_count[b] = excl;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = excl + v;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        p.doc_count[p.n_docs] = carry;
        p.row_ptr[p.total_tokens] = carry;
    }
}

// Stable per-document counting sort (Alg. 3 step 1 for the rows of one
// document).  Candidates are the n_q * lq_max argmax entries of the document
// in ascending flat order; warp w owns a contiguous segment of them.
__global__ void __launch_bounds__(kCsrThreads) csr_place_kernel(BwdParams p) {
    extern __shared__ int hist[];   // [W][ld]
    const int b = blockIdx.x;
    const int t0 = p.cu_seqlens[b];
    const int ld = p.cu_seqlens[b + 1] - t0;
    if (ld == 0) return;
    const int cap = kCsrSmemBytes / 4;
    int W = kCsrWarps;
    while (W > 1 && W * ld > cap) W >>= 1;
    if (W * ld > cap) {   // a single document longer than the shared histogram
        if (threadIdx.x == 0) atomicCAS(p.status, 0, ptx::kStatusDocTooLong);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_cand = p.n_q * p.lq_max;
    const int seg = ((n_cand + W - 1) / W + 31) / 32 * 32;
    for (int k = threadIdx.x; k < W * ld; k += blockDim.x) hist[k] = 0;
    __syncthreads();

    auto dest = [&](int k) -> int {   // token of candidate k, or -1
        if (k >= n_cand) return -1;
        const int q = k / p.lq_max;
        const int i = k - q * p.lq_max;
        if (!valid_row(p, q, i)) return -1;
        const int a = p.argmax[(static_cast<int64_t>(q) * p.n_docs + b) * p.lq_max + i];
        return (a >= 0 && a < ld) ? a : -1;
    };

    // 1. per-warp histograms
    if (warp < W) {
        for (int k = warp * seg + lane; k < min(n_cand, (warp + 1) * seg); k += 32) {
            const int a = dest(k);
            if (a >= 0) atomicAdd(&hist[warp * ld + a], 1);
        }
    }
    __syncthreads();

    // 2. row_ptr for the document's tokens, and each warp's first slot per
    //    token: offset + sum over earlier tokens + sum over earlier warps.
    //    Each thread owns a contiguous range of tokens.
    __shared__ int tot_scan[kCsrThreads];
    const int per = (ld + blockDim.x - 1) / blockDim.x;
    const int r0 = min(ld, threadIdx.x * per), r1 = min(ld, r0 + per);
    int local = 0;
    for (int t = r0; t < r1; ++t)
        for (int w = 0; w < W; ++w) local += hist[w * ld + t];
    tot_scan[threadIdx.x] = local;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int k = 0; k < static_cast<int>(blockDim.x); ++k) {
            const int v = tot_scan[k];
            tot_scan[k] = run;
            run += v;
        }
    }
    __syncthreads();
    int run = p.doc_count[b] + tot_scan[threadIdx.x];
    for (int t = r0; t < r1; ++t) {
        p.row_ptr[t0 + t] = run;
        for (int w = 0; w < W; ++w) {
            const int c = hist[w * ld + t];
            hist[w * ld + t] = run;
            run += c;
        }
    }
    __syncthreads();

    // 3. in-order placement, 32 candidates at a time per warp
    if (warp < W) {
        const int k_end = min(n_cand, (warp + 1) * seg);
        for (int kb = warp * seg; kb < k_end; kb += 32) {
            const int k = kb + lane;
            const int a = k < k_end ? dest(k) : -1;
            const int key = a >= 0 ? a : (0x40000000 | lane);   // invalid lanes never match
            const unsigned peers = __match_any_sync(0xffffffffu, key);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            int pos = 0;
            if (a >= 0) pos = hist[warp * ld + a] + rank;
            __syncwarp();
            if (a >= 0) {
                const int q = k / p.lq_max;
                const int i = k - q * p.lq_max;
                p.col_idx[pos] = (q * p.n_docs + b) * p.lq_max + i;
                if (rank == 0) hist[warp * ld + a] += __popc(peers);
            }
            __syncwarp();
        }
    }
}

__device__ __forceinline__ void load4(const void *base, int64_t row, int lane, bool bf16, float (&x)[4]) {
    const uint2 u = reinterpret_cast<const uint2 *>(static_cast<const uint8_t *>(base) + row * 256)[lane];
    if (bf16) {
        const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
        const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
        x[0] = __low2float(lo); x[1] = __high2float(lo);
        x[2] = __low2float(hi); x[3] = __high2float(hi);
    } else {
        const __half2 lo = *reinterpret_cast<const __half2 *>(&u.x);
        const __half2 hi = *reinterpret_cast<const __half2 *>(&u.y);
        x[0] = __low2float(lo); x[1] = __high2float(lo);
        x[2] = __low2float(hi); x[3] = __high2float(hi);
    }
}

// dD (Eq. (3), Alg. 3 step 2): one warp owns destination row r, walks its
// sources in CSR order accumulating g * Q_row in FP32, and writes the row
// once (rows with no source are written as 0).
__global__ void __launch_bounds__(256) grad_d_kernel(BwdParams p) {
    const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp_global >= p.total_tokens) return;
    const int r = warp_global;
    const int lo = p.row_ptr[r], hi = p.row_ptr[r + 1];
    const int per_q = p.n_docs * p.lq_max;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int base = lo; base < hi; base += 32) {
        const int n = min(32, hi - base);
        int s = 0;
        float gs = 0.f;
        int qrow = 0;
        if (lane < n) {
            s = p.col_idx[base + lane];
            const int q = s / per_q;
            const int rem = s - q * per_q;
            const int bb = rem / p.lq_max;
            const int i = rem - bb * p.lq_max;
            gs = p.grad[static_cast<int64_t>(q) * p.n_docs + bb];
            qrow = q * p.lq_max + i;
        }
        for (int j = 0; j < n; ++j) {
            const float g = __shfl_sync(0xffffffffu, gs, j);
            const int row = __shfl_sync(0xffffffffu, qrow, j);
            float x[4];
            load4(p.Q, row, lane, p.bf16, x);
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[c] = fmaf(g, x[c], acc[c]);
        }
    }
    reinterpret_cast<float4 *>(p.dD + static_cast<int64_t>(r) * 128)[lane] =
        make_float4(acc[0], acc[1], acc[2], acc[3]);
}

// dQ (Eq. (2), Alg. 3 step 3): one warp owns query row (q, i) and gathers
// g[q, b] * D[cu[b] + t*] over documents b in ascending order.
__global__ void __launch_bounds__(256) grad_q_kernel(BwdParams p) {
    const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp_global >= static_cast<int64_t>(p.n_q) * p.lq_max) return;
    const int q = static_cast<int>(warp_global / p.lq_max);
    const int i = static_cast<int>(warp_global - static_cast<int64_t>(q) * p.lq_max);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (i < p.q_lens[q]) {
        for (int b0 = 0; b0 < p.n_docs; b0 += 32) {
            const int n = min(32, p.n_docs - b0);
            int trow = -1;
            float gs = 0.f;
            if (lane < n) {
                const int b = b0 + lane;
                const int t = p.argmax[(static_cast<int64_t>(q) * p.n_docs + b) * p.lq_max + i];
                const int lo = p.cu_seqlens[b];
                const int ld = p.cu_seqlens[b + 1] - lo;
                if (t >= 0 && t < ld) {
                    trow = lo + t;
                    gs = p.grad[static_cast<int64_t>(q) * p.n_docs + b];
                }
            }
            for (int j = 0; j < n; ++j) {
                const int row = __shfl_sync(0xffffffffu, trow, j);
                const float g = __shfl_sync(0xffffffffu, gs, j);
                if (row < 0) continue;
                float x[4];
                load4(p.D, row, lane, p.bf16, x);
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[c] = fmaf(g, x[c], acc[c]);
            }
        }
    }
    reinterpret_cast<float4 *>(p.dQ + warp_global * 128)[lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
}

}  // namespace

cudaError_t launch_build_csr(const BwdParams &p, cudaStream_t stream) {
    if (p.n_docs == 0) {
        return cudaMemsetAsync(p.row_ptr, 0, sizeof(int32_t) * (p.total_tokens + 1), stream);
    }
    csr_count_kernel<<<p.n_docs, 256, 0, stream>>>(p);
    csr_doc_scan_kernel<<<1, 1024, 0, stream>>>(p);
    cudaError_t e = cudaFuncSetAttribute(csr_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kCsrSmemBytes);
    if (e != cudaSuccess) return e;
    csr_place_kernel<<<p.n_docs, kCsrThreads, kCsrSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_grad_d(const BwdParams &p, cudaStream_t stream) {
    if (p.total_tokens == 0) return cudaSuccess;
    const int64_t threads = static_cast<int64_t>(p.total_tokens) * 32;
    grad_d_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_grad_q(const BwdParams &p, cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(p.n_q) * p.lq_max;
    if (rows == 0) return cudaSuccess;
    grad_q_kernel<<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace maxsim
