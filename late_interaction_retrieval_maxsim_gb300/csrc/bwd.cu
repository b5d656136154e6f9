// bwd.cu -- training backward of the fused MaxSim operator.
//
// "FLASH-MAXSIM: IO-Aware Fused Kernels for Late-Interaction Retrieval"
// (arXiv 2605.29517) §4.2: with the forward winners t*(q, b, i) saved as
// the argmax, Eq. (2) is a gather and Eq. (3) a scatter; Alg. 3 inverts the
// argmax into a CSR map (bincount -> cumsum -> stable argsort) so that the
// scatter becomes a destination-owned, atomic-free reduction (§4.2.3).
//
// GB300 reading of Alg. 3 step 1: every source pointing into document b lies
// in argmax[:, b, :], so the sources are sorted document by document with a
// stable counting sort.  A document's candidates (its n_q * lq_max argmax
// entries in ascending flat order) are split into C contiguous chunks, one
// CTA each: chunk histograms, a scan over documents, a per-document scan over
// (token, chunk), then in-order placement inside each chunk (per-warp
// histograms, a prefix over (token, warp) order, ranks from
// __match_any_sync).  It produces exactly the global bincount / cumsum /
// stable-argsort CSR, with no global sort; the only global atomics add
// integer counts.
#include "internal.cuh"
#include "sm103.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace maxsim {
namespace {

constexpr int kCsrWarps = 8;
constexpr int kCsrThreads = 32 * kCsrWarps;
constexpr int kCsrSmemBytes = 96 * 1024;   // per-warp histograms of one document chunk
static_assert(kCsrSmemBytes / 4 == kCsrMaxDocTokens, "the forward's counts and the CSR agree on long documents");
// Documents of at most kCsrSmallDoc tokens (every workload here) run in a
// first launch with small shared-memory footprints, so many CTAs share an SM;
// longer ones run in a second launch with the full 96 KB.
constexpr int kCsrSmallDoc = 4096;
constexpr int kCsrSmallHistBytes = kCsrSmallDoc * 4;
constexpr int kCsrSmallPlaceBytes = 24 * 1024;

__device__ __forceinline__ bool valid_row(const BwdParams &p, int q, int i) {
    return i < p.q_lens[q];
}

__device__ __forceinline__ int chunk_len(int n_cand, int chunks) { return (n_cand + chunks - 1) / chunks; }

// k / lq_max for a flat candidate index k (< 2^31), by multiply-high.
__device__ __forceinline__ int query_of(const BwdParams &p, int k) {
    return static_cast<int>((static_cast<uint64_t>(static_cast<uint32_t>(k)) * p.lq_magic) >> (31 + p.lq_shift));
}

// Token counts of one chunk of a document's candidates (argmax entries of
// valid rows that name a token of the document), written to
// chunk_cnt[chunks * cu[b] + c * ld + t]; the chunk's total is added to
// doc_count[b] (an integer sum: the order of the additions does not matter).
// An entry outside [-1, Ld_b) is reported and skipped.
__global__ void __launch_bounds__(256) csr_chunk_hist_kernel(BwdParams p, bool large) {
    extern __shared__ int cnt[];   // [ld]
    const int b = blockIdx.x / p.chunks, c = blockIdx.x % p.chunks;
    const int t0 = p.cu_seqlens[b];
    const int ld = p.cu_seqlens[b + 1] - t0;
    if ((ld > kCsrSmallDoc) != large) return;   // the other launch's document
    if (ld > kCsrSmemBytes / 4) {
        if (threadIdx.x == 0 && c == 0) atomicCAS(p.status, 0, ptx::kStatusDocTooLong);
        return;
    }
    const int n_cand = p.n_q * p.lq_max;
    const int k0 = c * chunk_len(n_cand, p.chunks);
    const int k1 = min(n_cand, k0 + chunk_len(n_cand, p.chunks));
    for (int t = threadIdx.x; t < ld; t += blockDim.x) cnt[t] = 0;
    __syncthreads();
    int total = 0;
    // four independent loads in flight per thread before their counts
    for (int kb = k0 + threadIdx.x; kb < k1; kb += 4 * blockDim.x) {
        int a[4];
        bool v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = kb + u * blockDim.x;
            const int q = query_of(p, k);
            const int i = k - q * p.lq_max;
            v[u] = k < k1 && valid_row(p, q, i);
            a[u] = v[u] ? p.argmax[(static_cast<int64_t>(q) * p.n_docs + b) * p.lq_max + i] : -1;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (!v[u]) continue;
            if (a[u] >= 0 && a[u] < ld) {
                atomicAdd(&cnt[a[u]], 1);
                ++total;
            } else if (a[u] < -1 || a[u] >= ld) {
                atomicCAS(p.status, 0, ptx::kStatusBadArgmax);
            }
        }
    }
    __shared__ int red[256 / 32];
    for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = total;
    __syncthreads();
    int32_t *out = p.chunk_cnt + static_cast<int64_t>(p.chunks) * t0 + static_cast<int64_t>(c) * ld;
    for (int t = threadIdx.x; t < ld; t += blockDim.x) out[t] = cnt[t];
    if (threadIdx.x == 0) {
        int sum = 0;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) sum += red[w];
        if (sum) atomicAdd(&p.doc_count[b], sum);
    }
}

// Per document (one CTA), when the forward left the token counts:
// doc_count[b] = the sum of the document's chunks * ld counts (a contiguous
// range of chunk_cnt), in a fixed order.
__global__ void __launch_bounds__(256) csr_doc_total_kernel(BwdParams p) {
    const int b = blockIdx.x;
    const int64_t lo = static_cast<int64_t>(p.chunks) * p.cu_seqlens[b];
    const int64_t hi = static_cast<int64_t>(p.chunks) * p.cu_seqlens[b + 1];
    int sum = 0;
    for (int64_t k = lo + threadIdx.x; k < hi; k += blockDim.x) sum += p.chunk_cnt[k];
    __shared__ int red[256 / 32];
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        int s = 0;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) s += red[w];
        p.doc_count[b] = s;
    }
}

// Per document (one CTA): row_ptr of its tokens, and chunk_cnt[c][t] turned
// into the first CSR slot of chunk c's sources for token t
// (row_ptr[t] + the counts of the earlier chunks for t).
__global__ void __launch_bounds__(256) csr_token_scan_kernel(BwdParams p) {
    const int b = blockIdx.x;
    const int t0 = p.cu_seqlens[b];
    const int ld = p.cu_seqlens[b + 1] - t0;
    if (ld > kCsrSmemBytes / 4) {
        // too long for the shared histograms (reported by the other kernels):
        // its sources are left out, so every row is empty
        for (int t = threadIdx.x; t < ld; t += blockDim.x) p.row_ptr[t0 + t] = p.doc_count[b];
        return;
    }
    if (ld == 0) return;
    int32_t *cc = p.chunk_cnt + static_cast<int64_t>(p.chunks) * t0;
    __shared__ int tot_scan[256];
    const int per = (ld + blockDim.x - 1) / blockDim.x;
    const int r0 = min(ld, static_cast<int>(threadIdx.x) * per), r1 = min(ld, r0 + per);
    int local = 0;
    for (int t = r0; t < r1; ++t)
        for (int c = 0; c < p.chunks; ++c) local += cc[c * ld + t];
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
        for (int c = 0; c < p.chunks; ++c) {
            const int v = cc[c * ld + t];
            cc[c * ld + t] = run;
            run += v;
        }
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

// Stable placement of one chunk of a document's candidates (Alg. 3 step 1):
// warp w owns a contiguous segment of the chunk; a source's slot is its
// chunk's first slot for its token + the counts of earlier warps for that
// token + its rank among equal tokens earlier in its warp.
__global__ void __launch_bounds__(kCsrThreads) csr_place_kernel(BwdParams p, bool large) {
    extern __shared__ int hist[];   // [W][ld]
    const int b = blockIdx.x / p.chunks, chunk = blockIdx.x % p.chunks;
    const int t0 = p.cu_seqlens[b];
    const int ld = p.cu_seqlens[b + 1] - t0;
    if (ld == 0 || (ld > kCsrSmallDoc) != large) return;
    const int cap = (large ? kCsrSmemBytes : kCsrSmallPlaceBytes) / 4;
    int W = kCsrWarps;
    while (W > 1 && W * ld > cap) W >>= 1;
    if (W * ld > cap) {   // a single document longer than the shared histogram
        if (threadIdx.x == 0) atomicCAS(p.status, 0, ptx::kStatusDocTooLong);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_all = p.n_q * p.lq_max;
    const int k_lo = chunk * chunk_len(n_all, p.chunks);
    const int n_cand = min(n_all, k_lo + chunk_len(n_all, p.chunks));   // end of this chunk
    const int seg = ((n_cand - k_lo + W - 1) / W + 31) / 32 * 32;
    for (int k = threadIdx.x; k < W * ld; k += blockDim.x) hist[k] = 0;
    __syncthreads();

    auto dest = [&](int k) -> int {   // token of candidate k, or -1
        if (k >= n_cand) return -1;
        const int q = query_of(p, k);
        const int i = k - q * p.lq_max;
        if (!valid_row(p, q, i)) return -1;
        const int a = p.argmax[(static_cast<int64_t>(q) * p.n_docs + b) * p.lq_max + i];
        return (a >= 0 && a < ld) ? a : -1;
    };

    // 1. per-warp histograms (four independent loads in flight per lane)
    if (warp < W) {
        const int k_end = min(n_cand, k_lo + (warp + 1) * seg);
        for (int kb = k_lo + warp * seg + lane; kb < k_end; kb += 128) {
            int a[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) a[u] = kb + 32 * u < k_end ? dest(kb + 32 * u) : -1;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (a[u] >= 0) atomicAdd(&hist[warp * ld + a[u]], 1);
        }
    }
    __syncthreads();

    // 2. each warp's first slot per token: the chunk's first slot for the
    //    token + the counts of earlier warps
    const int32_t *first = p.chunk_cnt + static_cast<int64_t>(p.chunks) * t0 + static_cast<int64_t>(chunk) * ld;
    for (int t = threadIdx.x; t < ld; t += blockDim.x) {
        int run = first[t];
        for (int w = 0; w < W; ++w) {
            const int c = hist[w * ld + t];
            hist[w * ld + t] = run;
            run += c;
        }
    }
    __syncthreads();

    // 3. in-order placement, 32 candidates at a time per warp
    if (warp < W) {
        const int k_end = min(n_cand, k_lo + (warp + 1) * seg);
        int a_next = k_lo + warp * seg + lane < k_end ? dest(k_lo + warp * seg + lane) : -1;
        for (int kb = k_lo + warp * seg; kb < k_end; kb += 32) {
            const int k = kb + lane;
            const int a = a_next;   // the next 32 candidates load while these are placed
            a_next = k + 32 < k_end ? dest(k + 32) : -1;
            const int key = a >= 0 ? a : (0x40000000 | lane);   // invalid lanes never match
            const unsigned peers = __match_any_sync(0xffffffffu, key);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            int pos = 0;
            if (a >= 0) pos = hist[warp * ld + a] + rank;
            __syncwarp();
            if (a >= 0) {
                const int q = query_of(p, k);
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

int csr_chunks(int32_t n_q, int32_t lq_max, int32_t n_docs) {
    // enough CTAs to fill the GPU (about 300), at most 16 chunks per document,
    // at least 2,048 candidates per chunk; a function of the shape only, so
    // workspace sizes need no device
    const int64_t n_cand = static_cast<int64_t>(n_q) * lq_max;
    if (n_docs <= 0 || n_cand <= 0) return 1;
    int64_t c = (300 + n_docs - 1) / n_docs;
    c = c < 16 ? c : 16;
    const int64_t by_size = n_cand / 2048;
    c = c < by_size ? c : by_size;
    return static_cast<int>(c < 1 ? 1 : c);
}

cudaError_t launch_build_csr(const BwdParams &p, cudaStream_t stream, bool counts_ready) {
    if (p.n_docs == 0) {
        return cudaMemsetAsync(p.row_ptr, 0, sizeof(int32_t) * (p.total_tokens + 1), stream);
    }
    cudaError_t e = cudaSuccess;
    const unsigned grid = static_cast<unsigned>(p.n_docs) * p.chunks;
    // a document longer than kCsrSmallDoc needs a second, large-footprint launch
    const bool any_large = p.total_tokens > kCsrSmallDoc;
    if (!counts_ready) {
        if ((e = cudaMemsetAsync(p.doc_count, 0, sizeof(int32_t) * (p.n_docs + 1), stream)) != cudaSuccess)
            return e;
        if ((e = cudaFuncSetAttribute(csr_chunk_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kCsrSmemBytes)) != cudaSuccess)
            return e;
        csr_chunk_hist_kernel<<<grid, 256, kCsrSmallHistBytes, stream>>>(p, false);
        if (any_large) csr_chunk_hist_kernel<<<grid, 256, kCsrSmemBytes, stream>>>(p, true);
    }
    // (with counts from the forward, documents too long for the CSR are
    // reported by csr_place_kernel)
    if (counts_ready) csr_doc_total_kernel<<<p.n_docs, 256, 0, stream>>>(p);
    csr_doc_scan_kernel<<<1, 1024, 0, stream>>>(p);
    csr_token_scan_kernel<<<p.n_docs, 256, 0, stream>>>(p);
    if ((e = cudaFuncSetAttribute(csr_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kCsrSmemBytes)) != cudaSuccess)
        return e;
    csr_place_kernel<<<grid, kCsrThreads, kCsrSmallPlaceBytes, stream>>>(p, false);
    if (any_large) csr_place_kernel<<<grid, kCsrThreads, kCsrSmemBytes, stream>>>(p, true);
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
