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
// stable counting sort.  Two forms:
//  * maxsim_build_csr (the exact CSR as its own entry point): a document's
//    candidates (its n_q * lq_max argmax entries in ascending flat order)
//    are split into C contiguous chunks, one CTA each: chunk histograms, a
//    scan over documents, a per-document scan over (token, chunk), then
//    in-order placement inside each chunk (per-warp histograms, a prefix
//    over (token, warp) order, ranks from __match_any_sync).  It produces
//    exactly the global bincount / cumsum / stable-argsort CSR, with no
//    global sort; the only global atomics add integer counts.
//  * maxsim_backward: one kernel sorts each (document, chunk) into fixed
//    slots with per-(chunk, token) run bounds, needing no prefix over
//    documents (bwd_sort_kernel); dD reads a row's runs chunk after chunk,
//    which is its CSR row (grad_d_kernel); dQ gathers straight from the
//    argmax (grad_q_kernel), on a second stream.
#include "internal.cuh"
#include "sm103.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

namespace maxsim {
namespace {

constexpr int kCsrWarps = 8;
constexpr int kCsrThreads = 32 * kCsrWarps;
constexpr int kCsrSmemBytes = 96 * 1024;   // per-warp histograms of one document chunk
static_assert(kCsrSmemBytes / 4 == kCsrMaxDocTokens, "the shared histograms hold the longest document");
// Documents of at most kCsrSmallDoc tokens (every workload here) run in a
// first launch with small shared-memory footprints, so many CTAs share an SM;
// longer ones run in a second launch with the full 96 KB.
constexpr int kCsrSmallDoc = 4096;
constexpr int kCsrSmallHistBytes = kCsrSmallDoc * 4;
constexpr int kCsrSmallPlaceBytes = 32 * 1024;   // eight warps' histograms of a 1024-token document

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

// ---------------------------------------------------------------- gathers
//
// Both gradients are sums of weighted 256-byte rows (128 FP16/BF16 values)
// gathered from an L2-resident Q or D: dD row r = sum over its sources of
// g * Q_row, dQ row (q, i) = sum over documents of g * D_row.  One warp owns
// one output row; each half-warp gathers every other row of the list (half h
// the positions j = h mod 2), each lane 16 bytes (8 values) of it, so one
// warp instruction moves two rows, and the FMAs are packed two per
// instruction: about 8 instructions per gathered row (ncu showed the
// one-row-per-step form issuing 29 and the schedulers, not L2, setting the
// pace).  Each lane keeps four 16-byte loads in flight: the gathers are
// bound by L2 latency, not its bandwidth (ncu: L2 throughput 35-38 %, long
// scoreboard the top stall with two in flight; four took the training-shape
// backward from 145 to 129 us, eight were slower).  At the end the half sums
// are added (half 0 + half 1).  The order is fixed by the list, so the bits
// are the same on every run.

__device__ __forceinline__ uint4 load_row16(const void *base, int64_t row, int c) {
    return __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(base) + row * 256) + c);
}

// acc[k] += w * (values 2k, 2k+1 of the 8 in u), FP16 or BF16.
__device__ __forceinline__ void fma8(uint4 u, float w, bool bf16, float2 (&acc)[4]) {
    const float2 ww = make_float2(w, w);
    const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float2 x;
        if (bf16) {   // a bfloat16 is the upper half of a binary32
            x.x = __uint_as_float(v[k] << 16);
            x.y = __uint_as_float(v[k] & 0xffff0000u);
        } else {
            x = __half22float2(*reinterpret_cast<const __half2 *>(&v[k]));
        }
        acc[k] = ptx::fma2(ww, x, acc[k]);
    }
}

// acc (this lane's 8 columns, 8 * (lane & 15) ..) += the sum, over the list
// positions j = h (mod 2) of this lane's half-warp h in ascending order, of
// w_j * X[row_j, :]; every lane l evaluates entry(base + l, base + l < n,
// row, w) for each batch of 32 (the whole warp, so the entry may shuffle;
// row < 0: no contribution), the next batch's entries while the current
// batch's rows are gathered.  Whole warp, same n.
template <typename Entry>
__device__ __forceinline__ void warp_gather(const void *X, bool bf16, int n, Entry entry, float2 (&acc)[4]) {
    const int lane = threadIdx.x & 31, h = lane >> 4, c = lane & 15;
    if (n <= 0) return;
    int rv = -1;
    float wv = 0.f;
    entry(lane, lane < n, rv, wv);
    if (lane >= n) rv = -1;
    for (int base = 0; base < n; base += 32) {
        int nrv = -1;
        float nwv = 0.f;
        if (base + 32 < n) {
            entry(base + 32 + lane, base + 32 + lane < n, nrv, nwv);
            if (base + 32 + lane >= n) nrv = -1;
        }
        const int cnt = min(32, n - base);
        for (int jb = 0; jb < cnt; jb += 8) {
            int row[4];
            float w[4];
            uint4 raw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = jb + 2 * u + h;   // <= 31
                row[u] = __shfl_sync(0xffffffffu, rv, j);
                w[u] = __shfl_sync(0xffffffffu, wv, j);
                if (j >= cnt) row[u] = -1;
                raw[u] = row[u] >= 0 ? load_row16(X, row[u], c) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (row[u] >= 0) fma8(raw[u], w[u], bf16, acc);
        }
        rv = nrv;
        wv = nwv;
    }
}

// Adds the two half-warp sums (half 0 + half 1) and writes the 128-float row.
__device__ __forceinline__ void warp_store_row(float *out_row, float2 (&acc)[4]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float ox = __shfl_xor_sync(0xffffffffu, acc[k].x, 16);
        const float oy = __shfl_xor_sync(0xffffffffu, acc[k].y, 16);
        acc[k] = (lane < 16) ? make_float2(acc[k].x + ox, acc[k].y + oy) : make_float2(ox + acc[k].x, oy + acc[k].y);
    }
    if (lane < 16) {
        float4 *o = reinterpret_cast<float4 *>(out_row) + 2 * lane;
        o[0] = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
        o[1] = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
    }
}

// The backward's own inverse map (the per-document reading of Alg. 3 step
// 1: every source of document b lies in argmax[:, b, :]).  A document's
// n_cand = n_q * lq_max candidates (flat order k = q * lq_max + i) are cut
// into C <= 32 chunks; one CTA per (document, chunk) keeps its chunk's
// tokens in shared memory and sorts the chunk's sources by token with a
// stable counting sort (per-warp histograms, a prefix over (token, warp),
// ranks within a warp from lane masks), WIN tokens at a time.  It writes the
// sorted candidates k (the source's Q row) to the fixed slots
// [b * n_cand + k0, b * n_cand + k1) of col_idx, each source's g[q, b] to the
// same slot of col_w, and for every token r of the document the bounds of
// its run there to row_start / row_end at run_bound_index(r, c, C).  No
// prefix over documents is needed, and token r's runs read chunk after chunk
// give its sources in ascending order: the CSR's row.  (Measured
// alternatives: a two-pass LSD radix sort on 5-bit digits was slower, 38.5
// vs 23.5 us on the training shape.)
constexpr int kSortQueries = 256;   // queries of a chunk whose q_lens and g are staged

// Per-warp histograms are stored with one pad word after every 32 tokens, so
// the scan's threads (each reading PER consecutive tokens) hit distinct banks.
// (Two tokens per word as 16-bit halves, which halves this array, measured
// 264 -> 260 us for the ColPali-shape backward but 145 -> 149 us for the
// training shape, and is not used.)
template <int WIN>
struct SortHist {
    static constexpr int kStride = WIN + WIN / 32;   // words per warp
    __device__ static __forceinline__ int at(int t) { return t + (t >> 5); }
};

// The lanes of the warp whose (key, valid) equals this lane's, for keys below
// 2^BITS: one ballot per key bit and one for validity (what
// __match_any_sync returns; measured far cheaper than that instruction on 32
// mostly distinct keys: the training-shape sort 29 -> 23.5 us).
template <int BITS>
__device__ __forceinline__ unsigned match_lanes(int key, bool valid) {
    unsigned eq = __ballot_sync(0xffffffffu, valid);
    if (!valid) eq = ~eq;
#pragma unroll
    for (int bit = 0; bit < BITS; ++bit) {
        const bool on = (key >> bit) & 1;
        const unsigned m = __ballot_sync(0xffffffffu, on);
        eq &= on ? m : ~m;
    }
    return eq;
}

// WIN tokens per window: 256 for documents of a few hundred tokens, 1024 for
// page-length ones (each window rescans the chunk's tokens in shared memory);
// W warps, each owning a contiguous segment of the chunk.  Short documents
// use 16 warps; the 1024-token histograms leave room for 8.
template <int WIN, int W>
size_t sort_smem_bytes(int chunk_len) {
    // tokens, per-warp histograms, run starts, and the window's sorted
    // candidates staged for coalesced writes (their weights are looked up as
    // they are written: staging them too cost the 256-token form a CTA per SM)
    return static_cast<size_t>(chunk_len) * 4 * 2 + W * SortHist<WIN>::kStride * 4 + (WIN + 1) * 4 + 16;
}

template <int WIN, int W>
__global__ void __launch_bounds__(32 * W) bwd_sort_kernel(BwdParams p) {
    constexpr int T = 32 * W;
    constexpr int PER = WIN >= T ? WIN / T : 1;   // tokens per thread in the scan
    constexpr int KB = WIN == 256 ? 8 : 10;       // token bits
    static_assert((1 << KB) == WIN, "window tokens fit the key bits");
    using H = SortHist<WIN>;
    constexpr int HS = H::kStride;
    // Ranks within a warp: at 256-token windows from per-warp lane masks in
    // shared memory (each lane ORs its bit into its token's word, reads the
    // word back, and the lowest lane clears it: order-free, so the same
    // result on every run; training-shape backward 129 -> 127 us), at
    // 1024-token windows (where the masks would cost 32 KB and a CTA per SM)
    // from ballots.
    constexpr bool kMaskRank = WIN == 256;
    extern __shared__ __align__(16) uint8_t ssm[];
    int32_t *tok = reinterpret_cast<int32_t *>(ssm);                 // [chunk_len]
    int32_t *hist = tok + p.sort_chunk_len;                          // [W][HS], token t at H::at(t)
    int32_t *start = hist + W * HS;                                  // [WIN + 1]
    int32_t *out_k = start + WIN + 1;                                // [chunk_len] the window's sorted sources
    __shared__ int32_t warp_tot[W];
    __shared__ uint32_t s_mask[kMaskRank ? W * WIN : 1];
    __shared__ int32_t s_ql[kSortQueries];
    __shared__ float s_g[kSortQueries];
    const int C = p.sort_chunks;
    const int b = blockIdx.x / C, c = blockIdx.x - b * C;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = p.cu_seqlens[b];
    const int ld = p.cu_seqlens[b + 1] - t0;
    if (ld <= 0) return;
    const int n_cand = p.n_q * p.lq_max;
    const int k0 = min(n_cand, c * p.sort_chunk_len);
    const int len = min(n_cand, k0 + p.sort_chunk_len) - k0;

    // q_lens and g[., b] of the chunk's queries, when they are few enough
    const int q_lo = len > 0 ? query_of(p, k0) : 0;
    const int n_qr = len > 0 ? query_of(p, k0 + len - 1) - q_lo + 1 : 0;
    const bool staged = n_qr <= kSortQueries;
    if (staged)
        for (int qq = threadIdx.x; qq < n_qr; qq += T) {
            s_ql[qq] = p.q_lens[q_lo + qq];
            s_g[qq] = p.grad[static_cast<int64_t>(q_lo + qq) * p.n_docs + b];
        }
    for (int k = threadIdx.x; k < W * HS; k += T) hist[k] = 0;
    if constexpr (kMaskRank)
        for (int k = threadIdx.x; k < W * WIN; k += T) s_mask[k] = 0u;
    __syncthreads();
    auto qlen_of = [&](int q) { return staged ? s_ql[q - q_lo] : p.q_lens[q]; };
    auto g_of = [&](int q) { return staged ? s_g[q - q_lo] : p.grad[static_cast<int64_t>(q) * p.n_docs + b]; };

    const int seg = ((len + W - 1) / W + 31) / 32 * 32;
    const int s_lo = min(len, warp * seg), s_hi = min(len, s_lo + seg);
    // 1. the warp's segment: the token each candidate names, or -1, counted at
    //    once for the first window.  With lq_max and k0 multiples of 4 and a
    //    16-byte aligned argmax, a lane loads four consecutive candidates (one
    //    query row, 16 bytes) at once; otherwise four loads at stride 32.
    auto record = [&](int kk, int v) {
        if (v < -1 || v >= ld) {
            atomicCAS(p.status, 0, ptx::kStatusBadArgmax);
            v = -1;
        }
        tok[kk] = v;
        if (v >= 0 && v < WIN) atomicAdd(&hist[warp * HS + H::at(v)], 1);
    };
    const bool vec = (p.lq_max & 3) == 0 && (k0 & 3) == 0 && (reinterpret_cast<uintptr_t>(p.argmax) & 15) == 0;
    if (vec)
        for (int kb = s_lo + 4 * lane; kb < s_hi; kb += 4 * 32) {
            const int k = k0 + kb;
            const int q = query_of(p, k);
            const int i = k - q * p.lq_max;
            const int32_t *src = p.argmax + (static_cast<int64_t>(q) * p.n_docs + b) * p.lq_max + i;
            int4 a4 = make_int4(-1, -1, -1, -1);
            if (kb + 3 < s_hi) {
                a4 = *reinterpret_cast<const int4 *>(src);
            } else {
                a4.x = src[0];
                if (kb + 1 < s_hi) a4.y = src[1];
                if (kb + 2 < s_hi) a4.z = src[2];
            }
            const int ql = qlen_of(q);
            const int av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (kb + u < s_hi) record(kb + u, i + u < ql ? av[u] : -1);
        }
    else
    for (int kb = s_lo + lane; kb < s_hi; kb += 4 * 32) {
        int a[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int kk = kb + 32 * u;
            a[u] = -1;
            if (kk < s_hi) {
                const int k = k0 + kk;
                const int q = query_of(p, k);
                const int i = k - q * p.lq_max;
                if (i < qlen_of(q)) a[u] = p.argmax[(static_cast<int64_t>(q) * p.n_docs + b) * p.lq_max + i];
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int kk = kb + 32 * u;
            if (kk < s_hi) record(kk, a[u]);
        }
    }
    int32_t win_base = b * n_cand + k0;   // first slot of the current window's sources (< 2^31)

    for (int w0 = 0; w0 < ld; w0 += WIN) {
        const int win = min(WIN, ld - w0);
        if (w0 > 0) {
            for (int k = threadIdx.x; k < W * HS; k += T) hist[k] = 0;
            __syncthreads();
            // 2. per-warp histograms of the window's tokens
            for (int kk = s_lo + lane; kk < s_hi; kk += 32) {
                const int t = tok[kk] - w0;
                if (t >= 0 && t < win) atomicAdd(&hist[warp * HS + H::at(t)], 1);
            }
        }
        __syncthreads();
        // 3. token totals -> exclusive scan -> each warp's first slot per
        //    token (thread t holds tokens PER * t .. PER * t + PER - 1)
        const int t = threadIdx.x;
        int tot = 0;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const int tk = PER * t + e;
            if (tk < WIN)
#pragma unroll
                for (int w = 0; w < W; ++w) tot += hist[w * HS + H::at(tk)];
        }
        int x = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        int run = x - tot;
        for (int w = 0; w < warp; ++w) run += warp_tot[w];
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const int tk = PER * t + e;
            if (tk >= WIN) break;
            start[tk] = run;
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const int v = hist[w * HS + H::at(tk)];
                hist[w * HS + H::at(tk)] = run;
                run += v;
            }
        }
        if (t == T - 1) start[WIN] = run;   // the last thread's tokens end the window
        __syncthreads();
        for (int tk = t; tk < win; tk += T) {
            const int64_t at = run_bound_index(t0 + w0 + tk, c, C);
            p.row_start[at] = win_base + start[tk];
            p.row_end[at] = win_base + start[tk + 1];
        }
        // 4. stable placement, 32 candidates at a time per warp
        for (int kb = s_lo; kb < s_hi; kb += 32) {
            const int kk = kb + lane;
            const int tt = kk < s_hi ? tok[kk] - w0 : -1;
            const bool mine = tt >= 0 && tt < win;
            unsigned peers;
            if constexpr (kMaskRank) {
                if (mine) atomicOr(&s_mask[warp * WIN + tt], 1u << lane);
                __syncwarp();
                peers = mine ? s_mask[warp * WIN + tt] : 0u;
            } else {
                peers = match_lanes<KB>(mine ? tt : 0, mine);
            }
            const int rank = __popc(peers & ((1u << lane) - 1u));
            int pos = 0;
            if (mine) pos = hist[warp * HS + H::at(tt)] + rank;
            __syncwarp();
            if (mine) {
                out_k[pos] = k0 + kk;
                if (rank == 0) {
                    hist[warp * HS + H::at(tt)] += __popc(peers);
                    if constexpr (kMaskRank) s_mask[warp * WIN + tt] = 0u;
                }
            }
            __syncwarp();
        }
        __syncthreads();
        // 5. the window's sorted sources to their slots, coalesced
        const int n_win = start[WIN];
        for (int e = threadIdx.x; e < n_win; e += T) {
            const int k = out_k[e];
            p.col_idx[win_base + e] = k;
            p.col_w[win_base + e] = g_of(query_of(p, k));
        }
        win_base += n_win;
        __syncthreads();
    }
}

// The gathers of one output row start at a position derived from the row's
// index and wrap around (a fixed order): rows that run at the same time then
// read different parts of Q / D instead of all starting at the same
// documents or queries and contending for the same L2 lines.
__device__ __forceinline__ int rotation(int64_t row, int n) {
    return n > 0 ? static_cast<int>((static_cast<uint64_t>(row) * 0x9E3779B1ull >> 7) % static_cast<uint64_t>(n)) : 0;
}

// dD (Eq. (3), Alg. 3 step 2): one warp owns destination row r and sums
// g[q, b] * Q[q, i, :] over its sources, writing the row once (rows with no
// source are 0).  Its sources are its runs read chunk after chunk
// (ascending source order, the CSR's row) as one list of n entries: lane c <
// C holds run c's bounds, and a position maps to its run by a prefix over the
// run lengths.  The sum visits the list from position rotation(r, n),
// wrapping around.  A CTA's kRunBlock rows share the sectors that hold
// their bounds (run_bound_index), so its warps read them through L1.
__global__ void __launch_bounds__(32 * kRunBlock) grad_d_kernel(BwdParams p) {
    const int C = p.sort_chunks;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kRunBlock;
    const int64_t base = r0 * C;   // run_bound_index(r0, 0, C)
    const int r = static_cast<int>(r0) + (threadIdx.x >> 5);
    if (r >= p.total_tokens) return;
    const int lane = threadIdx.x & 31;
    const int wr = threadIdx.x >> 5;   // this warp's row within the block
    int lo = 0, len = 0;
    if (lane < C) {
        lo = __ldg(p.row_start + base + lane * kRunBlock + wr);
        len = __ldg(p.row_end + base + lane * kRunBlock + wr) - lo;
    }
    int incl = len;   // inclusive prefix of the run lengths over lanes
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const int n = __shfl_sync(0xffffffffu, incl, 31);
    const int excl = incl - len;
    const int first = rotation(r, n);
    // the binary search's first step: the largest power of two below C
    const int top = C > 1 ? 1 << (31 - __clz(C - 1)) : 0;
    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    warp_gather(p.Q, p.bf16 != 0, n,
                [&](int j, bool valid, int &row, float &w) {
                    int pos = j + first;   // the list position visited j-th
                    if (pos >= n) pos -= n;
                    // the run holding pos: the number of runs whose end is <= pos,
                    // found by a binary search over the C lanes' inclusive ends
                    int run = 0;
#pragma unroll
                    for (int step = 16; step > 0; step >>= 1)
                        if (step <= top)   // uniform
                            if (__shfl_sync(0xffffffffu, incl, run + step - 1) <= pos) run += step;
                    run = min(run, C - 1);
                    const int at = __shfl_sync(0xffffffffu, lo, run) + pos - __shfl_sync(0xffffffffu, excl, run);
                    if (!valid) return;
                    row = p.col_idx[at];
                    w = p.col_w[at];
                },
                acc);
    warp_store_row(p.dD + static_cast<int64_t>(r) * 128, acc);
}

// dQ (Eq. (2), Alg. 3 step 3): one warp owns query row (q, i) and sums
// g[q, b] * D[cu[b] + argmax[q, b, i]] over the documents, its list visited
// from rotation(row, n_docs) upward, wrapping around.  The argmax entries of
// a CTA's 8 rows (consecutive i of one query) share 32-byte sectors, so its
// warps read them through L1; an entry outside its document contributes
// nothing (the sort reports it).  (Transposing the argmax into per-row lists
// first, in a kernel of its own, measured slower once the gathers kept four
// loads in flight: training-shape backward 127 -> 119 us without it.)
__global__ void __launch_bounds__(256, 5) grad_q_kernel(BwdParams p) {
    const int64_t R = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
    if (R >= static_cast<int64_t>(p.n_q) * p.lq_max) return;
    const int q = query_of(p, static_cast<int>(R));
    const int i = static_cast<int>(R) - q * p.lq_max;
    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    if (i < p.q_lens[q]) {
        const int first = rotation(R, p.n_docs);
        const int32_t *am = p.argmax + static_cast<int64_t>(q) * p.n_docs * p.lq_max + i;
        const float *g = p.grad + static_cast<int64_t>(q) * p.n_docs;
        warp_gather(p.D, p.bf16 != 0, p.n_docs,
                    [&](int j, bool valid, int &row, float &w) {
                        if (!valid) return;
                        int b = j + first;
                        if (b >= p.n_docs) b -= p.n_docs;
                        const int a = __ldg(am + static_cast<int64_t>(b) * p.lq_max);
                        const int lo = __ldg(p.cu_seqlens + b), hi = __ldg(p.cu_seqlens + b + 1);
                        row = (a >= 0 && a < hi - lo) ? lo + a : -1;
                        w = g[b];
                    },
                    acc);
    }
    warp_store_row(p.dQ + R * 128, acc);
}

// A plain L2-resident read: every CTA streams the buffer's 16-byte words
// `passes` times (grid-stride), folding them into one word per thread so the
// loads cannot be dropped; sink[blockIdx.x] receives the fold.
__global__ void __launch_bounds__(512) l2_read_probe_kernel(const uint4 *buf, int64_t n16, int passes,
                                                            unsigned long long *sink) {
    uint32_t f = 0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int pass = 0; pass < passes; ++pass)
        for (int64_t k = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; k < n16; k += 4 * stride) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = k + u * stride < n16 ? __ldcg(buf + k + u * stride) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 4; ++u) f ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
        }
    for (int off = 16; off > 0; off >>= 1) f ^= __shfl_xor_sync(0xffffffffu, f, off);
    if ((threadIdx.x & 31) == 0) atomicXor(sink + blockIdx.x, static_cast<unsigned long long>(f));
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

cudaError_t launch_build_csr(const BwdParams &p, cudaStream_t stream) {
    if (p.n_docs == 0) {
        return cudaMemsetAsync(p.row_ptr, 0, sizeof(int32_t) * (p.total_tokens + 1), stream);
    }
    cudaError_t e = cudaSuccess;
    const unsigned grid = static_cast<unsigned>(p.n_docs) * p.chunks;
    // a document longer than kCsrSmallDoc needs a second, large-footprint launch
    const bool any_large = p.total_tokens > kCsrSmallDoc;
    if ((e = cudaMemsetAsync(p.doc_count, 0, sizeof(int32_t) * (p.n_docs + 1), stream)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(csr_chunk_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kCsrSmemBytes)) != cudaSuccess)
        return e;
    csr_chunk_hist_kernel<<<grid, 256, kCsrSmallHistBytes, stream>>>(p, false);
    if (any_large) csr_chunk_hist_kernel<<<grid, 256, kCsrSmemBytes, stream>>>(p, true);
    csr_doc_scan_kernel<<<1, 1024, 0, stream>>>(p);
    csr_token_scan_kernel<<<p.n_docs, 256, 0, stream>>>(p);
    if ((e = cudaFuncSetAttribute(csr_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kCsrSmemBytes)) != cudaSuccess)
        return e;
    csr_place_kernel<<<grid, kCsrThreads, kCsrSmallPlaceBytes, stream>>>(p, false);
    if (any_large) csr_place_kernel<<<grid, kCsrThreads, kCsrSmemBytes, stream>>>(p, true);
    return cudaGetLastError();
}

// (Chunks of 4096 for page-length documents halve the scan work per
// candidate but fit fewer CTAs per SM: the ColPali-shape sort went 52 -> 57 us.)
int sort_chunks(int32_t n_q, int32_t lq_max) {
    const int64_t n_cand = static_cast<int64_t>(n_q) * lq_max;
    const int64_t c = (n_cand + kSortChunkTarget - 1) / kSortChunkTarget;
    return static_cast<int>(c < 1 ? 1 : (c > kSortMaxChunks ? kSortMaxChunks : c));
}

static_assert(kSortMaxChunkLen * 8 + 8 * SortHist<1024>::kStride * 4 + 1025 * 4 + 16 + 8 * kSortQueries + 64 <=
                  227 * 1024,
              "the largest sort chunk fits one CTA's shared memory (1024-token windows, 8 warps)");
static_assert(kSortMaxChunkLen * 8 + 16 * SortHist<256>::kStride * 4 + 257 * 4 + 16 + 8 * kSortQueries + 64 +
                      16 * 256 * 4 <= 227 * 1024,
              "the largest sort chunk fits one CTA's shared memory (256-token windows, 16 warps)");

template <int WIN, int W>
cudaError_t launch_sort(const BwdParams &p, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(bwd_sort_kernel<WIN, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sort_smem_bytes<WIN, W>(kSortMaxChunkLen)));
    if (e != cudaSuccess) return e;
    bwd_sort_kernel<WIN, W><<<static_cast<unsigned>(p.n_docs) * p.sort_chunks, 32 * W,
                              sort_smem_bytes<WIN, W>(p.sort_chunk_len), stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_sort_and_grad_d(const BwdParams &p, cudaStream_t stream) {
    if (p.total_tokens == 0 || p.n_docs == 0) return cudaSuccess;
    if (static_cast<int64_t>(p.n_q) * p.lq_max == 0)   // no source: every row is 0
        return cudaMemsetAsync(p.dD, 0, sizeof(float) * 128 * static_cast<size_t>(p.total_tokens), stream);
    // windows of 1024 tokens when documents average more than 256
    const bool long_docs = sort_long_docs(p.total_tokens, p.n_docs);
    cudaError_t e = long_docs ? launch_sort<1024, 8>(p, stream) : launch_sort<256, 16>(p, stream);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (static_cast<int64_t>(p.total_tokens) + kRunBlock - 1) / kRunBlock;
    grad_d_kernel<<<static_cast<unsigned>(blocks), 32 * kRunBlock, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_grad_q(const BwdParams &p, cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(p.n_q) * p.lq_max;
    if (rows == 0) return cudaSuccess;
    grad_q_kernel<<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_l2_read_probe(const void *buf, size_t bytes, int passes, unsigned long long *sink, int ctas,
                                 cudaStream_t stream) {
    l2_read_probe_kernel<<<ctas, 512, 0, stream>>>(static_cast<const uint4 *>(buf),
                                                   static_cast<int64_t>(bytes / 16), passes, sink);
    return cudaGetLastError();
}

}  // namespace maxsim
