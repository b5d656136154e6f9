// chamfer.cu -- fused Chamfer distance with its inverse-grid backward.
//
// "FLASH-MAXSIM: IO-Aware Fused Kernels for Late-Interaction Retrieval"
// (arXiv 2605.29517) §4.2 "Generalization to Chamfer Distance": the MaxSim
// skeleton with a minimum over squared Euclidean distances instead of a
// maximum over inner products, and a backward that inverts the saved
// argmin through the same destination-owned CSR as Alg. 3.
//
//   CD(P, Q) = 1/N sum_p min_q |p - q|^2 + 1/M sum_q min_p |q - p|^2
//
// GB300 design.  Points have three coordinates, so the contraction is far
// too thin for the tensor cores: the search is bound by FP32 issue.  One
// thread owns four source points (two packed pairs) and streams target
// tiles from shared memory, where every coordinate is stored twice so one
// 64-bit register feeds both halves of a packed f32x2 instruction: each
// distance costs three packed instructions per two sources.  Sixteen
// distances are reduced with three-input minima before the rare update of
// the running (min, argmin).  Large target sets are split into slices that
// run as separate CTAs and are merged in slice order (lowest index wins).
//
// The ranked distance is fma(dz, dz, fma(dy, dy, dx * dx)) with
// dx = s.x - t.x, every step rounded to nearest even.
#include "internal.cuh"
#include "sm103.cuh"

#include <algorithm>
#include <cstdint>

namespace maxsim {
namespace {

using namespace ptx;

constexpr int kNnThreads = 256;
constexpr int kNnPerThread = 4;                          // two packed source pairs
constexpr int kNnSources = kNnThreads * kNnPerThread;    // sources per CTA
constexpr int kNnTile = 1024;                            // targets per shared tile
constexpr int kNnChunk = 16;                             // distances per min tree

// A target with each coordinate duplicated into both halves of a 64-bit word.
struct __align__(16) TargetPair {
    uint64_t xx, yy, zz, pad;
};

__device__ __forceinline__ uint64_t pack2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void unpack2(uint64_t v, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}

__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t fma2l(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Squared distances of two sources (packed) to one target.
__device__ __forceinline__ uint64_t dist2(uint64_t sx, uint64_t sy, uint64_t sz, const TargetPair &t) {
    const uint64_t dx = sub2(sx, t.xx);
    uint64_t d = mul2(dx, dx);
    const uint64_t dy = sub2(sy, t.yy);
    d = fma2l(dy, dy, d);
    const uint64_t dz = sub2(sz, t.zz);
    return fma2l(dz, dz, d);
}

__device__ __forceinline__ float min16(const float (&v)[kNnChunk]) {
    const float a = fmin3(v[0], v[1], v[2]), b = fmin3(v[3], v[4], v[5]);
    const float c = fmin3(v[6], v[7], v[8]), d = fmin3(v[9], v[10], v[11]);
    const float e = fmin3(v[12], v[13], v[14]);
    return fmin3(fmin3(a, b, c), fmin3(d, e, v[15]), INFINITY);
}

__device__ __forceinline__ int item_of(const int32_t *cu, int n_items, int64_t i) {
    // the item whose range [cu[b], cu[b+1]) holds i
    int lo = 0, hi = n_items - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= i) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Nearest target of each source.  CTA = (item, tile of 1024 sources, slice
// of the item's targets).  With slices > 1 the results go to per-slice
// partials (slice-major, stride total_s) merged by chamfer_merge_kernel.
__global__ void __launch_bounds__(kNnThreads, 2)
chamfer_nn_kernel(const float *__restrict__ S, const int32_t *__restrict__ cu_s, const float *__restrict__ T,
                  const int32_t *__restrict__ cu_t, int32_t tiles_s, int32_t slices, int32_t max_s, int32_t max_t,
                  int64_t total_s, float *__restrict__ out_d, int32_t *__restrict__ out_a, int32_t *status) {
    __shared__ TargetPair tile[kNnTile];
    const int tid = threadIdx.x;
    const int slice = blockIdx.x % slices;
    const int rest = blockIdx.x / slices;
    const int st = rest % tiles_s;
    const int b = rest / tiles_s;
    const int64_t s_begin = cu_s[b], s_end = cu_s[b + 1];
    const int64_t t_begin = cu_t[b];
    const int64_t m = static_cast<int64_t>(cu_t[b + 1]) - t_begin;
    if (tid == 0 && st == 0 && slice == 0 && (s_end - s_begin > max_s || m > max_t))
        atomicCAS(status, 0, kStatusSetTooLarge);
    const int64_t s0 = s_begin + static_cast<int64_t>(st) * kNnSources;
    if (s0 >= s_end) return;
    const int64_t lo = m * slice / slices, hi = m * (slice + 1) / slices;

    uint64_t sx[2], sy[2], sz[2];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        float c[2][3];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t s = s0 + tid + (2 * p + h) * kNnThreads;
#pragma unroll
            for (int k = 0; k < 3; ++k) c[h][k] = s < s_end ? S[3 * s + k] : 0.0f;
        }
        sx[p] = pack2(c[0][0], c[1][0]);
        sy[p] = pack2(c[0][1], c[1][1]);
        sz[p] = pack2(c[0][2], c[1][2]);
    }
    float best[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
    int32_t arg[4] = {-1, -1, -1, -1};

    for (int64_t t0 = lo; t0 < hi; t0 += kNnTile) {
        const int cnt = static_cast<int>(hi - t0 < kNnTile ? hi - t0 : kNnTile);
        __syncthreads();
        for (int j = tid; j < kNnTile; j += kNnThreads) {
            float x = INFINITY, y = INFINITY, z = INFINITY;  // padding never wins
            if (j < cnt) {
                const float *pt = T + 3 * (t_begin + t0 + j);
                x = pt[0];
                y = pt[1];
                z = pt[2];
            }
            tile[j] = TargetPair{pack2(x, x), pack2(y, y), pack2(z, z), 0ull};
        }
        __syncthreads();
        const int n_chunks = (cnt + kNnChunk - 1) / kNnChunk;
#pragma unroll 1
        for (int c = 0; c < n_chunks; ++c) {
            float d[4][kNnChunk];
#pragma unroll
            for (int j = 0; j < kNnChunk; ++j) {
                const TargetPair t = tile[c * kNnChunk + j];
#pragma unroll
                for (int p = 0; p < 2; ++p) unpack2(dist2(sx[p], sy[p], sz[p], t), d[2 * p][j], d[2 * p + 1][j]);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float cm = min16(d[r]);
                if (cm < best[r]) {
                    int idx = 0;
#pragma unroll
                    for (int j = kNnChunk - 1; j >= 0; --j) idx = d[r][j] == cm ? j : idx;
                    best[r] = cm;
                    arg[r] = static_cast<int32_t>(t0 + c * kNnChunk + idx);
                }
            }
        }
    }
    const int64_t base = slices > 1 ? static_cast<int64_t>(slice) * total_s : 0;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int64_t s = s0 + tid + r * kNnThreads;
        if (s < s_end) {
            out_d[base + s] = best[r];
            out_a[base + s] = arg[r];
        }
    }
}

// Merge per-slice results in slice order: a later slice replaces the
// running best only when strictly closer, so ties keep the lower index.
__global__ void chamfer_merge_kernel(const float *__restrict__ part_d, const int32_t *__restrict__ part_a,
                                     int32_t slices, int64_t total_s, float *__restrict__ dist,
                                     int32_t *__restrict__ arg) {
    for (int64_t s = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; s < total_s;
         s += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float best = INFINITY;
        int32_t a = -1;
        for (int k = 0; k < slices; ++k) {
            const float v = part_d[k * total_s + s];
            if (v < best) {
                best = v;
                a = part_a[k * total_s + s];
            }
        }
        dist[s] = best;
        arg[s] = a;
    }
}

__device__ __forceinline__ double block_sum_f64(double v, double *red) {
    // fixed-shape tree over the CTA (256 threads): deterministic
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    double t = 0.0;
    if (warp == 0) {
        t = lane < (blockDim.x >> 5) ? red[lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    }
    __syncthreads();
    return t;
}

// cd[b] = mean of dist_pq over item b's P + mean of dist_qp over its Q,
// summed in binary64 in a fixed order (a mean over an empty set is 0).
__global__ void __launch_bounds__(256)
chamfer_reduce_kernel(const float *__restrict__ dist_pq, const int32_t *__restrict__ cu_p,
                      const float *__restrict__ dist_qp, const int32_t *__restrict__ cu_q, float *__restrict__ cd) {
    __shared__ double red[8];
    const int b = blockIdx.x;
    double a = 0.0, c = 0.0;
    for (int64_t i = cu_p[b] + threadIdx.x; i < cu_p[b + 1]; i += blockDim.x) a += static_cast<double>(dist_pq[i]);
    for (int64_t j = cu_q[b] + threadIdx.x; j < cu_q[b + 1]; j += blockDim.x) c += static_cast<double>(dist_qp[j]);
    a = block_sum_f64(a, red);
    c = block_sum_f64(c, red);
    if (threadIdx.x == 0) {
        const int64_t n = static_cast<int64_t>(cu_p[b + 1]) - cu_p[b];
        const int64_t mm = static_cast<int64_t>(cu_q[b + 1]) - cu_q[b];
        cd[b] = static_cast<float>((n ? a / static_cast<double>(n) : 0.0) + (mm ? c / static_cast<double>(mm) : 0.0));
    }
}

// ------------------------------------------------------------------ CSR
// Stable LSD radix sort of the destinations (8-bit digits), payload = the
// source index: sources within a destination stay in ascending order, the
// order of a stable argsort.  Sources without a destination (index -1) get
// the key total_dst and sort after every real destination.

constexpr int kRadixThreads = 256;
constexpr int kRadixPer = 16;
constexpr int kRadixTile = kRadixThreads * kRadixPer;  // keys per tile
constexpr int kRadixWarps = kRadixThreads / 32;

__global__ void csr_keys_kernel(const int32_t *__restrict__ arg, const int32_t *__restrict__ cu_src,
                                const int32_t *__restrict__ cu_dst, int32_t n_items, int64_t total_src,
                                int32_t total_dst, int32_t *__restrict__ keys, int32_t *__restrict__ vals,
                                int32_t *status) {
    for (int64_t s = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; s < total_src;
         s += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int b = item_of(cu_src, n_items, s);
        const int32_t a = arg[s];
        int32_t key = total_dst;
        if (a >= 0) {
            if (a < cu_dst[b + 1] - cu_dst[b]) key = cu_dst[b] + a;
            else atomicCAS(status, 0, kStatusBadArgmax);
        }
        keys[s] = key;
        vals[s] = static_cast<int32_t>(s);
    }
}

__global__ void __launch_bounds__(kRadixThreads)
radix_hist_kernel(const int32_t *__restrict__ keys, int64_t n, int shift, int32_t n_tiles,
                  int32_t *__restrict__ tile_hist) {
    __shared__ int32_t hist[256];
    hist[threadIdx.x] = 0;
    __syncthreads();
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kRadixTile;
    for (int k = 0; k < kRadixPer; ++k) {
        const int64_t i = base + k * kRadixThreads + threadIdx.x;
        if (i < n) atomicAdd(&hist[(static_cast<uint32_t>(keys[i]) >> shift) & 255u], 1);
    }
    __syncthreads();
    tile_hist[static_cast<int64_t>(threadIdx.x) * n_tiles + blockIdx.x] = hist[threadIdx.x];
}

// In-place exclusive scan of `len` counts, one CTA of 1024 threads, each
// scanning a contiguous run.
__global__ void __launch_bounds__(1024) exclusive_scan_kernel(int32_t *__restrict__ v, int64_t len) {
    __shared__ int32_t warp_sum[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t per = (len + 1023) / 1024;
    const int64_t b = tid * per, e = b + per < len ? b + per : len;
    int32_t local = 0;
    for (int64_t i = b; i < e; ++i) local += v[i];
    int32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int32_t w = warp_sum[lane], wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t t = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += t;
        }
        warp_sum[lane] = wi - w;
    }
    __syncthreads();
    int32_t run = warp_sum[warp] + incl - local;
    for (int64_t i = b; i < e; ++i) {
        const int32_t x = v[i];
        v[i] = run;
        run += x;
    }
}

// Stable scatter of one tile: keys are taken 256 at a time in index order;
// within a round a key's rank among equal digits is the count in earlier
// rounds + earlier warps + earlier lanes of its own warp.
__global__ void __launch_bounds__(kRadixThreads)
radix_scatter_kernel(const int32_t *__restrict__ keys, const int32_t *__restrict__ vals, int64_t n, int shift,
                     int32_t n_tiles, const int32_t *__restrict__ tile_off, int32_t *__restrict__ keys_out,
                     int32_t *__restrict__ vals_out) {
    __shared__ int32_t running[256];
    __shared__ int32_t warp_cnt[kRadixWarps][256];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    running[tid] = tile_off[static_cast<int64_t>(tid) * n_tiles + blockIdx.x];
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kRadixTile;
    for (int k = 0; k < kRadixPer; ++k) {
        for (int w = 0; w < kRadixWarps; ++w) warp_cnt[w][tid] = 0;
        __syncthreads();
        const int64_t i = base + k * kRadixThreads + tid;
        const bool valid = i < n;
        const int32_t key = valid ? keys[i] : 0;
        const int digit = valid ? static_cast<int>((static_cast<uint32_t>(key) >> shift) & 255u) : 256 + lane;
        const uint32_t peers = __match_any_sync(0xffffffffu, digit);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (valid && rank == 0) warp_cnt[warp][digit] = __popc(peers);
        __syncthreads();
        if (valid) {
            int pos = running[digit] + rank;
            for (int w = 0; w < warp; ++w) pos += warp_cnt[w][digit];
            keys_out[pos] = key;
            vals_out[pos] = vals[i];
        }
        __syncthreads();
        int add = 0;
        for (int w = 0; w < kRadixWarps; ++w) add += warp_cnt[w][tid];
        running[tid] += add;
        __syncthreads();
    }
}

// row_ptr[d] = number of sorted keys below d, for d = 0 .. total_dst.
__global__ void csr_row_ptr_kernel(const int32_t *__restrict__ sorted, int64_t n, int32_t total_dst,
                                   int32_t *__restrict__ row_ptr) {
    for (int64_t d = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; d <= total_dst;
         d += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int64_t lo = 0, hi = n;
        while (lo < hi) {
            const int64_t mid = (lo + hi) >> 1;
            if (sorted[mid] < d) lo = mid + 1; else hi = mid;
        }
        row_ptr[d] = static_cast<int32_t>(lo);
    }
}

// ------------------------------------------------------------- backward
// One thread per point x of set A (its item's other set is B):
//   dA[x] = 2 g / |A_b| (x - B[arg_ab[x]])                     (own term)
//         + 2 g / |B_b| sum_{y in CSR_ba[x]} (x - B[y])          (inverse)
// accumulated in FP32 in that order, CSR sources ascending.
__global__ void chamfer_grad_kernel(const float *__restrict__ grad, const float *__restrict__ A,
                                    const int32_t *__restrict__ cu_a, const float *__restrict__ B,
                                    const int32_t *__restrict__ cu_b, int32_t n_items,
                                    const int32_t *__restrict__ arg_ab, const int32_t *__restrict__ row_ptr_ba,
                                    const int32_t *__restrict__ col_ba, int64_t total_a, float *__restrict__ dA) {
    for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < total_a;
         x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int b = item_of(cu_a, n_items, x);
        const float g = grad[b];
        const int64_t na = static_cast<int64_t>(cu_a[b + 1]) - cu_a[b];
        const int64_t nb = static_cast<int64_t>(cu_b[b + 1]) - cu_b[b];
        const float px = A[3 * x], py = A[3 * x + 1], pz = A[3 * x + 2];
        float ax = 0.f, ay = 0.f, az = 0.f;
        const int32_t a = arg_ab[x];
        if (a >= 0 && a < nb) {
            const float w = 2.0f * g / static_cast<float>(na);
            const float *y = B + 3 * (static_cast<int64_t>(cu_b[b]) + a);
            ax = w * (px - y[0]);
            ay = w * (py - y[1]);
            az = w * (pz - y[2]);
        }
        const int32_t e0 = row_ptr_ba[x], e1 = row_ptr_ba[x + 1];
        if (e1 > e0) {
            const float w = 2.0f * g / static_cast<float>(nb);
            for (int32_t e = e0; e < e1; ++e) {
                const float *y = B + 3 * static_cast<int64_t>(col_ba[e]);
                ax = fmaf(w, px - y[0], ax);
                ay = fmaf(w, py - y[1], ay);
                az = fmaf(w, pz - y[2], az);
            }
        }
        dA[3 * x] = ax;
        dA[3 * x + 1] = ay;
        dA[3 * x + 2] = az;
    }
}

int grid_of(int64_t n, int threads, int cap) {
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((n + threads - 1) / threads, cap)));
}

}  // namespace

int chamfer_slices(int32_t n_items, int32_t max_s, int32_t max_t, int sm_count) {
    // CTAs = items x source tiles x slices run in waves of `slots` (two per
    // SM); a CTA's time is proportional to its slice, 1 / s of the targets,
    // so the search takes ceil(ctas / slots) / s.  Take the smallest s within
    // 5 % of the best (fewer, larger CTAs; each slice keeps at least one
    // shared-memory tile of targets, at most 64 slices).
    const int64_t tiles = static_cast<int64_t>(n_items) * ((max_s + kNnSources - 1) / kNnSources);
    const int64_t slots = 2LL * std::max(sm_count, 1);
    const int64_t cap = std::max<int64_t>(1, std::min<int64_t>(64, max_t / kNnTile));
    if (tiles <= 0) return 1;
    auto cost = [&](int64_t sl) {
        return static_cast<double>((tiles * sl + slots - 1) / slots) / static_cast<double>(sl);
    };
    double best = cost(1);
    for (int64_t sl = 2; sl <= cap; ++sl) best = std::min(best, cost(sl));
    for (int64_t sl = 1; sl <= cap; ++sl)
        if (cost(sl) <= best * 1.05) return static_cast<int>(sl);
    return 1;
}

cudaError_t launch_chamfer_nn(const float *S, const int32_t *cu_s, const float *T, const int32_t *cu_t,
                              int32_t n_items, int32_t max_s, int32_t max_t, int64_t total_s, int slices,
                              float *dist, int32_t *arg, float *part_d, int32_t *part_a, int32_t *status,
                              cudaStream_t stream) {
    if (n_items == 0 || total_s == 0 || max_s == 0) return cudaSuccess;
    const int tiles_s = (max_s + kNnSources - 1) / kNnSources;
    const int64_t grid = static_cast<int64_t>(n_items) * tiles_s * slices;
    if (grid > INT32_MAX) return cudaErrorInvalidConfiguration;
    float *od = slices > 1 ? part_d : dist;
    int32_t *oa = slices > 1 ? part_a : arg;
    chamfer_nn_kernel<<<static_cast<int>(grid), kNnThreads, 0, stream>>>(S, cu_s, T, cu_t, tiles_s, slices, max_s,
                                                                         max_t, total_s, od, oa, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || slices == 1) return e;
    chamfer_merge_kernel<<<grid_of(total_s, 256, 4096), 256, 0, stream>>>(part_d, part_a, slices, total_s, dist,
                                                                           arg);
    return cudaGetLastError();
}

cudaError_t launch_chamfer_reduce(const float *dist_pq, const int32_t *cu_p, const float *dist_qp,
                                  const int32_t *cu_q, int32_t n_items, float *cd, cudaStream_t stream) {
    if (n_items == 0) return cudaSuccess;
    chamfer_reduce_kernel<<<n_items, 256, 0, stream>>>(dist_pq, cu_p, dist_qp, cu_q, cd);
    return cudaGetLastError();
}

size_t chamfer_csr_scratch_bytes(int64_t total_src, int32_t total_dst) {
    const int64_t tiles = std::max<int64_t>(1, (total_src + kRadixTile - 1) / kRadixTile);
    (void)total_dst;
    return static_cast<size_t>(4 * total_src + 256 * tiles) * sizeof(int32_t) + 1024;
}

cudaError_t launch_chamfer_csr(const int32_t *arg, const int32_t *cu_src, const int32_t *cu_dst, int32_t n_items,
                               int64_t total_src, int32_t total_dst, int32_t *row_ptr, int32_t *col_idx,
                               void *scratch, int32_t *status, cudaStream_t stream) {
    int32_t *keys0 = static_cast<int32_t *>(scratch);
    int32_t *vals0 = keys0 + total_src;
    int32_t *keys1 = vals0 + total_src;
    int32_t *vals1 = keys1 + total_src;
    int32_t *tile_hist = vals1 + total_src;
    const int64_t n = total_src;
    cudaError_t e = cudaSuccess;
    if (n > 0) {
        csr_keys_kernel<<<grid_of(n, 256, 8192), 256, 0, stream>>>(arg, cu_src, cu_dst, n_items, n, total_dst,
                                                                    keys0, vals0, status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const int32_t n_tiles = static_cast<int32_t>((n + kRadixTile - 1) / kRadixTile);
        int bits = 1;
        while (bits < 31 && (static_cast<int64_t>(1) << bits) <= total_dst) ++bits;
        for (int shift = 0; shift < bits; shift += 8) {
            radix_hist_kernel<<<n_tiles, kRadixThreads, 0, stream>>>(keys0, n, shift, n_tiles, tile_hist);
            exclusive_scan_kernel<<<1, 1024, 0, stream>>>(tile_hist, static_cast<int64_t>(256) * n_tiles);
            radix_scatter_kernel<<<n_tiles, kRadixThreads, 0, stream>>>(keys0, vals0, n, shift, n_tiles, tile_hist,
                                                                        keys1, vals1);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
            std::swap(keys0, keys1);
            std::swap(vals0, vals1);
        }
    }
    csr_row_ptr_kernel<<<grid_of(static_cast<int64_t>(total_dst) + 1, 256, 8192), 256, 0, stream>>>(
        keys0, n, total_dst, row_ptr);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (n > 0) e = cudaMemcpyAsync(col_idx, vals0, sizeof(int32_t) * n, cudaMemcpyDeviceToDevice, stream);
    return e;
}

cudaError_t launch_chamfer_grad(const float *grad, const float *A, const int32_t *cu_a, const float *B,
                                const int32_t *cu_b, int32_t n_items, const int32_t *arg_ab,
                                const int32_t *row_ptr_ba, const int32_t *col_ba, int64_t total_a, float *dA,
                                cudaStream_t stream) {
    if (total_a == 0) return cudaSuccess;
    chamfer_grad_kernel<<<grid_of(total_a, 256, 8192), 256, 0, stream>>>(grad, A, cu_a, B, cu_b, n_items, arg_ab,
                                                                          row_ptr_ba, col_ba, total_a, dA);
    return cudaGetLastError();
}

}  // namespace maxsim
