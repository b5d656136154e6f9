// fwd_tc.cu -- launches of the fused MaxSim forward (the kernel itself is in
// fwd_kernel.cuh) and its small companion kernels: the per-chunk partial-sum
// pass, the all-empty fill, the INT8 query widening, the block-offset rebase
// of the out-of-core path and the bounded-wait self-test.
//
// "FLASH-MAXSIM: IO-Aware Fused Kernels for Late-Interaction Retrieval"
// (arXiv 2605.29517) §4.1 (Alg. 2), §4.3.1, §4.3.2.
#include "internal.cuh"
#include "sm103.cuh"
#include "fwd_kernel.cuh"

#include <cuda_fp16.h>

namespace maxsim {
namespace {

using namespace ptx;

// Sum the per-32-token-chunk partials of queries longer than 32 tokens, in
// chunk order (the query-chunk decomposition of §4.1).
__global__ void finalize_partials_kernel(FwdParams p, int n_chunks, bool int8) {
    const int64_t n_pairs = static_cast<int64_t>(p.n_q) * p.n_docs;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n_pairs;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int q = static_cast<int>(idx / p.n_docs);
        const int b = static_cast<int>(idx - static_cast<int64_t>(q) * p.n_docs);
        const int64_t out = static_cast<int64_t>(q) * p.ld_out + b;
        if (int8) {
            long long s = 0;
            for (int c = 0; c < n_chunks; ++c) s += p.ipartials[c * n_pairs + idx];
            const bool neg_inf = p.cu_seqlens[b + 1] == p.cu_seqlens[b] && p.q_lens[q] > 0;
            if (p.raw_scores) p.raw_scores[out] = neg_inf ? INT64_MIN : s;
            p.scores[out] = neg_inf ? -INFINITY : static_cast<float>(static_cast<double>(s) * p.int8_scale);
        } else {
            float s = 0.0f;
            for (int c = 0; c < n_chunks; ++c) s += p.partials[c * n_pairs + idx];
            p.scores[out] = s;
        }
    }
}

// No document has a token (or no query has a row): every score is an empty
// maximum (-inf) for a query with tokens, an empty sum (0) otherwise.
__global__ void fill_empty_kernel(FwdParams p, bool int8) {
    const int64_t n_pairs = static_cast<int64_t>(p.n_q) * p.n_docs;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n_pairs;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int q = static_cast<int>(idx / p.n_docs);
        const int b = static_cast<int>(idx - static_cast<int64_t>(q) * p.n_docs);
        const int64_t out = static_cast<int64_t>(q) * p.ld_out + b;
        const bool has = p.q_lens[q] > 0;
        p.scores[out] = has ? -INFINITY : 0.0f;
        if (int8 && p.raw_scores) p.raw_scores[out] = has ? INT64_MIN : 0;
        if (p.argmax)
            for (int i = 0; i < p.lq_max; ++i) p.argmax[out * p.lq_max + i] = -1;
    }
}

__global__ void int8_to_f16_kernel(const int8_t *__restrict__ src, __half *__restrict__ dst, int64_t n) {
    for (int64_t k = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; k < n;
         k += static_cast<int64_t>(gridDim.x) * blockDim.x)
        dst[k] = __int2half_rn(static_cast<int>(src[k]));
}

template <int NMT, bool ARGMAX, bool INT8, bool SCALE>
cudaError_t launch_one(const CUtensorMap &tmQ, const CUtensorMap &tmD, const FwdParams &p,
                       cudaStream_t stream) {
    using C = Cfg<NMT, INT8>;
    auto kern = maxsim_fwd_kernel<NMT, ARGMAX, INT8, SCALE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    kern<<<p.groups * p.parts, C::kThreads, C::kSmem, stream>>>(tmQ, tmD, p);
    return cudaGetLastError();
}

template <bool ARGMAX, bool INT8, bool SCALE>
cudaError_t launch_nmt(int nmt, const CUtensorMap &tmQ, const CUtensorMap &tmD, const FwdParams &p,
                       cudaStream_t stream) {
    switch (nmt) {
        case 1: return launch_one<1, ARGMAX, INT8, SCALE>(tmQ, tmD, p, stream);
        case 2: return launch_one<2, ARGMAX, INT8, SCALE>(tmQ, tmD, p, stream);
        default: return launch_one<4, ARGMAX, INT8, SCALE>(tmQ, tmD, p, stream);
    }
}

int grid_for(int64_t n, int threads) {
    return static_cast<int>(std::min<int64_t>((n + threads - 1) / threads, 4096));
}

}  // namespace

int forward_smem_bytes(int nmt, bool int8) {
    if (int8) return nmt == 1 ? Cfg<1, true>::kSmem : nmt == 2 ? Cfg<2, true>::kSmem : Cfg<4, true>::kSmem;
    return nmt == 1 ? Cfg<1, false>::kSmem : nmt == 2 ? Cfg<2, false>::kSmem : Cfg<4, false>::kSmem;
}

int forward_ctas_per_sm(int nmt, bool int8) {
    if (int8) return nmt == 1 ? Cfg<1, true>::kCtasPerSm : nmt == 2 ? Cfg<2, true>::kCtasPerSm : Cfg<4, true>::kCtasPerSm;
    return nmt == 1 ? Cfg<1, false>::kCtasPerSm : nmt == 2 ? Cfg<2, false>::kCtasPerSm : Cfg<4, false>::kCtasPerSm;
}

bool forward_stage_split(int nmt, bool int8) {
    if (int8) return nmt == 1 ? Cfg<1, true>::kKSplit : nmt == 2 ? Cfg<2, true>::kKSplit : Cfg<4, true>::kKSplit;
    return nmt == 1 ? Cfg<1, false>::kKSplit : nmt == 2 ? Cfg<2, false>::kKSplit : Cfg<4, false>::kKSplit;
}

int forward_threads(int nmt, bool int8) {
    if (int8) return nmt == 1 ? Cfg<1, true>::kThreads : nmt == 2 ? Cfg<2, true>::kThreads : Cfg<4, true>::kThreads;
    return nmt == 1 ? Cfg<1, false>::kThreads : nmt == 2 ? Cfg<2, false>::kThreads : Cfg<4, false>::kThreads;
}

cudaError_t launch_forward(const CUtensorMap &tmQ, const CUtensorMap &tmD, const FwdParams &p,
                           int nmt, bool with_argmax, FwdMode mode, cudaStream_t stream) {
    switch (mode) {
        case FwdMode::kInt8Tensor:
            return with_argmax ? launch_nmt<true, true, false>(nmt, tmQ, tmD, p, stream)
                               : launch_nmt<false, true, false>(nmt, tmQ, tmD, p, stream);
        case FwdMode::kInt8Token:
            return with_argmax ? launch_nmt<true, true, true>(nmt, tmQ, tmD, p, stream)
                               : launch_nmt<false, true, true>(nmt, tmQ, tmD, p, stream);
        default:
            return with_argmax ? launch_nmt<true, false, false>(nmt, tmQ, tmD, p, stream)
                               : launch_nmt<false, false, false>(nmt, tmQ, tmD, p, stream);
    }
}

cudaError_t launch_finalize_partials(const FwdParams &p, bool int8, cudaStream_t stream) {
    const int64_t n = static_cast<int64_t>(p.n_q) * p.n_docs;
    if (n == 0) return cudaSuccess;
    finalize_partials_kernel<<<grid_for(n, 256), 256, 0, stream>>>(p, p.lq_pad / 32, int8);
    return cudaGetLastError();
}

cudaError_t launch_fill_empty(const FwdParams &p, bool int8, cudaStream_t stream) {
    const int64_t n = static_cast<int64_t>(p.n_q) * p.n_docs;
    if (n == 0) return cudaSuccess;
    fill_empty_kernel<<<grid_for(n, 256), 256, 0, stream>>>(p, int8);
    return cudaGetLastError();
}

// Offsets of a block of documents [b0, b0 + n) of a larger corpus, rebased
// so the block reads as a corpus of its own: dst[k] = src[k] - src[0] for
// k = 0 .. n, with src = corpus offsets + b0.
__global__ void rebase_offsets_kernel(const int32_t *src, int32_t *dst, int32_t n) {
    const int32_t base = src[0];
    for (int32_t k = blockIdx.x * blockDim.x + threadIdx.x; k <= n; k += gridDim.x * blockDim.x)
        dst[k] = src[k] - base;
}

cudaError_t launch_rebase_offsets(const int32_t *src, int32_t *dst, int32_t n, cudaStream_t stream) {
    rebase_offsets_kernel<<<grid_for(static_cast<int64_t>(n) + 1, 256), 256, 0, stream>>>(src, dst, n);
    return cudaGetLastError();
}

// The forward's failure path in miniature: warp 1 holds TMEM, thread 0 waits
// on a barrier that nothing completes until its bounded wait gives up
// (raising the CTA's abort flag and recording the status code), thread 32
// waits on the same barrier until it sees the abort flag; then the CTA
// releases TMEM and exits as the forward does.
__global__ void __launch_bounds__(64) wait_selftest_kernel(int32_t *status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    __shared__ int32_t abort_word;
    volatile int32_t *abort_flag = &abort_word;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        abort_word = 0;
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 32);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, abort_flag, status, kStatusSelfTestExpired, limit_ns);
    if (threadIdx.x == 32) mbar_wait(&bar, 0, abort_flag, status, kStatusSelfTestExpired, 4 * limit_ns);
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 32);
}

cudaError_t launch_wait_selftest(int32_t *status, uint64_t limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 64, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_int8_to_f16(const int8_t *src, uint16_t *dst, int64_t n, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    int8_to_f16_kernel<<<grid_for(n, 256), 256, 0, stream>>>(src, reinterpret_cast<__half *>(dst), n);
    return cudaGetLastError();
}

}  // namespace maxsim
