// noalloc.cu -- maxsim_forward without a caller-supplied workspace.
//
// Some callers cannot allocate device memory at the point where they score:
// a plugin that runs inside a host framework which owns every device
// allocation and hands its plugins no allocator, or a latency-critical
// serving loop that must never call cudaMalloc / cudaFree (both can
// synchronise the whole device and stall every stream).  For them this file
// keeps the forward's scratch -- the per-32-token partial sums of queries
// longer than 32 tokens, and the FP16 copy of an INT8 query -- in one
// fixed-size array in device memory that the library owns for the life of
// the process.
//
// The array is a file-scope __device__ variable: each GPU that loads the
// library holds kNoAllocScratchBytes for it until the process exits.  Its
// device address is looked up once per device and context (the first call
// with that device current, and again after the device's context has been
// destroyed and re-created, e.g. by cudaDeviceReset) and cached.
#include "maxsim.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <unordered_map>

namespace {

// 4 MiB: room for about one million FP32 partial sums, e.g. a 1024-token
// query against 32,000 documents.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct ScratchAddress {
    CUcontext ctx = nullptr;   // the context the address belongs to
    void *ptr = nullptr;
};

std::mutex g_noalloc_mu;
std::unordered_map<int, ScratchAddress> g_noalloc_ptr;   // device ordinal -> address in its current context
PFN_cuCtxGetCurrent_v4000 g_ctx_get_current = nullptr;

// Device address of the scratch array on the current device.  In host code
// the array's name only stands in for the symbol; the real address must come
// from cudaGetSymbolAddress with the device current.
maxsim_status_t scratch_on_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MAXSIM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_ctx_get_current == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return MAXSIM_ERR_CUDA;
        g_ctx_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    }
    // Before the runtime's first call on this device no context may be
    // current (ctx == nullptr): the symbol lookup below makes the primary
    // context current, and the context is read again after it.
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return MAXSIM_ERR_CUDA;
    auto it = g_noalloc_ptr.find(dev);
    if (it == g_noalloc_ptr.end() || ctx == nullptr || it->second.ctx != ctx) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return MAXSIM_ERR_CUDA;
        if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return MAXSIM_ERR_CUDA;
        it = g_noalloc_ptr.insert_or_assign(dev, ScratchAddress{ctx, ptr}).first;
    }
    *out = it->second.ptr;
    return MAXSIM_OK;
}

}  // namespace

extern "C" {

maxsim_status_t maxsim_forward_noalloc(const void *Q, const int32_t *q_lens, int32_t n_q, int32_t lq_max,
                                       const void *D, const int32_t *cu_seqlens, int32_t n_docs,
                                       int64_t total_d_tokens, int32_t dim, maxsim_dtype_t dtype,
                                       float q_scale, float d_scale, float *scores, int64_t *raw_scores,
                                       int32_t *argmax, void *stream) {
    const size_t need = maxsim_forward_workspace_size(n_q, lq_max, n_docs, dim, dtype);
    if (need > kNoAllocScratchBytes) return MAXSIM_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0) {
        const maxsim_status_t st = scratch_on_current_device(&scratch);
        if (st != MAXSIM_OK) return st;
    }
    // Nothing in the scratch needs clearing: every partial sum the final
    // pass reads, and every FP16 query element, is written earlier in the
    // same call.
    return maxsim_forward(Q, q_lens, n_q, lq_max, D, cu_seqlens, n_docs, total_d_tokens, dim, dtype,
                          q_scale, d_scale, scores, raw_scores, argmax, scratch, need, stream);
}

}  // extern "C"
