// Bias gradient for callers that cannot allocate device memory.
//
// gpt2_op_bias_grad needs a workspace for its per-row-block partial sums, which the
// caller normally allocates.  Some callers cannot: a plugin running inside a host
// framework whose caching allocator has already reserved the device's memory (a
// cudaMalloc of its own would fail or fragment that pool), or a deployment that
// forbids device allocation once it has started.  gpt2_op_bias_grad_noalloc keeps the
// partial sums in a fixed array that lives in the library's own device image instead.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "../../include/gpt2.h"
#include "../../include/gpt2_ops.h"
#include "kernels.h"

void g2_op_set_error(const char* msg);

namespace {

// Partial sums of the bias gradient: ceil(M/256) * N floats at most.  4 MiB, held by
// every device that loads the library until the process exits.
constexpr size_t kNoAllocScratchFloats = size_t(1) << 20;
__device__ __align__(256) float g_bias_grad_scratch[kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};
// Id of the context the cached address belongs to.  A cudaDeviceReset destroys the
// device's primary context; the next one loads the library's device image afresh, so
// the array may sit at another address and the cache must be refreshed.  Context ids
// are unique for the life of the process (a new context never reuses an old id).
unsigned long long g_scratch_ctx[kMaxDevices] = {};

// Id of the calling thread's current context (0 if it cannot be read: the address is
// then looked up on every call, which is always correct).
unsigned long long current_ctx_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = (GetCurrent)f;
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = (GetId)f;
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

int set_error(int code, const char* msg) {
    g2_op_set_error(msg);
    return code;
}

}  // namespace

extern "C" size_t gpt2_op_bias_grad_noalloc_max_floats(void) { return kNoAllocScratchFloats; }

extern "C" int gpt2_op_bias_grad_noalloc(int dtype, const void* dout, int M, int N, float* dbias,
                                         void* stream) {
    char msg[256];
    if (dtype != GPT2_DT_F32 && dtype != GPT2_DT_BF16)
        return set_error(GPT2_ERR_ARG, "bias_grad_noalloc: bad dtype");
    if (M < 0 || N <= 0) return set_error(GPT2_ERR_ARG, "bias_grad_noalloc: bad shape");
    if (!dbias || (M > 0 && !dout)) return set_error(GPT2_ERR_ARG, "bias_grad_noalloc: null pointer");
    size_t need = g2::colsum_partial_floats(M, N);
    if (need > kNoAllocScratchFloats) {
        snprintf(msg, sizeof msg,
                 "bias_grad_noalloc: M=%d N=%d needs %zu scratch floats, the fixed array holds %zu "
                 "(ceil(M/256)*N must not exceed it); use gpt2_op_bias_grad with a workspace",
                 M, N, need, kNoAllocScratchFloats);
        return set_error(GPT2_ERR_ARG, msg);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(GPT2_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return set_error(GPT2_ERR_ARG, "bias_grad_noalloc: device id too large");
    // (before the runtime has made a context current this is 0 and the lookup below,
    // which creates the context, runs again on the next call)
    const unsigned long long ctx = current_ctx_id();
    float* scratch;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_scratch_ptr[dev] || ctx == 0 || g_scratch_ctx[dev] != ctx) {
            // the device address of the array on the current device (host code cannot
            // use the symbol itself)
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_bias_grad_scratch);
            if (e != cudaSuccess) {
                snprintf(msg, sizeof msg, "bias_grad_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
                return set_error(GPT2_ERR_CUDA, msg);
            }
            g_scratch_ptr[dev] = (float*)p;
            g_scratch_ctx[dev] = ctx;
        }
        scratch = g_scratch_ptr[dev];
    }
    // Every partial is written before it is read, so the array needs no clearing.
    e = g2::colsum(dtype == GPT2_DT_BF16 ? g2::ACT_BF16 : g2::ACT_F32, dbias, dout, M, N, scratch,
                   (cudaStream_t)stream);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "bias_grad_noalloc: %s", cudaGetErrorString(e));
        return set_error(GPT2_ERR_CUDA, msg);
    }
    return GPT2_OK;
}
