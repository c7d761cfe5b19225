// Kernel selection for GEMM and attention.
#include "dispatch.h"

namespace g2 {

size_t gemm_workspace_bytes(int, int, int, int) { return 256; }

cudaError_t gemm_dispatch(const GemmArgs& a, float*, size_t, cudaStream_t s) {
    return gemm_simt(a, s);
}

cudaError_t attention_forward(ActType at, void* out, float* lse, const void* qkv, int B, int T,
                              int C, int NH, cudaStream_t s) {
    return attention_forward_simt(at, out, lse, qkv, B, T, C, NH, s);
}

cudaError_t attention_backward(ActType at, void* dqkv, const void* dout, const void* qkv,
                               const void* out, const float* lse, int B, int T, int C, int NH,
                               float* scratch_D, cudaStream_t s) {
    return attention_backward_simt(at, dqkv, dout, qkv, out, lse, B, T, C, NH, scratch_D, s);
}

}  // namespace g2
