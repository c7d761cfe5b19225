// Kernel selection for GEMM and attention.
#include "dispatch.h"

#include <algorithm>

#include "gemm_tc.h"

namespace g2 {

// The largest split-K workspace of the weight-gradient products of one model.
size_t gemm_workspace_bytes(int M, int C, int Vp, int) {
    size_t b = 256;
    const int shapes[][2] = {{3 * C, C}, {C, C}, {4 * C, C}, {C, 4 * C}, {Vp, C}};
    for (auto& sh : shapes) b = std::max(b, gemm_tc_workspace_bytes(sh[0], sh[1], M));
    return b;
}

bool gemm_tc_path(const GemmArgs& a) { return gemm_tc_supported(a); }

cudaError_t gemm_dispatch(const GemmArgs& a, float* ws, size_t ws_bytes, cudaStream_t s) {
    if (a.in_type == ACT_F32 && a.tf32) return gemm_dispatch_tf32(a, ws, ws_bytes, s);
    if (gemm_tc_supported(a)) return gemm_tc(a, ws, ws_bytes, a.flags, s);
    gemm_tc_note_variant("simt");
    return gemm_simt(a, s);
}

cudaError_t attention_forward(ActType at, void* out, float* lse, const void* qkv, int B, int T,
                              int C, int NH, cudaStream_t s, int* flags) {
    if (attention_tc_supported(at, C, NH, qkv)) {
        cudaError_t e = attention_forward_tc(out, lse, qkv, B, T, C, NH, flags, s);
        if (e != cudaErrorNotSupported) return e;  // else: no tensor map for this shape
    }
    return attention_forward_simt(at, out, lse, qkv, B, T, C, NH, s);
}

cudaError_t attention_backward(ActType at, void* dqkv, const void* dout, const void* qkv,
                               const void* out, const float* lse, int B, int T, int C, int NH,
                               float* scratch_D, cudaStream_t s, int* flags) {
    if (attention_tc_supported(at, C, NH, qkv)) {
        cudaError_t e = attention_backward_tc(dqkv, dout, qkv, out, lse, B, T, C, NH, scratch_D, flags, s);
        if (e != cudaErrorNotSupported) return e;
    }
    return attention_backward_simt(at, dqkv, dout, qkv, out, lse, B, T, C, NH, scratch_D, s);
}

}  // namespace g2
