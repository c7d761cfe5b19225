// Choice of kernel for the two contraction-shaped steps (GEMM, attention).
#pragma once
#include "kernels.h"

namespace g2 {

// Device workspace the GEMM path needs for a model of this size (split-K partials).
size_t gemm_workspace_bytes(int M, int C, int Vp, int L);
// Runs D = epi(A . B^T) on the fastest kernel that takes the shape: the tcgen05
// tensor-core kernel for bf16 operands it supports, the SIMT kernel otherwise.
cudaError_t gemm_dispatch(const GemmArgs& a, float* ws, size_t ws_bytes, cudaStream_t s);
// True when the tensor-core kernel takes this product (else the SIMT kernel would).
bool gemm_tc_path(const GemmArgs& a);
// TF32 products (fp32 operands, a.tf32 set): bytes of a.tws that K-major copies of the
// M/N-major operands need, and the product itself (tensor cores on K-major copies, then
// the residual / GELU / GELU' epilogue as an fp32 pass; exact fp32 SIMT if it cannot).
size_t gemm_tf32_pack_bytes(int M, int N, int K, bool a_kmajor, bool b_kmajor);
cudaError_t gemm_dispatch_tf32(const GemmArgs& a, float* ws, size_t ws_bytes, cudaStream_t s);

// flags (may be null): device error flags, G2_FLAG_TIMEOUT is OR-ed in if a bounded
// wait of the tensor-core kernel expires.
cudaError_t attention_forward(ActType at, void* out, float* lse, const void* qkv, int B, int T,
                              int C, int NH, cudaStream_t s, int* flags = nullptr);
cudaError_t attention_backward(ActType at, void* dqkv, const void* dout, const void* qkv,
                               const void* out, const float* lse, int B, int T, int C, int NH,
                               float* scratch_D, cudaStream_t s, int* flags = nullptr);

}  // namespace g2
