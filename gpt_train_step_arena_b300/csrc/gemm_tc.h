// tcgen05 tensor-core GEMM (bf16 operands, fp32 accumulation).
#pragma once
#include "kernels.h"

namespace g2 {

// True when the product's layout, alignment and sizes fit the tensor-core kernel.
bool gemm_tc_supported(const GemmArgs& a);
// Workspace the kernel wants for split-K partial sums of an fp32-output product.
size_t gemm_tc_workspace_bytes(int M, int N, int K);
// Workspace of a product with one row tile (M <= 128) launched with skinny_split set.
size_t gemm_tc_skinny_workspace_bytes(int M, int N, int K);
// flags (may be null): G2_FLAG_TIMEOUT is OR-ed in if a bounded wait expires.
cudaError_t gemm_tc(const GemmArgs& a, float* ws, size_t ws_bytes, int* flags, cudaStream_t s);

}  // namespace g2
