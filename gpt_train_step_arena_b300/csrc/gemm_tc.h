// tcgen05 tensor-core GEMM (bf16 operands, fp32 accumulation).
#pragma once
#include "kernels.h"

namespace g2 {

// True when the product's layout, alignment and sizes fit the tensor-core kernel: bf16
// operands, or fp32 operands with tf32 set (then K-major only, fp32 output, store or bias
// epilogue).
bool gemm_tc_supported(const GemmArgs& a);
// True when gemm_tc writes the per-32-row column sums of a GELU' product's output into
// a.colsum_part (set, bf16, EPI_GELU_BWD, N even, 8-byte aligned, tensor-core path).
bool gemm_tc_fuses_colsum(const GemmArgs& a);
// Workspace the kernel wants for split-K partial sums of an fp32-output product.
size_t gemm_tc_workspace_bytes(int M, int N, int K);
// Workspace of a product with one row tile (M <= 128) launched with skinny_split set.
size_t gemm_tc_skinny_workspace_bytes(int M, int N, int K);
// flags (may be null): G2_FLAG_TIMEOUT is OR-ed in if a bounded wait expires.
cudaError_t gemm_tc(const GemmArgs& a, float* ws, size_t ws_bytes, int* flags, cudaStream_t s);
// Tile override for every later product (128 or 256 rows on one SM, 2 for two-SM CTA
// pairs; anything else: chosen per shape); returns the previous setting.  Products with a
// staged epilogue input never take 256-row tiles on one SM.
int gemm_tc_force_tile_rows(int rows);
// "rows=.. cols=.. splits=.. a=k|mn b=k|mn epi=.." of the last launch ("none" before any).
void gemm_tc_last_variant(char* out, size_t n);
// Replaces that description (the dispatcher notes a product it sent elsewhere).
void gemm_tc_note_variant(const char* v);

}  // namespace g2
