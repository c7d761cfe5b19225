/*
 * gpt2_ops.h — single operations of the GPT-2 training step on caller-owned device
 * memory.  These are the kernels the model in gpt2.h chains, exposed one by one so a
 * caller (or a test) can run a step of the chain on its own buffers.
 *
 * Conventions:
 *  - Every pointer argument is a device pointer unless its name ends in _host.
 *    Arrays are dense row-major.  The caller owns all memory; nothing is allocated.
 *  - `dtype` selects the element type of activation-like arrays: GPT2_DT_F32 (float)
 *    or GPT2_DT_BF16 (bfloat16).  Parameters, gradients and statistics are fp32.
 *  - Work is queued on `stream` (a cudaStream_t; NULL = legacy default stream) and the
 *    call returns without waiting.  The return value is a gpt2_status (gpt2.h);
 *    gpt2_op_last_error() describes the last failure of any gpt2_op_* call in the
 *    process.
 */
#ifndef GPT2_B300_OPS_H
#define GPT2_B300_OPS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* GPT2_DT_TF32 (gpt2_op_matmul only): fp32 operands and output, contracted on the tensor
 * cores with the operands read as TF32 and fp32 accumulation. */
enum gpt2_dtype { GPT2_DT_F32 = 0, GPT2_DT_BF16 = 1, GPT2_DT_TF32 = 2 };

const char* gpt2_op_last_error(void);

/* Bias gradient of a linear layer (llm.c annotated listing, §1.6 matmul_backward:
 * dbias[o] accumulates dout[b,t,o] over all positions).  dbias[n] = sum over m of
 * dout[m,n], for dout (M,N) of `dtype`; dbias (N) fp32 is overwritten.  The sum order is
 * fixed by (M,N), so results are bitwise reproducible.  `workspace` must hold
 * gpt2_op_bias_grad_workspace(M,N) bytes (GPT2_ERR_ARG if smaller); its contents on
 * entry do not matter. */
size_t gpt2_op_bias_grad_workspace(int M, int N);
int gpt2_op_bias_grad(int dtype, const void* dout, int M, int N, float* dbias, void* workspace,
                      size_t workspace_bytes, void* stream);

/* Bias gradient without a caller workspace.  The paper has no counterpart: this is an
 * interface for callers that cannot allocate device memory, for example a plugin
 * running inside a host framework whose caching allocator already holds the device's
 * memory, or a deployment that forbids device allocation after start-up.  Same result
 * as gpt2_op_bias_grad (same kernels, same summation order), but the partial sums live
 * in a fixed array inside the library: 2^20 floats (4 MiB), which every device that
 * loads the library keeps until the process exits.  It requires ceil(M/256) * N <=
 * gpt2_op_bias_grad_noalloc_max_floats() and returns GPT2_ERR_ARG (with a message in
 * gpt2_op_last_error) beyond that.  It allocates nothing.  The first call on a device
 * looks up the array's device address with that device current; make that first call
 * before any stream capture.  After a cudaDeviceReset the device gets a new context
 * (and the array a possibly new address): the first call in that context looks the
 * address up again, so it too belongs before any capture.  All calls share the one
 * array, which keeps the last call's partial sums (every partial is written before it
 * is read, so nothing needs clearing): calls whose work overlaps on the GPU (different
 * streams, or different host threads) race on it and must be serialised by the
 * caller.  dout needs no particular alignment. */
int gpt2_op_bias_grad_noalloc(int dtype, const void* dout, int M, int N, float* dbias,
                              void* stream);
size_t gpt2_op_bias_grad_noalloc_max_floats(void);

/* Matrix product (llm.c §1.5 matmul_forward, §1.6 matmul_backward):
 *   D[m,n] = sum_k A(m,k) * B(n,k) (+ bias[n]),  0 <= m < M, 0 <= n < N, 0 <= k < K.
 * A is stored K-major (A(m,k) at A[m*lda + k]) when a_kmajor != 0, else M-major
 * (A(m,k) at A[k*lda + m]); likewise B with b_kmajor and ldb.  A and B are `dtype`;
 * D (row stride ldd) is fp32 when d_f32 != 0, else `dtype`.  bias (N floats) may be
 * NULL.  The three products of a linear layer map onto this as: forward
 * (X . W^T: both K-major), input gradient (dY . W: A K-major, B N-major) and weight
 * gradient (dY^T . X: both M/N-major, fp32 out).  `workspace` (may be NULL when
 * workspace_bytes is 0) receives split-K partial sums when the kernel uses them. */
int gpt2_op_matmul(int dtype, int M, int N, int K, const void* A, long long lda, int a_kmajor,
                   const void* B, long long ldb, int b_kmajor, void* D, long long ldd, int d_f32,
                   const float* bias, void* workspace, size_t workspace_bytes, void* stream);
/* Workspace bytes gpt2_op_matmul can use for this product: split-K partial sums (optional:
 * with less, the product is not split) and, for GPT2_DT_TF32, K-major copies of the
 * operands given M- or N-major (required; the workspace must then be 256-byte aligned).
 * With GPT2_DT_TF32, D is always fp32 (d_f32 is ignored). */
size_t gpt2_op_matmul_workspace(int dtype, int M, int N, int K, int a_kmajor, int b_kmajor);

/* The same product with the epilogues the training step fuses into it (llm.c §1.5
 * matmul_forward with §1.11 residual_forward or §1.9 gelu_forward; §1.6 with §1.10
 * gelu_backward), bf16 tensor-core path only (GPT2_DT_BF16, D bf16):
 *   GPT2_EPI_STORE     D = A.B^T (+ bias[n]) (+ R[m,n])           R: (M,N) bf16, row stride ldr
 *   GPT2_EPI_GELU      D = A.B^T + bias[n]; D2 = gelu_tanh(D)      D2: (M,N) bf16, row stride ldd2
 *   GPT2_EPI_GELU_BWD  D = (A.B^T) * gelu_tanh'(P[m,n])            P: (M,N) bf16, row stride ldp
 * Unused pointers may be NULL.  Returns GPT2_ERR_ARG for an epilogue the layout or dtype
 * cannot take (the fused path needs 16-byte aligned operands and strides that are
 * multiples of 8 elements). */
enum gpt2_epilogue { GPT2_EPI_STORE = 0, GPT2_EPI_GELU = 1, GPT2_EPI_GELU_BWD = 2 };
int gpt2_op_matmul_ex(int dtype, int M, int N, int K, const void* A, long long lda, int a_kmajor,
                      const void* B, long long ldb, int b_kmajor, void* D, long long ldd, const float* bias,
                      const void* R, long long ldr, void* D2, long long ldd2, const void* P, long long ldp,
                      int epilogue, void* workspace, size_t workspace_bytes, void* stream);

/* The FC layer's pre-activation gradient and its bias gradient in one call (llm.c §1.6
 * matmul_backward: dbias[o] = sum over positions of dout[., o]; §1.10 gelu_backward),
 * bf16 only:
 *   D[m,n] = (A.B^T)[m,n] * gelu_tanh'(P[m,n])     as gpt2_op_matmul_ex with GPT2_EPI_GELU_BWD
 *   dbias[n] = sum over 0 <= m < M of D[m,n]        fp32, overwritten, over the stored bf16 D
 * The product's epilogue sums each 32-row group's columns into the workspace and a
 * fixed-order pass adds the groups (should the epilogue not take it, a separate column-sum
 * pass reads D, which then needs ldd == N).  Sums are in a fixed order, so two calls give
 * bitwise equal results.  workspace: device memory of at least
 * gpt2_op_matmul_gelu_bwd_bias_grad_workspace(M, N) bytes, 8-byte aligned.  Returns
 * GPT2_ERR_ARG (nothing launched) for null pointers, a layout the fused path cannot take
 * (as gpt2_op_matmul_ex) or a short workspace; M = 0 writes dbias = 0. */
size_t gpt2_op_matmul_gelu_bwd_bias_grad_workspace(int M, int N);
int gpt2_op_matmul_gelu_bwd_bias_grad(int M, int N, int K, const void* A, long long lda, int a_kmajor,
                                      const void* B, long long ldb, int b_kmajor, void* D, long long ldd,
                                      const void* P, long long ldp, float* dbias, void* workspace,
                                      size_t workspace_bytes, void* stream);

/* AdamW over n fp32 elements (llm.c §1.26 gpt2_update), in place on p, m, v; g is read.
 * shadow_bf16 (n bfloat16, may be NULL) receives the rounded updated parameters.
 * t >= 1 counts updates. */
int gpt2_op_adamw(float* p, const float* g, float* m, float* v, void* shadow_bf16, size_t n,
                  float lr, float b1, float b2, float eps, float wd, int t, void* stream);

/* Causal multi-head attention forward (llm.c §1.7; picoGPT attention with its causal
 * mask).  qkv (B,T,3C) holds query | key | value, head h at channels [h*hs,(h+1)*hs)
 * of each, hs = C/NH.  out (B,T,C) is overwritten with softmax(q k^T / sqrt(hs)) v
 * over keys t2 <= t; lse (B,NH,T) fp32 with each row's log-sum-exp of the scaled
 * scores (kept for the backward instead of the (T,T) probabilities). */
int gpt2_op_attention_forward(int dtype, void* out, float* lse, const void* qkv, int B, int T,
                              int C, int NH, void* stream);
/* Its backward (llm.c §1.8): dqkv (B,T,3C) is overwritten with the gradients of q, k
 * and v given dout (B,T,C), the forward's qkv, out and lse.  workspace: B*NH*T floats. */
int gpt2_op_attention_backward(int dtype, void* dqkv, const void* dout, const void* qkv,
                               const void* out, const float* lse, int B, int T, int C, int NH,
                               float* workspace, void* stream);

/* LayerNorm forward (llm.c annotated listing §1.3 layernorm_forward; picoGPT
 * layer_norm): for each of the M rows of inp (M,C) of `dtype`, out = (x - mean) * rstd
 * * w + b with the row mean, the biased variance and rstd = 1/sqrt(var + 1e-5).
 * out (M,C) `dtype` is overwritten; mean and rstd (M floats each) receive the row
 * statistics; w and b are C floats.  M may be 0. */
int gpt2_op_layernorm_forward(int dtype, void* out, float* mean, float* rstd, const void* inp,
                              const float* w, const float* b, int M, int C, void* stream);

/* Its backward (llm.c §1.4 layernorm_backward).  dinp (M,C) `dtype` is ACCUMULATED into
 * (dinp += d loss / d inp, as in the listing, which is how the residual stream's
 * gradient is carried); dw and db (C floats) are OVERWRITTEN with the weight and bias
 * gradients summed over the rows in a fixed order (the listing accumulates into zeroed
 * buffers: the same values).  mean and rstd are the forward's statistics.  workspace
 * must hold gpt2_op_layernorm_backward_workspace(C) bytes. */
size_t gpt2_op_layernorm_backward_workspace(int C);
int gpt2_op_layernorm_backward(int dtype, void* dinp, float* dw, float* db, const void* dout,
                               const void* inp, const float* w, const float* mean,
                               const float* rstd, int M, int C, void* workspace,
                               size_t workspace_bytes, void* stream);

/* RMSNorm forward, the normalisation of the microGPT block (page "microGPT 3D",
 * lesson 04; the page names the operation only, this is its standard definition with
 * LayerNorm's eps and gain and no shift): for each of the M rows of inp (M,C) of
 * `dtype`, out = x * rstd * w with rstd = 1/sqrt(mean(x^2) + 1e-5).  out (M,C) `dtype`
 * is overwritten; rstd (M floats) receives the row statistic; w is C floats.  M may
 * be 0. */
int gpt2_op_rmsnorm_forward(int dtype, void* out, float* rstd, const void* inp, const float* w, int M,
                            int C, void* stream);

/* Its backward: with n = x * rstd and g = w * dout, dinp += (g - n * mean(g * n)) * rstd
 * (ACCUMULATED, like gpt2_op_layernorm_backward) and dw (C floats) is OVERWRITTEN with
 * sum over rows of n * dout in a fixed order.  rstd is the forward's statistic.
 * workspace must hold gpt2_op_rmsnorm_backward_workspace(C) bytes. */
size_t gpt2_op_rmsnorm_backward_workspace(int C);
int gpt2_op_rmsnorm_backward(int dtype, void* dinp, float* dw, const void* dout, const void* inp,
                             const float* w, const float* rstd, int M, int C, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Fused softmax + cross-entropy forward and backward (llm.c §1.13 softmax_forward,
 * §1.14 crossentropy_forward, §1.15 crossentropy_softmax_backward; picoGPT lm_loss).
 * logits (M,Vp) of `dtype` with V <= Vp real columns: for each row, lse = logsumexp of
 * the V real logits, losses[m] = lse - logit[targets[m]], and the row is OVERWRITTEN
 * in place with (softmax - onehot(target)) * dloss over the V real columns and 0 over
 * the Vp - V padding columns.  targets: M int32 device ids; one outside [0, V) gives
 * that row loss 0 and no one-hot term, and the call returns GPT2_ERR_TOKEN after
 * waiting for the stream (flags, 4 bytes of device memory, must be given for that
 * check; pass NULL to skip it and return without waiting). */
int gpt2_op_softmax_xent(int dtype, void* logits, float* losses, const int32_t* targets, int M,
                         int V, int Vp, float dloss, int* flags, void* stream);

/* Token + position embedding (llm.c §1.1 encoder_forward; picoGPT gpt2's
 * wte[inputs] + wpe[range(len(inputs))]): out[b,t,:] = wte[tokens[b,t],:] + wpe[t,:] for
 * tokens (B,T) int32 device ids, wte (V,C) and wpe (>= T rows, C) of `dtype`, out (B,T,C)
 * of `dtype` overwritten.  An id outside [0,V) ORs 1 into *flags (4 bytes of device
 * memory, required; never cleared here) and gives that row wpe[t] alone. */
int gpt2_op_encoder_forward(int dtype, void* out, const int32_t* tokens, const void* wte, const void* wpe, int B,
                            int T, int C, int V, int* flags, void* stream);

/* Its backward (llm.c §1.2 encoder_backward), deterministic: dwpe (maxT,C) fp32 is
 * OVERWRITTEN (rows t < T get the sum over b, in ascending b, of dout[b,t,:]; rows
 * t >= T get 0) and dwte (V,C) fp32 is ACCUMULATED into (row k += the sum of the dout
 * rows whose id is k, in ascending position order; the listing's += into the gradient
 * the tied LM head already wrote).  Positions are bucketed by id with a stable integer
 * counting sort, so no float atomics are used and the result is bitwise reproducible.
 * Ids outside [0,V) are skipped.  workspace: gpt2_op_encoder_backward_workspace(B*T, V,
 * C) bytes, 256-byte aligned; its contents on entry do not matter. */
size_t gpt2_op_encoder_backward_workspace(int M, int V, int C);
int gpt2_op_encoder_backward(int dtype, float* dwte, float* dwpe, const void* dout, const int32_t* tokens, int B,
                             int T, int C, int V, int maxT, void* workspace, size_t workspace_bytes, void* stream);

/* Tile height of the tensor-core matrix product, a test and tuning hook: rows = 128 or
 * 256 makes every later bf16 tensor-core product of the process use tiles of that many
 * rows on one SM each; rows = 2 makes it use 256-row tiles computed by clusters of two
 * CTAs on two SMs (128 rows and half of each B tile per SM; products with 128-column
 * tiles or a single row tile keep the per-shape choice); any other value restores the
 * choice per shape (the default); returns the previous setting.  Products whose epilogue
 * reads a staged input (residual, GELU') never use 256-row tiles on one SM.  Not
 * synchronised with work in flight: set it between launches. */
int gpt2_op_gemm_force_tile_rows(int rows);
/* The kernel variant of the last matrix product launched by this process, as
 * "rows=R cols=N splits=S a=k|mn b=k|mn epi=...", or "simt" when the last product took
 * the CUDA-core kernel (fp32, or a layout the tensor-core path does not take; "none"
 * before any).  The string
 * belongs to the calling thread and stays valid until its next call. */
const char* gpt2_op_gemm_last_variant(void);

#ifdef __cplusplus
}
#endif
#endif /* GPT2_B300_OPS_H */
