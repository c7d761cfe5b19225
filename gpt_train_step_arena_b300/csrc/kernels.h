// Host-side launchers of the GPT-2 train-step kernels.  Every launcher is
// stream-ordered, allocates nothing and returns cudaGetLastError() of its launch(es).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace g2 {

typedef __nv_bfloat16 bf16;

// Activation element type of a launch.
enum ActType { ACT_F32 = 0, ACT_BF16 = 1 };

// Process-wide count of kernel launches queued by the launchers below.
void count_launches(unsigned n);
uint64_t launches_total();

// ---- diagnostics ------------------------------------------------------------------
// A one-thread kernel whose bounded mbarrier wait (limit limit_ns) expires: sets
// G2_FLAG_TIMEOUT in *flags and returns.
cudaError_t bounded_wait_check(int* flags, unsigned long long limit_ns, cudaStream_t s);

// ---- token ids (llm.c §1.23 validation) --------------------------------------
cudaError_t check_ids(const int32_t* ids, int M, int V, int* flags, int flag_bit, cudaStream_t s);

// ---- encoder (llm.c §1.1, §1.2) ----------------------------------------------
cudaError_t encoder_forward(ActType at, void* out, const int32_t* tok, const void* wte,
                            const void* wpe, int B, int T, int C, int V, int* flags, cudaStream_t s);
// dwpe (maxT,C) fp32 is overwritten: rows t<T get sum_b dout[b,t,:] (b ascending), rows t>=T get 0.
cudaError_t encoder_backward_wpe(ActType at, float* dwpe, const void* dout, int B, int T, int C,
                                 int maxT, cudaStream_t s);
// Scratch for the deterministic token-bucketed dwte accumulation.
struct EncoderBwdScratch {
    int* chunk_cnt;     // nchunks * V ints
    int* cnt;           // V
    int* start;         // V + 1
    int* item_start;    // V + 1
    int* item_tok;      // max_items
    int* perm;          // M
    float* partial;     // max_items * C
    int max_items;
};
size_t encoder_bwd_scratch_bytes(int M, int V, int C);
void encoder_bwd_scratch_carve(EncoderBwdScratch* sc, void* base, int M, int V, int C);
// dwte (V,C) fp32 += per-token sums of dout rows, summed in ascending position order.
cudaError_t encoder_backward_wte(ActType at, float* dwte, const void* dout, const int32_t* tok,
                                 int M, int C, int V, const EncoderBwdScratch* sc, cudaStream_t s);

// ---- layernorm (llm.c §1.3, §1.4) and RMSNorm ("microGPT 3D", lesson 04) ---------
// NORM_RMS: out = x * rstd * w with rstd = 1/sqrt(mean(x^2) + 1e-5); b is not read (may be
// null), mean (may be null) receives 0; the backward leaves db = 0 and ignores mean.
enum NormKind { NORM_LAYER = 0, NORM_RMS = 1 };
cudaError_t layernorm_forward(ActType at, void* out, float* mean, float* rstd, const void* inp,
                              const float* w, const float* b, int M, int C, NormKind nk, cudaStream_t s);
// dres (M,C) += LN-backward(dout); dw, db (C) fp32 overwritten.  part: ln_bwd_partial_floats().
// dres_sum (C floats, may be null) receives the column sums of the updated dres as stored
// (the bias gradient of the layer whose output gradient dres is); cs_part (colsum
// partials) is then required.
size_t ln_bwd_partial_floats(int C);
cudaError_t layernorm_backward(ActType at, void* dres, float* dw, float* db, float* dres_sum, const void* dout,
                               const void* inp, const float* w, const float* mean, const float* rstd, int M,
                               int C, float* part, float* cs_part, NormKind nk, cudaStream_t s);

// ---- bias gradient: out[n] = sum_m X[m,n] (fixed order) --------------------------
size_t colsum_partial_floats(int M, int N);
cudaError_t colsum(ActType at, float* out, const void* X, int M, int N, float* part, cudaStream_t s);
// out[c] = sum over i < n of part[i*N + c], rows added in a fixed order (the second pass
// of colsum; also the sum of a product epilogue's per-row-group column sums); n = 0
// writes zeros.
cudaError_t colsum_reduce(float* out, const float* part, int n, int N, cudaStream_t s);

// ---- fused softmax + cross-entropy forward and backward (llm.c §1.13-§1.15) -------
// logits (M,Vp) is overwritten in place by dlogits = (softmax - onehot) * dloss over the
// first V columns and 0 over the padding; losses[m] = logsumexp - logit[target].
cudaError_t softmax_xent(ActType at, void* logits, float* losses, const int32_t* targets, int M,
                         int V, int Vp, float dloss, int* flags, cudaStream_t s);
// out[0] = mean of x[0..n) in a fixed summation order.
cudaError_t mean_fixed_order(float* out, const float* x, int n, cudaStream_t s);

// ---- AdamW over a flat fp32 buffer (llm.c §1.26) --------------------------------
// shadow (optional) receives the bf16 rounding of the updated parameters.
cudaError_t adamw(float* p, const float* g, float* m, float* v, bf16* shadow, size_t n, float lr,
                  float b1, float b2, float eps, float wd, float c1, float c2, cudaStream_t s);
cudaError_t cast_f32_to_bf16(bf16* out, const float* in, size_t n, cudaStream_t s);

// ---- causal multi-head attention (llm.c §1.7, §1.8; flash-style recompute) -------
// out (B,T,C); lse (B,NH,T) fp32 log-sum-exp of each query row's scores.
cudaError_t attention_forward_simt(ActType at, void* out, float* lse, const void* qkv, int B,
                                   int T, int C, int NH, cudaStream_t s);
// dqkv (B,T,3C) overwritten.  scratch_D: B*NH*T floats.
cudaError_t attention_backward_simt(ActType at, void* dqkv, const void* dout, const void* qkv,
                                    const void* out, const float* lse, int B, int T, int C,
                                    int NH, float* scratch_D, cudaStream_t s);

// D[b,h,t] = sum_d dout[b,t,h,d] * out[b,t,h,d]  (B*NH*T floats)
cudaError_t attention_bwd_dot(ActType at, float* D, const void* dout, const void* out, int B, int T,
                              int C, int NH, cudaStream_t s);
// tcgen05 forward (bf16, head size 64, 16-byte aligned qkv).  flags (may be null):
// G2_FLAG_TIMEOUT is OR-ed in if a bounded wait expires.
bool attention_tc_supported(ActType at, int C, int NH, const void* qkv);
cudaError_t attention_forward_tc(void* out, float* lse, const void* qkv, int B, int T, int C, int NH, int* flags,
                                 cudaStream_t s);
// Its backward: dqkv (B,T,3C) overwritten; Dbuf (B*NH*T floats) receives rowsum(dout * out).
// cudaErrorNotSupported when the tensor maps cannot be built (caller falls back).
cudaError_t attention_backward_tc(void* dqkv, const void* dout, const void* qkv, const void* out, const float* lse,
                                  int B, int T, int C, int NH, float* Dbuf, int* flags, cudaStream_t s);

// ---- generation with a key/value cache (picoGPT generate; llm.c §1.35 sample_mult) ----
// Rows r = b*n + i are the new positions t0+i of sequence b; ids is (B, maxT) int32 and
// kv (B, maxT, 2C) holds [key | value] of every position computed so far.  dstate (may
// be null): 4 ints in device memory {t0, step, n_new, temperature bits} that replace the
// corresponding arguments (one-token steps replayed from a CUDA graph).
cudaError_t gen_embed(ActType at, void* x, const int32_t* ids, const void* wte, const void* wpe, int B, int n, int t0,
                      int maxT, int C, const int* dstate, cudaStream_t s);
cudaError_t gen_kv_append(ActType at, void* kv, const void* qkv, int B, int n, int t0, int maxT, int C,
                          const int* dstate, cudaStream_t s);
// out (B*n, C) = attention of each new query over the cached positions 0..t0+i.
size_t gen_attn_smem_bytes(int C, int NH, int maxT);
cudaError_t gen_attention(ActType at, void* out, const void* qkv, const void* kv, int B, int n, int t0, int maxT,
                          int C, int NH, const int* dstate, cudaStream_t s);
cudaError_t gen_last_rows(ActType at, void* last, const void* x, int B, int n, int C, cudaStream_t s);
// Next id per sequence from logits (B, Vp): argmax (temperature <= 0) or sample_mult over
// softmax(logits / temperature) with coins[b*n_new + step]; written to ids[b, t_next]
// (if t_next < maxT) and out[b*n_new + step].  With dstate: t_next = t0 + 1.
cudaError_t gen_sample(ActType at, int32_t* ids, int32_t* out, const void* logits, int B, int V, int Vp,
                       float temperature, const float* coins, int step, int n_new, int t_next, int maxT,
                       const int* dstate, cudaStream_t s);
// dstate t0 and step += 1.
cudaError_t gen_advance(int* dstate, cudaStream_t s);

// ---- seeded initial parameters (llm.c §1.33 random_u32, §1.34 random_f32) ----------
// Normal tensors in draw order: params + offset[k] receives n[k] values N(0, std[k]).
struct InitPlan {
    int count;
    size_t offset[8];
    size_t n[8];
    double std[8];
};
// Fills the n_ones arrays ones[i] (ones_n[i] floats) with 1 and draws the plan's normal
// tensors; everything else is left as it is (the caller zeroes it first).
cudaError_t init_params_device(float* params, const InitPlan& plan, const float* const* ones, const size_t* ones_n,
                               int n_ones, uint64_t seed, cudaStream_t s);

// ---- GEMM --------------------------------------------------------------------------
// D[m,n] = epilogue( sum_k A(m,k) * B(n,k) ), A(m,k) = A[m*sAm + k*sAk], B(n,k) = B[n*sBn + k*sBk].
enum Epilogue {
    EPI_STORE = 0,      // D = acc (+bias[n]) (+R[m,n])
    EPI_GELU = 1,       // D = acc + bias (pre-activation), D2 = gelu(acc + bias)
    EPI_GELU_BWD = 2,   // D = acc * gelu'(P[m,n])
};
struct GemmArgs {
    int M, N, K;
    ActType in_type;            // A and B element type
    const void* A; long long sAm, sAk;
    const void* B; long long sBn, sBk;
    void* D; long long ldd; int d_f32;   // D element type: fp32 if d_f32 else in_type
    const float* bias;          // [N] or null
    const void* R; long long ldr;        // residual added to D (in_type), or null
    void* D2; long long ldd2;            // EPI_GELU second output (in_type)
    const void* P; long long ldp;        // EPI_GELU_BWD pre-activation (in_type)
    int epi;
    int* flags;                 // device error flags (G2_FLAG_TIMEOUT), or null
    int skinny_split;           // one row tile (M <= 128): split K, epilogue in the fixed-order reduce
    int tf32;                   // fp32 operands: contract on the tensor cores as TF32 (else exact fp32)
    float* tws;                 // TF32: workspace for K-major copies of M/N-major operands, or null
    size_t tws_bytes;
    // EPI_GELU_BWD on the bf16 tensor-core path (gemm_tc_fuses_colsum): the epilogue also
    // writes the column sums of the stored bf16 output per 32-row group,
    // colsum_part[ceil(M/32)][N] fp32 (8-byte aligned), for colsum_reduce to add up; or null
    float* colsum_part;
};
cudaError_t gemm_simt(const GemmArgs& a, cudaStream_t s);

}  // namespace g2
