// C ABI of include/gpt2_ops.h: argument checks and one launcher call each.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/gpt2.h"
#include "../../include/gpt2_ops.h"
#include "dispatch.h"
#include "gemm_tc.h"
#include "kernels.h"

using namespace g2;

static std::mutex g_op_err_mu;
static std::string g_op_err;

static int op_fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    std::lock_guard<std::mutex> lk(g_op_err_mu);
    g_op_err = buf;
    return code;
}

static int op_cuda(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return GPT2_OK;
    return op_fail(GPT2_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static bool dtype_ok(int dt) { return dt == GPT2_DT_F32 || dt == GPT2_DT_BF16; }
static ActType act_of(int dt) { return dt == GPT2_DT_BF16 ? ACT_BF16 : ACT_F32; }

extern "C" const char* gpt2_op_last_error(void) {
    std::lock_guard<std::mutex> lk(g_op_err_mu);
    return g_op_err.c_str();
}

extern "C" size_t gpt2_op_bias_grad_workspace(int M, int N) {
    if (M < 0 || N <= 0) return 0;
    return colsum_partial_floats(M, N) * sizeof(float);
}

extern "C" int gpt2_op_bias_grad(int dtype, const void* dout, int M, int N, float* dbias,
                                 void* workspace, size_t workspace_bytes, void* stream) {
    if (!dtype_ok(dtype)) return op_fail(GPT2_ERR_ARG, "bias_grad: bad dtype %d", dtype);
    if (M < 0 || N <= 0) return op_fail(GPT2_ERR_ARG, "bias_grad: bad shape M=%d N=%d", M, N);
    if (!dbias || (M > 0 && !dout)) return op_fail(GPT2_ERR_ARG, "bias_grad: null pointer");
    size_t need = gpt2_op_bias_grad_workspace(M, N);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return op_fail(GPT2_ERR_ARG, "bias_grad: workspace of %zu bytes needed, %zu given", need,
                       workspace_bytes);
    return op_cuda(colsum(act_of(dtype), dbias, dout, M, N, (float*)workspace, (cudaStream_t)stream),
                   "bias_grad");
}

extern "C" size_t gpt2_op_matmul_workspace(int dtype, int M, int N, int K, int a_kmajor, int b_kmajor) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    size_t b = gemm_tc_workspace_bytes(M, N, K);
    if (dtype == GPT2_DT_TF32) b += gemm_tf32_pack_bytes(M, N, K, a_kmajor != 0, b_kmajor != 0);
    return b;
}

extern "C" int gpt2_op_matmul(int dtype, int M, int N, int K, const void* A, long long lda,
                              int a_kmajor, const void* B, long long ldb, int b_kmajor, void* D,
                              long long ldd, int d_f32, const float* bias, void* workspace,
                              size_t workspace_bytes, void* stream) {
    const bool tf32 = dtype == GPT2_DT_TF32;
    if (!dtype_ok(dtype) && !tf32) return op_fail(GPT2_ERR_ARG, "matmul: bad dtype %d", dtype);
    if (M < 0 || N < 0 || K < 0) return op_fail(GPT2_ERR_ARG, "matmul: negative size");
    if (M == 0 || N == 0) return GPT2_OK;
    if (!A || !B || !D) return op_fail(GPT2_ERR_ARG, "matmul: null pointer");
    GemmArgs a{};
    a.M = M; a.N = N; a.K = K; a.in_type = tf32 ? ACT_F32 : act_of(dtype);
    if (tf32) {
        // the operand copies first, the split-K partials after them
        const size_t pk = gemm_tf32_pack_bytes(M, N, K, a_kmajor != 0, b_kmajor != 0);
        if (pk && (!workspace || workspace_bytes < pk))
            return op_fail(GPT2_ERR_ARG, "matmul: TF32 needs %zu workspace bytes for operand copies", pk);
        if ((uintptr_t)workspace & 255) return op_fail(GPT2_ERR_ARG, "matmul: workspace must be 256-byte aligned");
        a.tf32 = 1;
        a.tws = (float*)workspace;
        a.tws_bytes = pk;
        workspace = pk ? (void*)((char*)workspace + pk) : workspace;
        workspace_bytes = workspace ? workspace_bytes - pk : 0;
        d_f32 = 1;
    }
    a.A = A;
    if (a_kmajor) { a.sAm = lda; a.sAk = 1; } else { a.sAm = 1; a.sAk = lda; }
    a.B = B;
    if (b_kmajor) { a.sBn = ldb; a.sBk = 1; } else { a.sBn = 1; a.sBk = ldb; }
    a.D = D; a.ldd = ldd; a.d_f32 = d_f32 ? 1 : 0;
    a.bias = bias;
    a.epi = EPI_STORE;
    return op_cuda(gemm_dispatch(a, (float*)workspace, workspace ? workspace_bytes : 0,
                                 (cudaStream_t)stream), "matmul");
}

extern "C" int gpt2_op_matmul_ex(int dtype, int M, int N, int K, const void* A, long long lda, int a_kmajor,
                                 const void* B, long long ldb, int b_kmajor, void* D, long long ldd,
                                 const float* bias, const void* R, long long ldr, void* D2, long long ldd2,
                                 const void* P, long long ldp, int epilogue, void* workspace,
                                 size_t workspace_bytes, void* stream) {
    if (dtype != GPT2_DT_BF16) return op_fail(GPT2_ERR_ARG, "matmul_ex: the fused epilogues take bf16 only");
    if (epilogue < GPT2_EPI_STORE || epilogue > GPT2_EPI_GELU_BWD)
        return op_fail(GPT2_ERR_ARG, "matmul_ex: bad epilogue %d", epilogue);
    if (M < 0 || N < 0 || K < 0) return op_fail(GPT2_ERR_ARG, "matmul_ex: negative size");
    if (M == 0 || N == 0) return GPT2_OK;
    if (!A || !B || !D) return op_fail(GPT2_ERR_ARG, "matmul_ex: null pointer");
    if (epilogue == GPT2_EPI_GELU && (!D2 || !bias)) return op_fail(GPT2_ERR_ARG, "matmul_ex: GELU needs bias and D2");
    if (epilogue == GPT2_EPI_GELU_BWD && !P) return op_fail(GPT2_ERR_ARG, "matmul_ex: GELU_BWD needs P");
    GemmArgs a{};
    a.M = M; a.N = N; a.K = K; a.in_type = ACT_BF16;
    a.A = A;
    if (a_kmajor) { a.sAm = lda; a.sAk = 1; } else { a.sAm = 1; a.sAk = lda; }
    a.B = B;
    if (b_kmajor) { a.sBn = ldb; a.sBk = 1; } else { a.sBn = 1; a.sBk = ldb; }
    a.D = D; a.ldd = ldd; a.d_f32 = 0;
    a.bias = epilogue == GPT2_EPI_GELU_BWD ? nullptr : bias;
    a.R = epilogue == GPT2_EPI_STORE ? R : nullptr; a.ldr = ldr;
    a.D2 = D2; a.ldd2 = ldd2;
    a.P = P; a.ldp = ldp;
    a.epi = epilogue == GPT2_EPI_GELU ? EPI_GELU : epilogue == GPT2_EPI_GELU_BWD ? EPI_GELU_BWD : EPI_STORE;
    if (!gemm_tc_path(a)) return op_fail(GPT2_ERR_ARG, "matmul_ex: layout or alignment outside the fused path");
    return op_cuda(gemm_dispatch(a, (float*)workspace, workspace ? workspace_bytes : 0, (cudaStream_t)stream),
                   "matmul_ex");
}

extern "C" size_t gpt2_op_matmul_gelu_bwd_bias_grad_workspace(int M, int N) {
    if (M <= 0 || N <= 0) return 0;
    const size_t groups = (size_t)((M + 31) / 32) * N;
    return std::max(groups, colsum_partial_floats(M, N)) * sizeof(float);
}

extern "C" int gpt2_op_matmul_gelu_bwd_bias_grad(int M, int N, int K, const void* A, long long lda, int a_kmajor,
                                                 const void* B, long long ldb, int b_kmajor, void* D, long long ldd,
                                                 const void* P, long long ldp, float* dbias, void* workspace,
                                                 size_t workspace_bytes, void* stream) {
    if (M < 0 || N < 0 || K < 0) return op_fail(GPT2_ERR_ARG, "gelu_bwd_bias_grad: negative size");
    if (N == 0) return GPT2_OK;
    if (!dbias) return op_fail(GPT2_ERR_ARG, "gelu_bwd_bias_grad: null dbias");
    cudaStream_t s = (cudaStream_t)stream;
    if (M == 0) return op_cuda(cudaMemsetAsync(dbias, 0, (size_t)N * sizeof(float), s), "gelu_bwd_bias_grad");
    if (!A || !B || !D || !P || !workspace) return op_fail(GPT2_ERR_ARG, "gelu_bwd_bias_grad: null pointer");
    const size_t need = gpt2_op_matmul_gelu_bwd_bias_grad_workspace(M, N);
    if (workspace_bytes < need || ((uintptr_t)workspace & 7))
        return op_fail(GPT2_ERR_ARG, "gelu_bwd_bias_grad: workspace of %zu bytes (8-byte aligned) needed, %zu given",
                       need, workspace_bytes);
    GemmArgs a{};
    a.M = M; a.N = N; a.K = K; a.in_type = ACT_BF16;
    a.A = A;
    if (a_kmajor) { a.sAm = lda; a.sAk = 1; } else { a.sAm = 1; a.sAk = lda; }
    a.B = B;
    if (b_kmajor) { a.sBn = ldb; a.sBk = 1; } else { a.sBn = 1; a.sBk = ldb; }
    a.D = D; a.ldd = ldd; a.d_f32 = 0;
    a.P = P; a.ldp = ldp;
    a.epi = EPI_GELU_BWD;
    a.colsum_part = (float*)workspace;
    if (!gemm_tc_path(a)) return op_fail(GPT2_ERR_ARG, "gelu_bwd_bias_grad: layout or alignment outside the fused path");
    const bool fused = gemm_tc_fuses_colsum(a);
    if (!fused && ldd != N) return op_fail(GPT2_ERR_ARG, "gelu_bwd_bias_grad: odd N needs ldd == N");
    int rc = op_cuda(gemm_dispatch(a, nullptr, 0, s), "gelu_bwd_bias_grad");
    if (rc) return rc;
    if (fused) return op_cuda(colsum_reduce(dbias, (const float*)workspace, (M + 31) / 32, N, s), "gelu_bwd_bias_grad");
    return op_cuda(colsum(ACT_BF16, dbias, D, M, N, (float*)workspace, s), "gelu_bwd_bias_grad");
}

extern "C" int gpt2_op_adamw(float* p, const float* g, float* m, float* v, void* shadow, size_t n,
                             float lr, float b1, float b2, float eps, float wd, int t, void* stream) {
    if (t < 1) return op_fail(GPT2_ERR_ARG, "adamw: t must be >= 1 (got %d)", t);
    if (n && (!p || !g || !m || !v)) return op_fail(GPT2_ERR_ARG, "adamw: null pointer");
    if ((((uintptr_t)p | (uintptr_t)g | (uintptr_t)m | (uintptr_t)v) & 15) != 0)
        return op_fail(GPT2_ERR_ARG, "adamw: p, g, m, v must be 16-byte aligned");
    float c1 = 1.0f - powf(b1, (float)t), c2 = 1.0f - powf(b2, (float)t);
    return op_cuda(adamw(p, g, m, v, (bf16*)shadow, n, lr, b1, b2, eps, wd, c1, c2,
                         (cudaStream_t)stream), "adamw");
}

extern "C" int gpt2_op_attention_forward(int dtype, void* out, float* lse, const void* qkv, int B,
                                         int T, int C, int NH, void* stream) {
    if (!dtype_ok(dtype)) return op_fail(GPT2_ERR_ARG, "attention: bad dtype %d", dtype);
    if (B < 0 || T < 0 || C <= 0 || NH <= 0 || C % NH)
        return op_fail(GPT2_ERR_ARG, "attention: bad shape");
    if ((size_t)B * T == 0) return GPT2_OK;
    if (!out || !lse || !qkv) return op_fail(GPT2_ERR_ARG, "attention: null pointer");
    return op_cuda(attention_forward(act_of(dtype), out, lse, qkv, B, T, C, NH, (cudaStream_t)stream),
                   "attention_forward");
}

extern "C" int gpt2_op_attention_backward(int dtype, void* dqkv, const void* dout, const void* qkv,
                                          const void* out, const float* lse, int B, int T, int C,
                                          int NH, float* workspace, void* stream) {
    if (!dtype_ok(dtype)) return op_fail(GPT2_ERR_ARG, "attention: bad dtype %d", dtype);
    if (B < 0 || T < 0 || C <= 0 || NH <= 0 || C % NH)
        return op_fail(GPT2_ERR_ARG, "attention: bad shape");
    if ((size_t)B * T == 0) return GPT2_OK;
    if (!dqkv || !dout || !qkv || !out || !lse || !workspace)
        return op_fail(GPT2_ERR_ARG, "attention: null pointer");
    return op_cuda(attention_backward(act_of(dtype), dqkv, dout, qkv, out, lse, B, T, C, NH, workspace,
                                      (cudaStream_t)stream), "attention_backward");
}

extern "C" int gpt2_op_layernorm_forward(int dtype, void* out, float* mean, float* rstd, const void* inp,
                                         const float* w, const float* b, int M, int C, void* stream) {
    if (!dtype_ok(dtype)) return op_fail(GPT2_ERR_ARG, "layernorm: bad dtype %d", dtype);
    if (M < 0 || C <= 0) return op_fail(GPT2_ERR_ARG, "layernorm: bad shape M=%d C=%d", M, C);
    if (M == 0) return GPT2_OK;
    if (!out || !mean || !rstd || !inp || !w || !b) return op_fail(GPT2_ERR_ARG, "layernorm: null pointer");
    return op_cuda(layernorm_forward(act_of(dtype), out, mean, rstd, inp, w, b, M, C, NORM_LAYER,
                                     (cudaStream_t)stream),
                   "layernorm_forward");
}

extern "C" int gpt2_op_rmsnorm_forward(int dtype, void* out, float* rstd, const void* inp, const float* w, int M,
                                       int C, void* stream) {
    if (!dtype_ok(dtype)) return op_fail(GPT2_ERR_ARG, "rmsnorm: bad dtype %d", dtype);
    if (M < 0 || C <= 0) return op_fail(GPT2_ERR_ARG, "rmsnorm: bad shape M=%d C=%d", M, C);
    if (M == 0) return GPT2_OK;
    if (!out || !rstd || !inp || !w) return op_fail(GPT2_ERR_ARG, "rmsnorm: null pointer");
    return op_cuda(layernorm_forward(act_of(dtype), out, nullptr, rstd, inp, w, nullptr, M, C, NORM_RMS,
                                     (cudaStream_t)stream),
                   "rmsnorm_forward");
}

extern "C" size_t gpt2_op_layernorm_backward_workspace(int C) {
    return C > 0 ? ln_bwd_partial_floats(C) * sizeof(float) : 0;
}

extern "C" size_t gpt2_op_rmsnorm_backward_workspace(int C) {
    return C > 0 ? (ln_bwd_partial_floats(C) + (size_t)C) * sizeof(float) : 0;
}

extern "C" int gpt2_op_layernorm_backward(int dtype, void* dinp, float* dw, float* db, const void* dout,
                                          const void* inp, const float* w, const float* mean,
                                          const float* rstd, int M, int C, void* workspace,
                                          size_t workspace_bytes, void* stream) {
    if (!dtype_ok(dtype)) return op_fail(GPT2_ERR_ARG, "layernorm_backward: bad dtype %d", dtype);
    if (M < 0 || C <= 0) return op_fail(GPT2_ERR_ARG, "layernorm_backward: bad shape M=%d C=%d", M, C);
    if (!dw || !db || !w || (M > 0 && (!dinp || !dout || !inp || !mean || !rstd)))
        return op_fail(GPT2_ERR_ARG, "layernorm_backward: null pointer");
    size_t need = gpt2_op_layernorm_backward_workspace(C);
    if (!workspace || workspace_bytes < need)
        return op_fail(GPT2_ERR_ARG, "layernorm_backward: workspace of %zu bytes needed, %zu given", need,
                       workspace_bytes);
    return op_cuda(layernorm_backward(act_of(dtype), dinp, dw, db, nullptr, dout, inp, w, mean, rstd, M, C,
                                      (float*)workspace, nullptr, NORM_LAYER, (cudaStream_t)stream),
                   "layernorm_backward");
}

extern "C" int gpt2_op_rmsnorm_backward(int dtype, void* dinp, float* dw, const void* dout, const void* inp,
                                        const float* w, const float* rstd, int M, int C, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    if (!dtype_ok(dtype)) return op_fail(GPT2_ERR_ARG, "rmsnorm_backward: bad dtype %d", dtype);
    if (M < 0 || C <= 0) return op_fail(GPT2_ERR_ARG, "rmsnorm_backward: bad shape M=%d C=%d", M, C);
    if (!dw || !w || (M > 0 && (!dinp || !dout || !inp || !rstd)))
        return op_fail(GPT2_ERR_ARG, "rmsnorm_backward: null pointer");
    // the shift's sums (all 0 for RMSNorm) land in the workspace tail, after the partials
    size_t need = gpt2_op_rmsnorm_backward_workspace(C);
    if (!workspace || workspace_bytes < need)
        return op_fail(GPT2_ERR_ARG, "rmsnorm_backward: workspace of %zu bytes needed, %zu given", need,
                       workspace_bytes);
    float* part = (float*)workspace;
    float* db_sink = part + ln_bwd_partial_floats(C);
    return op_cuda(layernorm_backward(act_of(dtype), dinp, dw, db_sink, nullptr, dout, inp, w, nullptr, rstd, M, C,
                                      part, nullptr, NORM_RMS, (cudaStream_t)stream),
                   "rmsnorm_backward");
}

extern "C" int gpt2_op_softmax_xent(int dtype, void* logits, float* losses, const int32_t* targets, int M,
                                    int V, int Vp, float dloss, int* flags, void* stream) {
    if (!dtype_ok(dtype)) return op_fail(GPT2_ERR_ARG, "softmax_xent: bad dtype %d", dtype);
    if (M < 0 || V <= 0 || Vp < V) return op_fail(GPT2_ERR_ARG, "softmax_xent: bad shape M=%d V=%d Vp=%d", M, V, Vp);
    if (M == 0) return GPT2_OK;
    if (!logits || !losses || !targets) return op_fail(GPT2_ERR_ARG, "softmax_xent: null pointer");
    cudaStream_t s = (cudaStream_t)stream;
    if (flags) {
        int rc = op_cuda(cudaMemsetAsync(flags, 0, sizeof(int), s), "softmax_xent");
        if (rc) return rc;
    }
    int scratch = 0;
    int rc = op_cuda(softmax_xent(act_of(dtype), logits, losses, targets, M, V, Vp, dloss,
                                  flags ? flags : nullptr, s),
                     "softmax_xent");
    if (rc || !flags) return rc;
    rc = op_cuda(cudaMemcpyAsync(&scratch, flags, sizeof(int), cudaMemcpyDeviceToHost, s), "softmax_xent");
    if (rc) return rc;
    rc = op_cuda(cudaStreamSynchronize(s), "softmax_xent");
    if (rc) return rc;
    if (scratch) return op_fail(GPT2_ERR_TOKEN, "softmax_xent: a target id is outside [0, %d)", V);
    return GPT2_OK;
}

extern "C" int gpt2_op_encoder_forward(int dtype, void* out, const int32_t* tokens, const void* wte, const void* wpe,
                                       int B, int T, int C, int V, int* flags, void* stream) {
    if (!dtype_ok(dtype)) return op_fail(GPT2_ERR_ARG, "encoder_forward: bad dtype %d", dtype);
    if (B < 0 || T < 0 || C <= 0 || V <= 0) return op_fail(GPT2_ERR_ARG, "encoder_forward: bad shape");
    if ((size_t)B * T == 0) return GPT2_OK;
    if (!out || !tokens || !wte || !wpe || !flags) return op_fail(GPT2_ERR_ARG, "encoder_forward: null pointer");
    return op_cuda(encoder_forward(act_of(dtype), out, tokens, wte, wpe, B, T, C, V, flags, (cudaStream_t)stream),
                   "encoder_forward");
}

extern "C" size_t gpt2_op_encoder_backward_workspace(int M, int V, int C) {
    if (M < 0 || V <= 0 || C <= 0) return 0;
    return encoder_bwd_scratch_bytes(M, V, C);
}

extern "C" int gpt2_op_encoder_backward(int dtype, float* dwte, float* dwpe, const void* dout, const int32_t* tokens,
                                        int B, int T, int C, int V, int maxT, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    if (!dtype_ok(dtype)) return op_fail(GPT2_ERR_ARG, "encoder_backward: bad dtype %d", dtype);
    if (B < 0 || T < 0 || C <= 0 || V <= 0 || T > maxT)
        return op_fail(GPT2_ERR_ARG, "encoder_backward: bad shape");
    if (!dwte || !dwpe) return op_fail(GPT2_ERR_ARG, "encoder_backward: null pointer");
    const int M = B * T;
    if (M > 0 && (!dout || !tokens)) return op_fail(GPT2_ERR_ARG, "encoder_backward: null pointer");
    const size_t need = gpt2_op_encoder_backward_workspace(M, V, C);
    if (!workspace || workspace_bytes < need)
        return op_fail(GPT2_ERR_ARG, "encoder_backward: workspace of %zu bytes needed, %zu given", need,
                       workspace_bytes);
    if ((uintptr_t)workspace & 255) return op_fail(GPT2_ERR_ARG, "encoder_backward: workspace must be 256-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    int rc = op_cuda(encoder_backward_wpe(act_of(dtype), dwpe, dout, B, T, C, maxT, s), "encoder_backward");
    if (rc) return rc;
    EncoderBwdScratch sc;
    encoder_bwd_scratch_carve(&sc, workspace, M, V, C);
    return op_cuda(encoder_backward_wte(act_of(dtype), dwte, dout, tokens, M, C, V, &sc, s), "encoder_backward");
}

extern "C" int gpt2_op_gemm_force_tile_rows(int rows) { return gemm_tc_force_tile_rows(rows); }

extern "C" const char* gpt2_op_gemm_last_variant(void) {
    static thread_local char buf[128];
    gemm_tc_last_variant(buf, sizeof buf);
    return buf;
}

// Sets the message returned by gpt2_op_last_error (for entry points in other files).
void g2_op_set_error(const char* msg) {
    std::lock_guard<std::mutex> lk(g_op_err_mu);
    g_op_err = msg;
}
