// Host driver of the GPT-2 training step: arenas, the launch sequence of forward,
// backward and AdamW, and the C ABI of include/gpt2.h.
//
// The layer chain is the one of the llm.c annotated listing (gpt2_forward §1.23,
// gpt2_backward §1.25, gpt2_update §1.26) with these B300 choices:
//  * one parameter arena (params | grads | m | v | bf16 weight copy), one activation
//    arena sized at the first forward, nothing allocated afterwards;
//  * residual additions fused into the epilogue of the projection GEMMs, GELU fused
//    into the FC GEMM epilogue and its derivative into the FC-proj dgrad epilogue;
//  * attention keeps only the per-row log-sum-exp (no (T,T) matrices);
//  * softmax and cross-entropy fused, dlogits written over the logits in place.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/gpt2.h"
#include "common.cuh"
#include "dispatch.h"
#include "gemm_tc.h"
#include "kernels.h"

namespace g2 {
bool pdl_enabled() {
    static const bool on = [] {
        const char* v = getenv("G2_PDL");
        return v && v[0] == '1';
    }();
    return on;
}
static std::atomic<uint64_t> g_launches{0};
void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
uint64_t launches_total() { return g_launches.load(std::memory_order_relaxed); }
}  // namespace g2

using namespace g2;

static std::string g_build_error;

enum { NP = 16 };

struct gpt2 {
    int L, C, NH, V, Vp, maxT, prec;
    ActType at;
    NormKind nk;  // LayerNorm (GPT-2) or RMSNorm (the microGPT variant)
    size_t esz;  // bytes per activation element
    size_t psize[NP], poff[NP];  // padded sizes / offsets (elements)
    size_t npad, nreal;
    void* parena;
    size_t pbytes;
    float *params, *grads, *mom1, *mom2;
    bf16* shadow;
    bool opt_init, have_grads, fwd_targets, loss_valid;
    // activation arena
    void* aarena;
    size_t abytes;
    int B, T;
    int32_t *tok, *tgt;
    int* flags;   // [0]: bad ids / non-finite loss of the current forward (cleared by each forward)
    int* tflags;  // G2_FLAG_TIMEOUT of any kernel since it was last reported (kept until reported)
    float *loss, *losses;
    char *res, *res2, *ln1, *qkv, *atty, *ln2, *fch, *fchg, *lnf, *logits;
    float *ln1_mean, *ln1_rstd, *ln2_mean, *ln2_rstd, *lnf_mean, *lnf_rstd, *lse;
    char *dres, *dln, *datty, *dqkv, *dfch;
    float *attD, *ln_part, *cs_part, *gemm_ws;
    size_t gemm_ws_bytes;
    float* tf32_ws;  // GPT2_TF32: K-major copies of the products' M/N-major operands
    size_t tf32_ws_bytes;
    EncoderBwdScratch enc;
    bool logits_valid;
    // per-kernel-class timing (gpt2_profile_*): one event pair per launched op
    bool prof_on;
    std::vector<cudaEvent_t> ev_a, ev_b;
    std::vector<int> ev_cls;
    std::vector<double> ev_work;
    size_t ev_used;
    double prof_ms[GPT2_K_COUNT], prof_work[GPT2_K_COUNT];
    uint64_t prof_calls[GPT2_K_COUNT];
    // generation (gpt2_generate): key/value cache of gB sequences of up to maxT positions
    // and the working rows of one extend step (up to gB*maxT rows for a prompt)
    void* garena;
    size_t gbytes;
    int gB;
    char *g_kv, *g_x, *g_x2, *g_ln, *g_qkv, *g_atty, *g_fch, *g_fchg, *g_last, *g_lnl, *g_logits;
    float *g_mean, *g_rstd, *g_coins, *g_ws;
    size_t g_ws_bytes;
    int32_t *g_ids, *g_out;
    int *g_flags, *g_state;
    bool gen_logits_valid;
    cudaStream_t g_stream;       // generation runs here (graph capture needs a non-legacy stream)
    cudaEvent_t g_ev;
    cudaGraphExec_t g_step;      // captured one-token step (position read from g_state)
    unsigned g_step_launches;    // kernels in it
    cudaStream_t stream;
    int status;
    std::string err;
};

// ------------------------------------------------------------------ helpers
static int fail(gpt2* m, int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (m) {
        m->status = code;
        m->err = buf;
    }
    return code;
}

#define CK(expr)                                                                          \
    do {                                                                                  \
        cudaError_t e_ = (expr);                                                          \
        if (e_ != cudaSuccess)                                                            \
            return fail(m, GPT2_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_)); \
    } while (0)

// Runs one op; with profiling on, brackets it with a CUDA event pair on the stream and
// books its algorithmic work (FLOPs or bytes) to kernel class `cls`.
static int prof_begin(gpt2* m, int cls, double work) {
    if (!m->prof_on) return -1;
    if (m->ev_used == m->ev_a.size()) {
        cudaEvent_t a, b;
        if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) return -1;
        m->ev_a.push_back(a);
        m->ev_b.push_back(b);
        m->ev_cls.push_back(0);
        m->ev_work.push_back(0);
    }
    size_t i = m->ev_used++;
    m->ev_cls[i] = cls;
    m->ev_work[i] = work;
    cudaEventRecord(m->ev_a[i], m->stream);
    return (int)i;
}
static void prof_end(gpt2* m, int i) {
    if (i >= 0) cudaEventRecord(m->ev_b[i], m->stream);
}
#define OP(cls, work, expr)                      \
    do {                                         \
        int pi_ = prof_begin(m, (cls), (work));  \
        CK(expr);                                \
        prof_end(m, pi_);                        \
    } while (0)

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// pointers into the parameter-shaped buffers
enum { P_WTE, P_WPE, P_LN1W, P_LN1B, P_QKVW, P_QKVB, P_APW, P_APB, P_LN2W, P_LN2B, P_FCW, P_FCB,
       P_FPW, P_FPB, P_LNFW, P_LNFB };

static float* pf(const gpt2* m, float* base, int t) { return base + m->poff[t]; }
// weight operand of a GEMM: bf16 copy in BF16 mode, the fp32 master otherwise
static const void* pw(const gpt2* m, int t, size_t elem_off) {
    if (m->at == ACT_BF16) return m->shadow + m->poff[t] + elem_off;
    return m->params + m->poff[t] + elem_off;
}
static char* act(const gpt2* m, char* base, size_t elems) { return base + elems * m->esz; }

// ------------------------------------------------------------------ GEMM dispatch
// TF32 mode: fp32 operands contracted on the tensor cores as TF32.
static void tf32_args(const gpt2* m, GemmArgs& a) {
    if (m->prec != GPT2_TF32) return;
    a.tf32 = 1;
    a.tws = m->tf32_ws;
    a.tws_bytes = m->tf32_ws_bytes;
}
// Y[M,N] = X[M,K] . W[N,K]^T (+bias) (+R) with optional GELU epilogue.
static cudaError_t gemm_fwd(gpt2* m, int M, int N, int K, const void* X, const void* W,
                            const float* bias, void* Y, const void* R, void* Y2) {
    GemmArgs a{};
    a.M = M; a.N = N; a.K = K; a.in_type = m->at;
    a.A = X; a.sAm = K; a.sAk = 1;
    a.B = W; a.sBn = K; a.sBk = 1;
    a.D = Y; a.ldd = N; a.d_f32 = 0;
    a.bias = bias; a.R = R; a.ldr = N;
    a.D2 = Y2; a.ldd2 = N;
    a.epi = Y2 ? EPI_GELU : EPI_STORE;
    a.flags = m->tflags;
    tf32_args(m, a);
    return gemm_dispatch(a, m->gemm_ws, m->gemm_ws_bytes, m->stream);
}
// dX[M,K] = dY[M,N] . W[N,K]  (optionally times gelu'(P)).  With cs_part, *cs_fused
// tells whether the product's epilogue also wrote the per-32-row column sums of dX there
// (the bias gradient's first pass).
static cudaError_t gemm_dgrad(gpt2* m, int M, int N, int K, const void* dY, const void* W, void* dX,
                              const void* P, float* cs_part = nullptr, bool* cs_fused = nullptr) {
    GemmArgs a{};
    a.M = M; a.N = K; a.K = N; a.in_type = m->at;
    a.A = dY; a.sAm = N; a.sAk = 1;
    a.B = W; a.sBn = 1; a.sBk = K;
    a.D = dX; a.ldd = K; a.d_f32 = 0;
    a.P = P; a.ldp = K;
    a.epi = P ? EPI_GELU_BWD : EPI_STORE;
    a.flags = m->tflags;
    a.colsum_part = cs_part;
    tf32_args(m, a);
    if (cs_fused) *cs_fused = cs_part && gemm_tc_fuses_colsum(a);
    return gemm_dispatch(a, m->gemm_ws, m->gemm_ws_bytes, m->stream);
}
// dW[N,K] (fp32, overwritten) = dY[M,N]^T . X[M,K]
static cudaError_t gemm_wgrad(gpt2* m, int M, int N, int K, const void* dY, const void* X, float* dW) {
    GemmArgs a{};
    a.M = N; a.N = K; a.K = M; a.in_type = m->at;
    a.A = dY; a.sAm = 1; a.sAk = N;
    a.B = X; a.sBn = 1; a.sBk = K;
    a.D = dW; a.ldd = K; a.d_f32 = 1;
    a.epi = EPI_STORE;
    a.flags = m->tflags;
    tf32_args(m, a);
    return gemm_dispatch(a, m->gemm_ws, m->gemm_ws_bytes, m->stream);
}

// ------------------------------------------------------------------ build / free
extern "C" gpt2_t* gpt2_build_norm(int L, int C, int H, int V, int maxT, int precision, int norm, int* status) {
    auto bail = [&](int code, const char* msg) -> gpt2_t* {
        g_build_error = msg;
        if (status) *status = code;
        return nullptr;
    };
    if (L <= 0 || C <= 0 || H <= 0 || V <= 0 || maxT <= 0 || C % H)
        return bail(GPT2_ERR_ARG, "bad shape: need L,C,H,V,maxT > 0 and C % H == 0");
    if (precision != GPT2_FP32 && precision != GPT2_TF32 && precision != GPT2_BF16)
        return bail(GPT2_ERR_ARG, "precision must be GPT2_FP32, GPT2_TF32 or GPT2_BF16");
    if (norm != GPT2_LAYERNORM && norm != GPT2_RMSNORM)
        return bail(GPT2_ERR_ARG, "norm must be GPT2_LAYERNORM or GPT2_RMSNORM");
    if (C % 8) return bail(GPT2_ERR_ARG, "C must be a multiple of 8");
    if (C / H > 256) return bail(GPT2_ERR_ARG, "head size above 256 is not supported");
    gpt2* m = new (std::nothrow) gpt2();
    if (!m) return bail(GPT2_ERR_OOM, "host allocation failed");
    m->L = L; m->C = C; m->NH = H; m->V = V; m->maxT = maxT; m->prec = precision;
    m->nk = norm == GPT2_RMSNORM ? NORM_RMS : NORM_LAYER;
    m->Vp = (V + 127) / 128 * 128;
    m->at = precision == GPT2_BF16 ? ACT_BF16 : ACT_F32;
    m->esz = m->at == ACT_BF16 ? 2 : 4;
    size_t Ls = L, Cs = C;
    size_t sz[NP] = {(size_t)m->Vp * Cs, (size_t)maxT * Cs, Ls * Cs, Ls * Cs, Ls * 3 * Cs * Cs,
                     Ls * 3 * Cs, Ls * Cs * Cs, Ls * Cs, Ls * Cs, Ls * Cs, Ls * 4 * Cs * Cs,
                     Ls * 4 * Cs, Ls * Cs * 4 * Cs, Ls * Cs, Cs, Cs};
    size_t off = 0;
    for (int i = 0; i < NP; i++) {
        m->psize[i] = sz[i];
        m->poff[i] = off;
        off += sz[i];
    }
    m->npad = off;
    m->nreal = off - (size_t)(m->Vp - V) * Cs;
    size_t fbytes = align256(m->npad * 4);
    m->pbytes = 4 * fbytes + (m->at == ACT_BF16 ? align256(m->npad * 2) : 0);
    cudaStream_t s0 = nullptr;
    m->stream = s0;
    cudaError_t e = cudaMalloc(&m->parena, m->pbytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        char buf[256];
        snprintf(buf, sizeof buf, "cudaMalloc of %zu bytes failed: %s", m->pbytes, cudaGetErrorString(e));
        delete m;
        return bail(e == cudaErrorMemoryAllocation ? GPT2_ERR_OOM : GPT2_ERR_CUDA, buf);
    }
    char* p = (char*)m->parena;
    m->params = (float*)p; p += fbytes;
    m->grads = (float*)p; p += fbytes;
    m->mom1 = (float*)p; p += fbytes;
    m->mom2 = (float*)p; p += fbytes;
    m->shadow = m->at == ACT_BF16 ? (bf16*)p : nullptr;
    e = cudaMemset(m->parena, 0, m->pbytes);
    if (e != cudaSuccess) {
        cudaFree(m->parena);
        delete m;
        return bail(GPT2_ERR_CUDA, cudaGetErrorString(e));
    }
    if (status) *status = GPT2_OK;
    return m;
}

extern "C" gpt2_t* gpt2_build_ex(int L, int C, int H, int V, int maxT, int precision, int* status) {
    return gpt2_build_norm(L, C, H, V, maxT, precision, GPT2_LAYERNORM, status);
}

extern "C" gpt2_t* gpt2_build(int L, int C, int H, int V, int maxT) {
    return gpt2_build_ex(L, C, H, V, maxT, GPT2_BF16, nullptr);
}

extern "C" void gpt2_free(gpt2_t* m) {
    if (!m) return;
    if (m->parena) cudaFree(m->parena);
    if (m->aarena) cudaFree(m->aarena);
    if (m->garena) cudaFree(m->garena);
    if (m->g_step) cudaGraphExecDestroy(m->g_step);
    if (m->g_ev) cudaEventDestroy(m->g_ev);
    if (m->g_stream) cudaStreamDestroy(m->g_stream);
    for (size_t i = 0; i < m->ev_a.size(); i++) {
        cudaEventDestroy(m->ev_a[i]);
        cudaEventDestroy(m->ev_b[i]);
    }
    delete m;
}

extern "C" size_t gpt2_num_params(const gpt2_t* m) { return m ? m->nreal : 0; }
extern "C" int gpt2_padded_vocab(const gpt2_t* m) { return m ? m->Vp : 0; }
extern "C" size_t gpt2_device_bytes(const gpt2_t* m) { return m ? m->pbytes + m->abytes + m->gbytes : 0; }
extern "C" uint64_t gpt2_kernel_launches(const gpt2_t*) { return launches_total(); }
extern "C" int gpt2_last_status(const gpt2_t* m) { return m ? m->status : GPT2_ERR_ARG; }
extern "C" const char* gpt2_last_error(const gpt2_t* m) { return m ? m->err.c_str() : "null handle"; }
extern "C" const char* gpt2_last_build_error(void) { return g_build_error.c_str(); }

extern "C" int gpt2_set_stream(gpt2_t* m, void* stream) {
    if (!m) return GPT2_ERR_ARG;
    m->stream = (cudaStream_t)stream;
    return GPT2_OK;
}

extern "C" int gpt2_sync(gpt2_t* m) {
    if (!m) return GPT2_ERR_ARG;
    CK(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

// Host layout (real V rows of wte) <-> device layout (Vp rows): two copies.
static int copy_params(gpt2* m, float* dev, const float* hin, float* hout) {
    size_t real_wte = (size_t)m->V * m->C;
    size_t rest = m->nreal - real_wte;
    if (hin) {
        CK(cudaMemcpyAsync(dev, hin, real_wte * 4, cudaMemcpyHostToDevice, m->stream));
        CK(cudaMemcpyAsync(dev + m->poff[P_WPE], hin + real_wte, rest * 4, cudaMemcpyHostToDevice,
                           m->stream));
    } else {
        CK(cudaMemcpyAsync(hout, dev, real_wte * 4, cudaMemcpyDeviceToHost, m->stream));
        CK(cudaMemcpyAsync(hout + real_wte, dev + m->poff[P_WPE], rest * 4, cudaMemcpyDeviceToHost,
                           m->stream));
    }
    CK(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

extern "C" int gpt2_set_params(gpt2_t* m, const float* host, size_t n) {
    if (!m || !host) return fail(m, GPT2_ERR_ARG, "null argument");
    if (n != m->nreal) return fail(m, GPT2_ERR_ARG, "expected %zu parameters, got %zu", m->nreal, n);
    int rc = copy_params(m, m->params, host, nullptr);
    if (rc) return rc;
    if (m->shadow) {
        CK(cast_f32_to_bf16(m->shadow, m->params, m->npad, m->stream));
        CK(cudaStreamSynchronize(m->stream));
    }
    return GPT2_OK;
}

extern "C" int gpt2_init_params(gpt2_t* m, uint64_t seed) {
    if (!m) return GPT2_ERR_ARG;
    const size_t L = m->L, C = m->C;
    const double std = 0.02, proj_std = 0.02 / std::sqrt(2.0 * (double)L);
    CK(cudaMemsetAsync(m->params, 0, m->npad * 4, m->stream));
    InitPlan plan{};
    const int normal[] = {P_WTE, P_WPE, P_QKVW, P_APW, P_FCW, P_FPW};
    for (int t : normal) {
        const int k = plan.count++;
        plan.offset[k] = m->poff[t];
        plan.n[k] = t == P_WTE ? (size_t)m->V * C : m->psize[t];   // real rows only: the padding stays 0
        plan.std[k] = (t == P_APW || t == P_FPW) ? proj_std : std;
    }
    const float* ones[3] = {pf(m, m->params, P_LN1W), pf(m, m->params, P_LN2W), pf(m, m->params, P_LNFW)};
    const size_t ones_n[3] = {L * C, L * C, C};
    CK(init_params_device(m->params, plan, ones, ones_n, 3, seed, m->stream));
    if (m->shadow) CK(cast_f32_to_bf16(m->shadow, m->params, m->npad, m->stream));
    return GPT2_OK;
}

extern "C" int gpt2_get_params(gpt2_t* m, float* host, size_t n) {
    if (!m || !host) return fail(m, GPT2_ERR_ARG, "null argument");
    if (n != m->nreal) return fail(m, GPT2_ERR_ARG, "expected %zu parameters, got %zu", m->nreal, n);
    return copy_params(m, m->params, nullptr, host);
}

extern "C" int gpt2_get_grads(gpt2_t* m, float* host, size_t n) {
    if (!m || !host) return fail(m, GPT2_ERR_ARG, "null argument");
    if (n != m->nreal) return fail(m, GPT2_ERR_ARG, "expected %zu values, got %zu", m->nreal, n);
    if (!m->have_grads) return fail(m, GPT2_ERR_STATE, "no backward has run");
    return copy_params(m, m->grads, nullptr, host);
}

extern "C" int gpt2_get_opt_state(gpt2_t* m, float* mh, float* vh, size_t n) {
    if (!m || !mh || !vh) return fail(m, GPT2_ERR_ARG, "null argument");
    if (n != m->nreal) return fail(m, GPT2_ERR_ARG, "expected %zu values, got %zu", m->nreal, n);
    int rc = copy_params(m, m->mom1, nullptr, mh);
    return rc ? rc : copy_params(m, m->mom2, nullptr, vh);
}

// ------------------------------------------------------------------ activation arena
static int alloc_acts(gpt2* m, int B, int T) {
    const size_t M = (size_t)B * T, C = m->C, L = m->L, es = m->esz, NH = m->NH;
    struct Item { void** slot; size_t bytes; };
    void *tok, *tgt, *flags, *loss, *losses, *res, *res2, *ln1, *qkv, *atty, *ln2, *fch, *fchg, *lnf,
        *logits, *ln1m, *ln1r, *ln2m, *ln2r, *lnfm, *lnfr, *lse, *dres, *dln, *datty, *dqkv, *dfch,
        *attD, *lnp, *csp, *enc, *ws, *tws;
    size_t ln_part = ln_bwd_partial_floats(m->C) * 4;
    size_t maxN = std::max<size_t>(4 * C, (size_t)m->Vp);
    // column-sum partials: the bias-gradient pass's row blocks, or the GELU' product's
    // 32-row groups over the 4C hidden columns
    size_t cs_part = std::max(colsum_partial_floats((int)M, (int)maxN), (M + 31) / 32 * 4 * C) * 4;
    size_t enc_bytes = encoder_bwd_scratch_bytes((int)M, m->V, m->C);
    m->gemm_ws_bytes = gemm_workspace_bytes((int)M, m->C, m->Vp, m->L);
    // TF32: the largest set of operand copies of one product (the LM-head weight gradient
    // packs dlogits^T and lnf^T; the input gradients pack a weight matrix)
    m->tf32_ws_bytes = 0;
    if (m->prec == GPT2_TF32) {
        const int Mi = (int)M, Ci = m->C;
        const int shapes[][2] = {{3 * Ci, Ci}, {Ci, Ci}, {4 * Ci, Ci}, {Ci, 4 * Ci}, {m->Vp, Ci}};
        for (auto& sh : shapes) {  // (out, in) of a linear layer
            m->tf32_ws_bytes = std::max(m->tf32_ws_bytes, gemm_tf32_pack_bytes(Mi, sh[1], sh[0], true, false));
            m->tf32_ws_bytes = std::max(m->tf32_ws_bytes, gemm_tf32_pack_bytes(sh[0], sh[1], Mi, false, false));
        }
    }
    Item items[] = {
        {&tok, M * 4}, {&tgt, M * 4}, {&flags, 64}, {&loss, 64}, {&losses, M * 4},
        {&res, (L + 1) * M * C * es}, {&res2, L * M * C * es}, {&ln1, L * M * C * es},
        {&qkv, L * M * 3 * C * es}, {&atty, L * M * C * es}, {&ln2, L * M * C * es},
        {&fch, L * M * 4 * C * es}, {&fchg, L * M * 4 * C * es}, {&lnf, M * C * es},
        {&logits, M * (size_t)m->Vp * es}, {&ln1m, L * M * 4}, {&ln1r, L * M * 4},
        {&ln2m, L * M * 4}, {&ln2r, L * M * 4}, {&lnfm, M * 4}, {&lnfr, M * 4},
        {&lse, L * M * NH * 4}, {&dres, M * C * es}, {&dln, M * C * es}, {&datty, M * C * es},
        {&dqkv, M * 3 * C * es}, {&dfch, M * 4 * C * es}, {&attD, M * NH * 4}, {&lnp, ln_part},
        {&csp, cs_part}, {&enc, enc_bytes}, {&ws, m->gemm_ws_bytes}, {&tws, m->tf32_ws_bytes},
    };
    size_t total = 0;
    for (auto& it : items) total += align256(it.bytes);
    void* base = nullptr;
    cudaError_t e = cudaMalloc(&base, total);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(m, e == cudaErrorMemoryAllocation ? GPT2_ERR_OOM : GPT2_ERR_CUDA,
                    "activation arena of %zu bytes: %s", total, cudaGetErrorString(e));
    }
    char* p = (char*)base;
    for (auto& it : items) {
        *it.slot = p;
        p += align256(it.bytes);
    }
    m->aarena = base;
    m->abytes = total;
    m->B = B; m->T = T;
    m->tok = (int32_t*)tok; m->tgt = (int32_t*)tgt; m->flags = (int*)flags; m->tflags = (int*)flags + 1;
    m->loss = (float*)loss; m->losses = (float*)losses;
    m->res = (char*)res; m->res2 = (char*)res2; m->ln1 = (char*)ln1; m->qkv = (char*)qkv;
    m->atty = (char*)atty; m->ln2 = (char*)ln2; m->fch = (char*)fch; m->fchg = (char*)fchg;
    m->lnf = (char*)lnf; m->logits = (char*)logits;
    m->ln1_mean = (float*)ln1m; m->ln1_rstd = (float*)ln1r; m->ln2_mean = (float*)ln2m;
    m->ln2_rstd = (float*)ln2r; m->lnf_mean = (float*)lnfm; m->lnf_rstd = (float*)lnfr;
    m->lse = (float*)lse;
    m->dres = (char*)dres; m->dln = (char*)dln; m->datty = (char*)datty; m->dqkv = (char*)dqkv;
    m->dfch = (char*)dfch; m->attD = (float*)attD; m->ln_part = (float*)lnp;
    m->cs_part = (float*)csp; m->gemm_ws = (float*)ws;
    m->tf32_ws = m->tf32_ws_bytes ? (float*)tws : nullptr;
    encoder_bwd_scratch_carve(&m->enc, enc, (int)M, m->V, m->C);
    CK(cudaMemsetAsync(m->flags, 0, 64, m->stream));
    return GPT2_OK;
}

// ------------------------------------------------------------------ forward
// Algorithmic work of one op (booked to its class when profiling).
static double gemm_flops(size_t M, size_t N, size_t K) { return 2.0 * M * N * K; }
static double attn_fwd_flops(const gpt2* m) {
    // QK^T and PV over the causal triangle t2 <= t: 2 * 2 * hs * T(T+1)/2 per (b, h)
    return 2.0 * m->B * m->NH * (double)(m->C / m->NH) * m->T * (m->T + 1.0);
}

static int forward_impl(gpt2* m, const int32_t* tokens, const int32_t* targets, int B, int T,
                        int where) {
    if (!m || !tokens) return fail(m, GPT2_ERR_ARG, "null argument");
    if (B <= 0 || T <= 0) return fail(m, GPT2_ERR_ARG, "B and T must be positive");
    if (T > m->maxT) return fail(m, GPT2_ERR_SHAPE, "T=%d exceeds maxT=%d", T, m->maxT);
    if (!m->aarena) {
        int rc = alloc_acts(m, B, T);
        if (rc) return rc;
    } else if (B != m->B || T != m->T) {
        return fail(m, GPT2_ERR_SHAPE, "activations were allocated for B=%d T=%d, got B=%d T=%d",
                    m->B, m->T, B, T);
    }
    const int L = m->L, C = m->C, NH = m->NH, V = m->V, Vp = m->Vp;
    const size_t M = (size_t)B * T, MC = M * C;
    const double es = (double)m->esz, actMC = es * MC;
    cudaStream_t s = m->stream;
    cudaMemcpyKind kind = where == GPT2_DEVICE ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
    CK(cudaMemcpyAsync(m->tok, tokens, M * 4, kind, s));
    if (targets) CK(cudaMemcpyAsync(m->tgt, targets, M * 4, kind, s));
    CK(cudaMemsetAsync(m->flags, 0, sizeof(int), s));  // timeouts (tflags) stay until reported
    OP(GPT2_K_ENCODER, 4.0 * M, check_ids(m->tok, (int)M, V, m->flags, G2_FLAG_BAD_TOKEN, s));
    if (targets) OP(GPT2_K_ENCODER, 4.0 * M, check_ids(m->tgt, (int)M, V, m->flags, G2_FLAG_BAD_TARGET, s));
    // gathered token rows + position rows + output
    OP(GPT2_K_ENCODER, 2 * actMC + es * (double)T * C + 4.0 * M,
       encoder_forward(m->at, m->res, m->tok, pw(m, P_WTE, 0), pw(m, P_WPE, 0), B, T, C, V, m->flags, s));
    const double ln_fwd_bytes = 2 * actMC + 8.0 * M + 8.0 * C;
    for (int l = 0; l < L; l++) {
        char* res_in = act(m, m->res, l * MC);
        char* res_out = act(m, m->res, (l + 1) * MC);
        char* res2 = act(m, m->res2, l * MC);
        char* ln1 = act(m, m->ln1, l * MC);
        char* qkv = act(m, m->qkv, l * 3 * MC);
        char* atty = act(m, m->atty, l * MC);
        char* ln2 = act(m, m->ln2, l * MC);
        char* fch = act(m, m->fch, l * 4 * MC);
        char* fchg = act(m, m->fchg, l * 4 * MC);
        OP(GPT2_K_LAYERNORM, ln_fwd_bytes,
           layernorm_forward(m->at, ln1, m->ln1_mean + l * M, m->ln1_rstd + l * M, res_in,
                             pf(m, m->params, P_LN1W) + l * C, pf(m, m->params, P_LN1B) + l * C,
                             (int)M, C, m->nk, s));
        OP(GPT2_K_GEMM, gemm_flops(M, 3 * C, C),
           gemm_fwd(m, (int)M, 3 * C, C, ln1, pw(m, P_QKVW, (size_t)l * 3 * C * C),
                    pf(m, m->params, P_QKVB) + l * 3 * C, qkv, nullptr, nullptr));
        OP(GPT2_K_ATTN_FWD, attn_fwd_flops(m),
           attention_forward(m->at, atty, m->lse + l * M * NH, qkv, B, T, C, NH, s, m->tflags));
        OP(GPT2_K_GEMM, gemm_flops(M, C, C),
           gemm_fwd(m, (int)M, C, C, atty, pw(m, P_APW, (size_t)l * C * C),
                    pf(m, m->params, P_APB) + l * C, res2, res_in, nullptr));
        OP(GPT2_K_LAYERNORM, ln_fwd_bytes,
           layernorm_forward(m->at, ln2, m->ln2_mean + l * M, m->ln2_rstd + l * M, res2,
                             pf(m, m->params, P_LN2W) + l * C, pf(m, m->params, P_LN2B) + l * C,
                             (int)M, C, m->nk, s));
        OP(GPT2_K_GEMM, gemm_flops(M, 4 * C, C),
           gemm_fwd(m, (int)M, 4 * C, C, ln2, pw(m, P_FCW, (size_t)l * 4 * C * C),
                    pf(m, m->params, P_FCB) + l * 4 * C, fch, nullptr, fchg));
        OP(GPT2_K_GEMM, gemm_flops(M, C, 4 * C),
           gemm_fwd(m, (int)M, C, 4 * C, fchg, pw(m, P_FPW, (size_t)l * 4 * C * C),
                    pf(m, m->params, P_FPB) + l * C, res_out, res2, nullptr));
    }
    OP(GPT2_K_LAYERNORM, ln_fwd_bytes,
       layernorm_forward(m->at, m->lnf, m->lnf_mean, m->lnf_rstd, act(m, m->res, (size_t)L * MC),
                         pf(m, m->params, P_LNFW), pf(m, m->params, P_LNFB), (int)M, C, m->nk, s));
    OP(GPT2_K_GEMM, gemm_flops(M, Vp, C),
       gemm_fwd(m, (int)M, Vp, C, m->lnf, pw(m, P_WTE, 0), nullptr, m->logits, nullptr, nullptr));
    if (targets) {
        // read the logits once, write the gradient once, targets and per-row losses
        OP(GPT2_K_XENT, 2.0 * es * M * Vp + 8.0 * M,
           softmax_xent(m->at, m->logits, m->losses, m->tgt, (int)M, V, Vp, 1.0f / (float)M, m->flags, s));
        OP(GPT2_K_XENT, 4.0 * M, mean_fixed_order(m->loss, m->losses, (int)M, s));
        m->fwd_targets = true;
        m->loss_valid = true;
        m->logits_valid = false;
    } else {
        m->fwd_targets = false;
        m->loss_valid = false;
        m->logits_valid = true;
    }
    return GPT2_OK;
}

extern "C" int gpt2_forward_async(gpt2_t* m, const int32_t* tokens, const int32_t* targets, int B,
                                  int T, int where) {
    if (!m) return GPT2_ERR_ARG;
    m->status = GPT2_OK;
    return forward_impl(m, tokens, targets, B, T, where);
}

extern "C" int gpt2_read_loss(gpt2_t* m, float* out) {
    if (!m || !out) return fail(m, GPT2_ERR_ARG, "null argument");
    if (!m->aarena) return fail(m, GPT2_ERR_STATE, "no forward has run");
    int hflags[2] = {0, 0};
    float loss = -1.0f;
    if (m->loss_valid) CK(cudaMemcpyAsync(&loss, m->loss, 4, cudaMemcpyDeviceToHost, m->stream));
    CK(cudaMemcpyAsync(hflags, m->flags, 8, cudaMemcpyDeviceToHost, m->stream));
    CK(cudaStreamSynchronize(m->stream));
    *out = loss;
    if ((hflags[0] | hflags[1]) & G2_FLAG_TIMEOUT) {
        CK(cudaMemsetAsync(m->flags, 0, 8, m->stream));  // reported once
        return fail(m, GPT2_ERR_TIMEOUT, "a device-side wait gave up (kernel reported a timeout)");
    }
    if (hflags[0] & G2_FLAG_BAD_TOKEN)
        return fail(m, GPT2_ERR_TOKEN, "an input id is outside [0, %d)", m->V);
    if (hflags[0] & G2_FLAG_BAD_TARGET)
        return fail(m, GPT2_ERR_TOKEN, "a target id is outside [0, %d)", m->V);
    if (m->loss_valid && !std::isfinite(loss))
        return fail(m, GPT2_ERR_NONFINITE, "mean loss is not finite (%f)", loss);
    return GPT2_OK;
}

extern "C" float gpt2_forward(gpt2_t* m, const int32_t* tokens, const int32_t* targets, int B, int T) {
    if (!m) return NAN;
    m->status = GPT2_OK;
    int rc = forward_impl(m, tokens, targets, B, T, GPT2_HOST);
    if (rc) return NAN;
    float loss;
    rc = gpt2_read_loss(m, &loss);
    if (rc) {
        m->fwd_targets = false;  // a failed forward cannot feed a backward
        m->loss_valid = false;
        return NAN;
    }
    return loss;
}

// ------------------------------------------------------------------ backward
extern "C" int gpt2_backward(gpt2_t* m) {
    if (!m) return GPT2_ERR_ARG;
    if (!m->fwd_targets) return fail(m, GPT2_ERR_STATE, "backward needs a forward with targets first");
    const int L = m->L, C = m->C, NH = m->NH, V = m->V, Vp = m->Vp, B = m->B, T = m->T;
    const size_t M = (size_t)B * T, MC = M * C;
    const double es = (double)m->esz, actMC = es * MC;
    cudaStream_t s = m->stream;
    float* g = m->grads;
    // bias gradient: read the (M,N) gradient once, write N floats
    auto cs_bytes = [&](size_t N) { return es * M * N + 4.0 * N; };
    // layernorm backward: read dout, x, dres; write dres; stats
    const double ln_bwd_bytes = 4 * actMC + 8.0 * M + 16.0 * C;
    // vocab projection (tied): dlnf = dlogits . wte ; dwte = dlogits^T . lnf (overwrites)
    OP(GPT2_K_GEMM, gemm_flops(M, C, Vp), gemm_dgrad(m, (int)M, Vp, C, m->logits, pw(m, P_WTE, 0), m->dln, nullptr));
    OP(GPT2_K_GEMM, gemm_flops(Vp, C, M), gemm_wgrad(m, (int)M, Vp, C, m->logits, m->lnf, pf(m, g, P_WTE)));
    CK(cudaMemsetAsync(m->dres, 0, MC * m->esz, s));
    OP(GPT2_K_LAYERNORM, ln_bwd_bytes,
       layernorm_backward(m->at, m->dres, pf(m, g, P_LNFW), pf(m, g, P_LNFB),
                          pf(m, g, P_FPB) + (size_t)(L - 1) * C,  // d res_out(L-1): fcproj bias
                          m->dln, act(m, m->res, (size_t)L * MC), pf(m, m->params, P_LNFW), m->lnf_mean,
                          m->lnf_rstd, (int)M, C, m->ln_part, m->cs_part, m->nk, s));
    for (int l = L - 1; l >= 0; l--) {
        char* res_in = act(m, m->res, l * MC);
        char* res2 = act(m, m->res2, l * MC);
        char* ln1 = act(m, m->ln1, l * MC);
        char* qkv = act(m, m->qkv, l * 3 * MC);
        char* atty = act(m, m->atty, l * MC);
        char* ln2 = act(m, m->ln2, l * MC);
        char* fch = act(m, m->fch, l * 4 * MC);
        char* fchg = act(m, m->fchg, l * 4 * MC);
        // fcproj: res_out = fchg . Wfp^T + bfp + res2   (dres = d res_out)
        // (its epilogue also sums the columns of dfch per 32 rows: the fc bias gradient)
        bool fcb_fused = false;
        OP(GPT2_K_GEMM, gemm_flops(M, 4 * C, C),
           gemm_dgrad(m, (int)M, C, 4 * C, m->dres, pw(m, P_FPW, (size_t)l * 4 * C * C), m->dfch, fch,
                      m->cs_part, &fcb_fused));
        OP(GPT2_K_GEMM, gemm_flops(C, 4 * C, M),
           gemm_wgrad(m, (int)M, C, 4 * C, m->dres, fchg, pf(m, g, P_FPW) + (size_t)l * 4 * C * C));
        // (the fcproj bias gradient, the column sum of dres, came out of the layernorm
        // backward that produced dres)
        // fc: fch = ln2 . Wfc^T + bfc   (dfch already multiplied by gelu')
        OP(GPT2_K_GEMM, gemm_flops(M, C, 4 * C),
           gemm_dgrad(m, (int)M, 4 * C, C, m->dfch, pw(m, P_FCW, (size_t)l * 4 * C * C), m->dln, nullptr));
        OP(GPT2_K_GEMM, gemm_flops(4 * C, C, M),
           gemm_wgrad(m, (int)M, 4 * C, C, m->dfch, ln2, pf(m, g, P_FCW) + (size_t)l * 4 * C * C));
        if (fcb_fused)
            OP(GPT2_K_BIAS_GRAD, 4.0 * ((M + 31) / 32 + 1) * 4 * C,
               colsum_reduce(pf(m, g, P_FCB) + l * 4 * C, m->cs_part, (int)((M + 31) / 32), 4 * C, s));
        else
            OP(GPT2_K_BIAS_GRAD, cs_bytes(4 * C),
               colsum(m->at, pf(m, g, P_FCB) + l * 4 * C, m->dfch, (int)M, 4 * C, m->cs_part, s));
        // ln2 (dres becomes d res2)
        OP(GPT2_K_LAYERNORM, ln_bwd_bytes,
           layernorm_backward(m->at, m->dres, pf(m, g, P_LN2W) + l * C, pf(m, g, P_LN2B) + l * C,
                              pf(m, g, P_APB) + l * C,  // d res2: attproj bias
                              m->dln, res2, pf(m, m->params, P_LN2W) + l * C,
                              m->ln2_mean + l * M, m->ln2_rstd + l * M, (int)M, C, m->ln_part, m->cs_part, m->nk, s));
        // attproj: res2 = atty . Wap^T + bap + res_in
        OP(GPT2_K_GEMM, gemm_flops(M, C, C),
           gemm_dgrad(m, (int)M, C, C, m->dres, pw(m, P_APW, (size_t)l * C * C), m->datty, nullptr));
        OP(GPT2_K_GEMM, gemm_flops(C, C, M),
           gemm_wgrad(m, (int)M, C, C, m->dres, atty, pf(m, g, P_APW) + (size_t)l * C * C));
        // attention
        OP(GPT2_K_ATTN_BWD, 2.0 * attn_fwd_flops(m),
           attention_backward(m->at, m->dqkv, m->datty, qkv, atty, m->lse + l * M * NH, B, T, C, NH,
                              m->attD, s, m->tflags));
        // qkv: qkv = ln1 . Wqkv^T + bqkv
        OP(GPT2_K_GEMM, gemm_flops(M, C, 3 * C),
           gemm_dgrad(m, (int)M, 3 * C, C, m->dqkv, pw(m, P_QKVW, (size_t)l * 3 * C * C), m->dln, nullptr));
        OP(GPT2_K_GEMM, gemm_flops(3 * C, C, M),
           gemm_wgrad(m, (int)M, 3 * C, C, m->dqkv, ln1, pf(m, g, P_QKVW) + (size_t)l * 3 * C * C));
        OP(GPT2_K_BIAS_GRAD, cs_bytes(3 * C),
           colsum(m->at, pf(m, g, P_QKVB) + l * 3 * C, m->dqkv, (int)M, 3 * C, m->cs_part, s));
        // ln1 (dres becomes d res_in)
        OP(GPT2_K_LAYERNORM, ln_bwd_bytes,
           layernorm_backward(m->at, m->dres, pf(m, g, P_LN1W) + l * C, pf(m, g, P_LN1B) + l * C,
                              l > 0 ? pf(m, g, P_FPB) + (size_t)(l - 1) * C : nullptr,  // d res_out(l-1)
                              m->dln, res_in, pf(m, m->params, P_LN1W) + l * C,
                              m->ln1_mean + l * M, m->ln1_rstd + l * M, (int)M, C, m->ln_part, m->cs_part, m->nk, s));
    }
    OP(GPT2_K_ENCODER, actMC + 4.0 * m->maxT * C,
       encoder_backward_wpe(m->at, pf(m, g, P_WPE), m->dres, B, T, C, m->maxT, s));
    // read the gradient rows once and the ids; read-modify-write of the touched wte rows
    OP(GPT2_K_ENCODER, actMC + 4.0 * M,
       encoder_backward_wte(m->at, pf(m, g, P_WTE), m->dres, m->tok, (int)M, C, V, &m->enc, s));
    m->fwd_targets = false;
    m->have_grads = true;
    return GPT2_OK;
}

extern "C" int gpt2_zero_grad(gpt2_t* m) {
    if (!m) return GPT2_ERR_ARG;
    CK(cudaMemsetAsync(m->grads, 0, m->npad * 4, m->stream));
    return GPT2_OK;
}

extern "C" int gpt2_update(gpt2_t* m, float lr, float b1, float b2, float eps, float wd, int t) {
    if (!m) return GPT2_ERR_ARG;
    if (t < 1) return fail(m, GPT2_ERR_ARG, "t must be >= 1 (got %d)", t);
    if (!m->have_grads) return fail(m, GPT2_ERR_STATE, "update needs gradients (run backward)");
    float c1 = 1.0f - powf(b1, (float)t), c2 = 1.0f - powf(b2, (float)t);
    // read p, g, m, v; write p, m, v (fp32) and the bf16 weight copy
    double bytes = (double)m->npad * (28.0 + (m->shadow ? 2.0 : 0.0));
    OP(GPT2_K_ADAMW, bytes,
       adamw(m->params, m->grads, m->mom1, m->mom2, m->shadow, m->npad, lr, b1, b2, eps, wd, c1, c2,
             m->stream));
    return GPT2_OK;
}

// ------------------------------------------------------------------ diagnostics
extern "C" int gpt2_check_bounded_wait(gpt2_t* m, unsigned timeout_us) {
    if (!m) return GPT2_ERR_ARG;
    if (!m->aarena) return fail(m, GPT2_ERR_STATE, "the check uses the activation arena's flags: run a forward first");
    if (timeout_us < 1 || timeout_us > 1000000) return fail(m, GPT2_ERR_ARG, "timeout_us must be in [1, 1e6]");
    int hflag = 0;
    CK(cudaMemsetAsync(m->tflags, 0, sizeof(int), m->stream));
    CK(bounded_wait_check(m->tflags, 1000ull * timeout_us, m->stream));
    CK(cudaMemcpyAsync(&hflag, m->tflags, 4, cudaMemcpyDeviceToHost, m->stream));
    CK(cudaStreamSynchronize(m->stream));
    CK(cudaMemsetAsync(m->tflags, 0, sizeof(int), m->stream));  // reported here: the handle starts clean
    if (hflag & G2_FLAG_TIMEOUT)
        return fail(m, GPT2_ERR_TIMEOUT, "a device-side wait gave up (kernel reported a timeout)");
    return fail(m, GPT2_ERR_STATE, "the bounded wait did not report a timeout");
}

// ------------------------------------------------------------------ profiling
extern "C" int gpt2_profile_enable(gpt2_t* m, int on) {
    if (!m) return GPT2_ERR_ARG;
    m->prof_on = on != 0;
    return GPT2_OK;
}

extern "C" int gpt2_profile_reset(gpt2_t* m) {
    if (!m) return GPT2_ERR_ARG;
    CK(cudaStreamSynchronize(m->stream));
    m->ev_used = 0;
    for (int k = 0; k < GPT2_K_COUNT; k++) {
        m->prof_ms[k] = m->prof_work[k] = 0;
        m->prof_calls[k] = 0;
    }
    return GPT2_OK;
}

extern "C" int gpt2_profile_read(gpt2_t* m, int cls, double* ms, double* work, uint64_t* calls) {
    if (!m || cls < 0 || cls >= GPT2_K_COUNT) return fail(m, GPT2_ERR_ARG, "bad kernel class");
    CK(cudaStreamSynchronize(m->stream));
    for (size_t i = 0; i < m->ev_used; i++) {
        float t = 0;
        CK(cudaEventElapsedTime(&t, m->ev_a[i], m->ev_b[i]));
        m->prof_ms[m->ev_cls[i]] += t;
        m->prof_work[m->ev_cls[i]] += m->ev_work[i];
        m->prof_calls[m->ev_cls[i]] += 1;
    }
    m->ev_used = 0;
    if (ms) *ms = m->prof_ms[cls];
    if (work) *work = m->prof_work[cls];
    if (calls) *calls = m->prof_calls[cls];
    return GPT2_OK;
}

extern "C" int gpt2_get_losses(gpt2_t* m, float* host, size_t n) {
    if (!m || !host) return fail(m, GPT2_ERR_ARG, "null argument");
    if (!m->aarena) return fail(m, GPT2_ERR_STATE, "no forward has run");
    if (n != (size_t)m->B * m->T) return fail(m, GPT2_ERR_ARG, "expected %d values", m->B * m->T);
    CK(cudaMemcpyAsync(host, m->losses, n * 4, cudaMemcpyDeviceToHost, m->stream));
    CK(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

extern "C" int gpt2_get_logits(gpt2_t* m, float* host, size_t n) {
    if (!m || !host) return fail(m, GPT2_ERR_ARG, "null argument");
    if (!m->aarena || !m->logits_valid)
        return fail(m, GPT2_ERR_STATE, "logits are only kept by a forward without targets");
    const size_t M = (size_t)m->B * m->T;
    if (n != M * m->V) return fail(m, GPT2_ERR_ARG, "expected %zu values", M * m->V);
    if (m->at == ACT_F32) {
        CK(cudaMemcpy2DAsync(host, (size_t)m->V * 4, m->logits, (size_t)m->Vp * 4, (size_t)m->V * 4, M,
                             cudaMemcpyDeviceToHost, m->stream));
        CK(cudaStreamSynchronize(m->stream));
        return GPT2_OK;
    }
    // bf16: widen on the host, row by row, through a small staging buffer
    const size_t rows_per = 64;
    std::string stage(rows_per * m->Vp * 2, '\0');
    for (size_t r0 = 0; r0 < M; r0 += rows_per) {
        size_t nr = std::min(rows_per, M - r0);
        CK(cudaMemcpyAsync(&stage[0], m->logits + r0 * m->Vp * 2, nr * m->Vp * 2,
                           cudaMemcpyDeviceToHost, m->stream));
        CK(cudaStreamSynchronize(m->stream));
        const uint16_t* src = (const uint16_t*)stage.data();
        for (size_t r = 0; r < nr; r++)
            for (int c = 0; c < m->V; c++) {
                uint32_t bits = (uint32_t)src[r * m->Vp + c] << 16;
                float f;
                memcpy(&f, &bits, 4);
                host[(r0 + r) * m->V + c] = f;
            }
    }
    return GPT2_OK;
}

extern "C" int gpt2_get_ids(gpt2_t* m, int32_t* tok, int32_t* tgt, size_t n) {
    if (!m || !tok) return fail(m, GPT2_ERR_ARG, "null argument");
    if (!m->aarena) return fail(m, GPT2_ERR_STATE, "no forward has run");
    if (n != (size_t)m->B * m->T) return fail(m, GPT2_ERR_ARG, "expected %d values", m->B * m->T);
    CK(cudaMemcpyAsync(tok, m->tok, n * 4, cudaMemcpyDeviceToHost, m->stream));
    if (tgt) CK(cudaMemcpyAsync(tgt, m->tgt, n * 4, cudaMemcpyDeviceToHost, m->stream));
    CK(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

// ------------------------------------------------------------------ generation
// picoGPT "generate" with a key/value cache: the prompt runs as one extend step over
// positions 0..T0-1, every further token as an extend of one position; each step ends
// with the LM head on the last position of every sequence and the choice of the next id.
static int alloc_gen(gpt2* m, int B) {
    if (m->g_step) {
        cudaGraphExecDestroy(m->g_step);
        m->g_step = nullptr;
    }
    if (m->garena) {
        cudaFree(m->garena);
        m->garena = nullptr;
        m->gB = 0;
    }
    if (!m->g_stream) {
        CK(cudaStreamCreateWithFlags(&m->g_stream, cudaStreamNonBlocking));
        CK(cudaEventCreateWithFlags(&m->g_ev, cudaEventDisableTiming));
    }
    const size_t R = (size_t)B * m->maxT, C = m->C, L = m->L, es = m->esz;
    struct Item { void** slot; size_t bytes; };
    void *kv, *x, *x2, *ln, *qkv, *atty, *fch, *fchg, *last, *lnl, *logits, *mean, *rstd, *coins, *ids, *out, *flags,
        *ws, *state;
    // split-K partials of the one-token steps' products (B rows)
    size_t wsb = 256;
    const size_t shapes[][2] = {{3 * C, C}, {C, C}, {4 * C, C}, {C, 4 * C}, {(size_t)m->Vp, C}};
    for (auto& sh : shapes) wsb = std::max(wsb, gemm_tc_skinny_workspace_bytes(B, (int)sh[0], (int)sh[1]));
    Item items[] = {
        {&kv, L * R * 2 * C * es}, {&x, R * C * es}, {&x2, R * C * es}, {&ln, R * C * es}, {&qkv, R * 3 * C * es},
        {&atty, R * C * es}, {&fch, R * 4 * C * es}, {&fchg, R * 4 * C * es}, {&last, (size_t)B * C * es},
        {&lnl, (size_t)B * C * es}, {&logits, (size_t)B * m->Vp * es}, {&mean, R * 4}, {&rstd, R * 4},
        {&coins, (size_t)B * (m->maxT + 1) * 4}, {&ids, R * 4}, {&out, (size_t)B * (m->maxT + 1) * 4},
        {&flags, 64}, {&ws, wsb}, {&state, 64},
    };
    size_t total = 0;
    for (auto& it : items) total += align256(it.bytes);
    void* base = nullptr;
    cudaError_t e = cudaMalloc(&base, total);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(m, e == cudaErrorMemoryAllocation ? GPT2_ERR_OOM : GPT2_ERR_CUDA,
                    "generation arena of %zu bytes: %s", total, cudaGetErrorString(e));
    }
    char* p = (char*)base;
    for (auto& it : items) {
        *it.slot = p;
        p += align256(it.bytes);
    }
    m->garena = base;
    m->gbytes = total;
    m->gB = B;
    m->g_kv = (char*)kv; m->g_x = (char*)x; m->g_x2 = (char*)x2; m->g_ln = (char*)ln; m->g_qkv = (char*)qkv;
    m->g_atty = (char*)atty; m->g_fch = (char*)fch; m->g_fchg = (char*)fchg; m->g_last = (char*)last;
    m->g_lnl = (char*)lnl; m->g_logits = (char*)logits;
    m->g_mean = (float*)mean; m->g_rstd = (float*)rstd; m->g_coins = (float*)coins;
    m->g_ids = (int32_t*)ids; m->g_out = (int32_t*)out; m->g_flags = (int*)flags;
    m->g_ws = (float*)ws; m->g_ws_bytes = wsb;
    m->g_state = (int*)state;
    return GPT2_OK;
}

// Y[M,N] = X[M,K] . W[N,K]^T (+bias) (+R) (GELU epilogue with Y2), timeouts into the
// generation flags.  Products of at most one 128-row tile (the one-token steps) split K
// over the SMs and apply their epilogue in the fixed-order reduce.
static cudaError_t gen_gemm(gpt2* m, int M, int N, int K, const void* X, const void* W, const float* bias, void* Y,
                            const void* R, void* Y2, cudaStream_t s) {
    GemmArgs a{};
    a.M = M; a.N = N; a.K = K; a.in_type = m->at;
    a.A = X; a.sAm = K; a.sAk = 1;
    a.B = W; a.sBn = K; a.sBk = 1;
    a.D = Y; a.ldd = N; a.d_f32 = 0;
    a.bias = bias; a.R = R; a.ldr = N;
    a.D2 = Y2; a.ldd2 = N;
    a.epi = Y2 ? EPI_GELU : EPI_STORE;
    a.flags = m->g_flags;
    a.skinny_split = 1;
    return gemm_dispatch(a, m->g_ws, m->g_ws_bytes, s);
}

// Forward of positions t0..t0+n-1 of the gB sequences (ids already in g_ids); leaves
// the logits of each sequence's last new position in g_logits.  dstate: the position
// comes from device memory instead (one-token steps, n = 1).
static int gen_extend(gpt2* m, int t0, int n, const int* dstate, cudaStream_t s) {
    const int B = m->gB, L = m->L, C = m->C, NH = m->NH, maxT = m->maxT;
    const int rows = B * n;
    float* P = m->params;
    CK(gen_embed(m->at, m->g_x, m->g_ids, pw(m, P_WTE, 0), pw(m, P_WPE, 0), B, n, t0, maxT, C, dstate, s));
    for (int l = 0; l < L; l++) {
        char* kv = act(m, m->g_kv, (size_t)l * B * maxT * 2 * C);
        CK(layernorm_forward(m->at, m->g_ln, m->g_mean, m->g_rstd, m->g_x, pf(m, P, P_LN1W) + l * C,
                             pf(m, P, P_LN1B) + l * C, rows, C, m->nk, s));
        CK(gen_gemm(m, rows, 3 * C, C, m->g_ln, pw(m, P_QKVW, (size_t)l * 3 * C * C), pf(m, P, P_QKVB) + l * 3 * C,
                    m->g_qkv, nullptr, nullptr, s));
        CK(gen_kv_append(m->at, kv, m->g_qkv, B, n, t0, maxT, C, dstate, s));
        CK(gen_attention(m->at, m->g_atty, m->g_qkv, kv, B, n, t0, maxT, C, NH, dstate, s));
        CK(gen_gemm(m, rows, C, C, m->g_atty, pw(m, P_APW, (size_t)l * C * C), pf(m, P, P_APB) + l * C, m->g_x2,
                    m->g_x, nullptr, s));
        CK(layernorm_forward(m->at, m->g_ln, m->g_mean, m->g_rstd, m->g_x2, pf(m, P, P_LN2W) + l * C,
                             pf(m, P, P_LN2B) + l * C, rows, C, m->nk, s));
        CK(gen_gemm(m, rows, 4 * C, C, m->g_ln, pw(m, P_FCW, (size_t)l * 4 * C * C), pf(m, P, P_FCB) + l * 4 * C,
                    m->g_fch, nullptr, m->g_fchg, s));
        CK(gen_gemm(m, rows, C, 4 * C, m->g_fchg, pw(m, P_FPW, (size_t)l * 4 * C * C), pf(m, P, P_FPB) + l * C,
                    m->g_x, m->g_x2, nullptr, s));
    }
    CK(gen_last_rows(m->at, m->g_last, m->g_x, B, n, C, s));
    CK(layernorm_forward(m->at, m->g_lnl, m->g_mean, m->g_rstd, m->g_last, pf(m, P, P_LNFW), pf(m, P, P_LNFB), B, C,
                         m->nk, s));
    CK(gen_gemm(m, B, m->Vp, C, m->g_lnl, pw(m, P_WTE, 0), nullptr, m->g_logits, nullptr, nullptr, s));
    return GPT2_OK;
}

// One one-token step with its position in g_state: extend, choose, advance.
static int gen_token_step(gpt2* m, cudaStream_t s) {
    int rc = gen_extend(m, 0, 1, m->g_state, s);
    if (rc) return rc;
    CK(gen_sample(m->at, m->g_ids, m->g_out, m->g_logits, m->gB, m->V, m->Vp, 0.f, m->g_coins, 0, 0, 0, m->maxT,
                  m->g_state, s));
    CK(gen_advance(m->g_state, s));
    return GPT2_OK;
}

// Capture one one-token step into a CUDA graph (kept until the arena changes).
static int gen_capture(gpt2* m) {
    cudaStream_t s = m->g_stream;
    const uint64_t l0 = launches_total();
    CK(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
    int rc = gen_token_step(m, s);
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(s, &graph);
    if (rc) {
        if (graph) cudaGraphDestroy(graph);
        return rc;
    }
    CK(e);
    e = cudaGraphInstantiate(&m->g_step, graph, 0);
    cudaGraphDestroy(graph);
    CK(e);
    m->g_step_launches = (unsigned)(launches_total() - l0);
    return GPT2_OK;
}

extern "C" int gpt2_generate(gpt2_t* m, const int32_t* prompt, int B, int T0, int n_new, float temperature,
                             const float* coins, int32_t* out) {
    if (!m || !prompt || !out) return fail(m, GPT2_ERR_ARG, "null argument");
    if (B <= 0 || T0 <= 0 || n_new < 0) return fail(m, GPT2_ERR_ARG, "need B > 0, T0 > 0, n_new >= 0");
    if (!(temperature == temperature)) return fail(m, GPT2_ERR_ARG, "temperature is NaN");
    if ((long long)T0 + n_new - 1 > m->maxT)
        return fail(m, GPT2_ERR_SHAPE, "T0 + n_new - 1 = %lld exceeds maxT = %d", (long long)T0 + n_new - 1,
                    m->maxT);
    if (gen_attn_smem_bytes(m->C, m->NH, m->maxT) > 227 * 1024)
        return fail(m, GPT2_ERR_SHAPE, "maxT = %d is too long for the cached attention", m->maxT);
    for (size_t i = 0; i < (size_t)B * T0; i++)
        if (prompt[i] < 0 || prompt[i] >= m->V) return fail(m, GPT2_ERR_TOKEN, "prompt id %d outside [0, V)", prompt[i]);
    if (temperature > 0.f) {
        if (!coins) return fail(m, GPT2_ERR_ARG, "sampling (temperature > 0) needs coins");
        for (size_t i = 0; i < (size_t)B * n_new; i++)
            if (!(coins[i] >= 0.f && coins[i] < 1.f)) return fail(m, GPT2_ERR_ARG, "coins must lie in [0, 1)");
    }
    if (n_new == 0) return GPT2_OK;
    if (!m->garena || m->gB != B) {
        int rc = alloc_gen(m, B);
        if (rc) return rc;
    }
    const int maxT = m->maxT;
    cudaStream_t s = m->g_stream;
    m->gen_logits_valid = false;
    // after the work already queued on the handle's stream
    CK(cudaEventRecord(m->g_ev, m->stream));
    CK(cudaStreamWaitEvent(s, m->g_ev, 0));
    CK(cudaMemsetAsync(m->g_flags, 0, 64, s));
    CK(cudaMemcpy2DAsync(m->g_ids, (size_t)maxT * 4, prompt, (size_t)T0 * 4, (size_t)T0 * 4, B,
                         cudaMemcpyHostToDevice, s));
    if (temperature > 0.f)
        CK(cudaMemcpyAsync(m->g_coins, coins, (size_t)B * n_new * 4, cudaMemcpyHostToDevice, s));
    // the prompt: all T0 positions at once, then the first new id
    int rc = gen_extend(m, 0, T0, nullptr, s);
    if (rc) return rc;
    CK(gen_sample(m->at, m->g_ids, m->g_out, m->g_logits, B, m->V, m->Vp, temperature, m->g_coins, 0, n_new, T0, maxT,
                  nullptr, s));
    if (n_new > 1) {
        float tbits = temperature;
        int st[4] = {T0, 1, n_new, 0};
        memcpy(&st[3], &tbits, 4);
        CK(cudaMemcpyAsync(m->g_state, st, sizeof st, cudaMemcpyHostToDevice, s));
        CK(cudaStreamSynchronize(s));  // st leaves scope; also keeps capture off a busy stream
        int step = 1;
        if (!m->g_step) {
            // first time for this arena: one step launched directly (sets every kernel's
            // attributes), then the step captured for the rest
            rc = gen_token_step(m, s);
            if (rc) return rc;
            step++;
            if (step < n_new) {
                rc = gen_capture(m);
                if (rc) return rc;
            }
        }
        for (; step < n_new; step++) {
            CK(cudaGraphLaunch(m->g_step, s));
            count_launches(m->g_step_launches);
        }
    }
    int hflags[2] = {0, 0};
    CK(cudaMemcpyAsync(out, m->g_out, (size_t)B * n_new * 4, cudaMemcpyDeviceToHost, s));
    CK(cudaMemcpyAsync(hflags, m->g_flags, 4, cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
    if (hflags[0] & G2_FLAG_TIMEOUT)
        return fail(m, GPT2_ERR_TIMEOUT, "a device-side wait gave up (kernel reported a timeout)");
    m->gen_logits_valid = true;
    return GPT2_OK;
}

extern "C" int gpt2_get_gen_logits(gpt2_t* m, float* host, size_t n) {
    if (!m || !host) return fail(m, GPT2_ERR_ARG, "null argument");
    if (!m->garena || !m->gen_logits_valid) return fail(m, GPT2_ERR_STATE, "no generation has run");
    const size_t B = m->gB;
    if (n != B * m->V) return fail(m, GPT2_ERR_ARG, "expected %zu values", B * m->V);
    if (m->at == ACT_F32) {
        CK(cudaMemcpy2DAsync(host, (size_t)m->V * 4, m->g_logits, (size_t)m->Vp * 4, (size_t)m->V * 4, B,
                             cudaMemcpyDeviceToHost, m->g_stream));
        CK(cudaStreamSynchronize(m->g_stream));
        return GPT2_OK;
    }
    std::string stage(B * m->Vp * 2, '\0');
    CK(cudaMemcpyAsync(&stage[0], m->g_logits, B * m->Vp * 2, cudaMemcpyDeviceToHost, m->g_stream));
    CK(cudaStreamSynchronize(m->g_stream));
    const uint16_t* src = (const uint16_t*)stage.data();
    for (size_t r = 0; r < B; r++)
        for (int c = 0; c < m->V; c++) {
            uint32_t bits = (uint32_t)src[r * m->Vp + c] << 16;
            float f;
            memcpy(&f, &bits, 4);
            host[r * m->V + c] = f;
        }
    return GPT2_OK;
}
