/*
 * CPU oracle for one GPT-2 training step (forward, backward, AdamW).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code with the CUDA library.
 *
 * Source of truth: the llm.c listing on the page "llm.c 的中文注解-20240421"
 * (sections 1.1-1.27, cited below as "llm.c §x.y"), with picoGPT's NumPy
 * statement ("60 行 NumPy 代码 ... 实现一个 GPT", functions gelu, softmax,
 * layer_norm, attention, mha, gpt2, lm_loss) as the second statement of the
 * forward and the loss.  The microGPT variant (page "microGPT 3D", lesson 04)
 * swaps every LayerNorm for RMSNorm (or_rmsnorm_forward/backward, or_build_ex).  Every function below restates what the listing
 * computes, loop by loop, in the order the listing uses; nothing is blocked,
 * fused or reordered, except that loops over independent (b, h) pairs run under
 * OpenMP where the sum order of every output element is unchanged.
 *
 * `real` is double by default (the truth for parity) and float when compiled
 * with -DORACLE_REAL_FLOAT (the listing's own precision, used for drift studies
 * over many AdamW steps).  Build without -ffast-math: the listing notes that
 * fast-math breaks the GELU backward (llm.c §1.10).
 *
 * Readings where the pages are silent or loose (each also listed in the design
 * notes of the repository):
 *  - softmax / attention maxima start at -infinity instead of the listing's
 *    -10000 placeholder (marked "TODO something better" there); identical
 *    whenever any score exceeds -10000.
 *  - the loss uses the real vocabulary V only; the CUDA library may pad the
 *    vocabulary internally but this oracle never does.
 *  - errors return codes instead of exit()/assert() (llm.c §1.22, §1.23, §1.25).
 *
 * Parity pins: see tests/test_oracle_pins.py (worked values from the picoGPT
 * page, closed forms, finite differences, invariances).  No function here is
 * unpinned.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifdef ORACLE_REAL_FLOAT
typedef float real;
#define R_EXP expf
#define R_LOG logf
#define R_SQRT sqrtf
#define R_TANH tanhf
#define R_COSH coshf
#define R_POW powf
#else
typedef double real;
#define R_EXP exp
#define R_LOG log
#define R_SQRT sqrt
#define R_TANH tanh
#define R_COSH cosh
#define R_POW pow
#endif

#define OR_EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------------- */
/* per-layer primitives                                                       */
/* ------------------------------------------------------------------------- */

/* llm.c §1.1 encoder_forward; picoGPT gpt2(): wte[inputs] + wpe[range(n)].
 * out (B,T,C) = token row + position row. */
OR_EXPORT void or_encoder_forward(real* out, const int* inp, const real* wte, const real* wpe,
                                  int B, int T, int C) {
    for (int b = 0; b < B; b++) {
        for (int t = 0; t < T; t++) {
            const real* tok_row = wte + (size_t)inp[b * T + t] * C;
            const real* pos_row = wpe + (size_t)t * C;
            real* o = out + ((size_t)b * T + t) * C;
            for (int c = 0; c < C; c++) o[c] = tok_row[c] + pos_row[c];
        }
    }
}

/* llm.c §1.2 encoder_backward: the gradient at (b,t) is added into the token's
 * row of dwte and the position's row of dwpe, visiting (b,t) in row-major order. */
OR_EXPORT void or_encoder_backward(real* dwte, real* dwpe, const real* dout, const int* inp,
                                   int B, int T, int C) {
    for (int b = 0; b < B; b++) {
        for (int t = 0; t < T; t++) {
            const real* d = dout + ((size_t)b * T + t) * C;
            real* gt = dwte + (size_t)inp[b * T + t] * C;
            real* gp = dwpe + (size_t)t * C;
            for (int c = 0; c < C; c++) {
                gt[c] += d[c];
                gp[c] += d[c];
            }
        }
    }
}

/* llm.c §1.3 layernorm_forward; picoGPT layer_norm(eps=1e-5).
 * Per position: mean, biased variance (divide by C), rstd = 1/sqrt(var+1e-5),
 * out = (x-mean)*rstd*w + b.  mean and rstd are kept for the backward. */
OR_EXPORT void or_layernorm_forward(real* out, real* mean, real* rstd, const real* inp,
                                    const real* w, const real* bias, int B, int T, int C) {
    const real eps = (real)1e-5;
    for (int bt = 0; bt < B * T; bt++) {
        const real* x = inp + (size_t)bt * C;
        real m = 0;
        for (int c = 0; c < C; c++) m += x[c];
        m = m / C;
        real v = 0;
        for (int c = 0; c < C; c++) {
            real d = x[c] - m;
            v += d * d;
        }
        v = v / C;
        real s = (real)1 / R_SQRT(v + eps);
        real* o = out + (size_t)bt * C;
        for (int c = 0; c < C; c++) o[c] = (s * (x[c] - m)) * w[c] + bias[c];
        mean[bt] = m;
        rstd[bt] = s;
    }
}

/* llm.c §1.4 layernorm_backward.  With n = (x-mean)*rstd and g = w*dout:
 *   dbias += dout, dw += n*dout,
 *   dinp  += (g - mean(g) - n*mean(g*n)) * rstd. */
OR_EXPORT void or_layernorm_backward(real* dinp, real* dw, real* db, const real* dout,
                                     const real* inp, const real* w, const real* mean,
                                     const real* rstd, int B, int T, int C) {
    for (int bt = 0; bt < B * T; bt++) {
        const real* d = dout + (size_t)bt * C;
        const real* x = inp + (size_t)bt * C;
        real* dx = dinp + (size_t)bt * C;
        real m = mean[bt], s = rstd[bt];
        real g_mean = 0, gn_mean = 0;
        for (int c = 0; c < C; c++) {
            real n = (x[c] - m) * s;
            real g = w[c] * d[c];
            g_mean += g;
            gn_mean += g * n;
        }
        g_mean = g_mean / C;
        gn_mean = gn_mean / C;
        for (int c = 0; c < C; c++) {
            real n = (x[c] - m) * s;
            real g = w[c] * d[c];
            db[c] += d[c];
            dw[c] += n * d[c];
            real val = g;
            val -= g_mean;
            val -= n * gn_mean;
            val *= s;
            dx[c] += val;
        }
    }
}

/* RMSNorm, the normalisation of the microGPT page's transformer block ("microGPT 3D",
 * lesson 04: embedding -> RMSNorm -> attention -> residual -> MLP -> residual ->
 * logits).  The page names the operation only; this is its standard definition
 * (root-mean-square normalisation, no mean subtraction) with the same eps as the
 * LayerNorm above and a per-channel gain w, no shift:
 *   ms = sum_c x[c]^2 / C,  rstd = 1/sqrt(ms + 1e-5),  out = x*rstd*w.
 * rstd is kept for the backward. */
OR_EXPORT void or_rmsnorm_forward(real* out, real* rstd, const real* inp, const real* w, int B, int T,
                                  int C) {
    const real eps = (real)1e-5;
    for (int bt = 0; bt < B * T; bt++) {
        const real* x = inp + (size_t)bt * C;
        real ms = 0;
        for (int c = 0; c < C; c++) ms += x[c] * x[c];
        ms = ms / C;
        real s = (real)1 / R_SQRT(ms + eps);
        real* o = out + (size_t)bt * C;
        for (int c = 0; c < C; c++) o[c] = (s * x[c]) * w[c];
        rstd[bt] = s;
    }
}

/* Backward of or_rmsnorm_forward.  With n = x*rstd and g = w*dout (the chain rule
 * through ms, which depends on every x[c]):
 *   dw += n*dout,
 *   dinp += (g - n*mean(g*n)) * rstd. */
OR_EXPORT void or_rmsnorm_backward(real* dinp, real* dw, const real* dout, const real* inp, const real* w,
                                   const real* rstd, int B, int T, int C) {
    for (int bt = 0; bt < B * T; bt++) {
        const real* d = dout + (size_t)bt * C;
        const real* x = inp + (size_t)bt * C;
        real* dx = dinp + (size_t)bt * C;
        real s = rstd[bt];
        real gn_mean = 0;
        for (int c = 0; c < C; c++) gn_mean += (w[c] * d[c]) * (x[c] * s);
        gn_mean = gn_mean / C;
        for (int c = 0; c < C; c++) {
            real n = x[c] * s;
            dw[c] += n * d[c];
            dx[c] += (w[c] * d[c] - n * gn_mean) * s;
        }
    }
}

/* llm.c §1.5 matmul_forward: out[bt,o] = bias[o] + sum_i inp[bt,i]*W[o,i],
 * W stored (OC, C) row-major; bias may be NULL (the tied vocab projection). */
OR_EXPORT void or_matmul_forward(real* out, const real* inp, const real* W, const real* bias,
                                 int B, int T, int C, int OC) {
    #pragma omp parallel for
    for (int bt = 0; bt < B * T; bt++) {
        const real* x = inp + (size_t)bt * C;
        real* o = out + (size_t)bt * OC;
        for (int oc = 0; oc < OC; oc++) {
            const real* wr = W + (size_t)oc * C;
            real acc = bias ? bias[oc] : (real)0;
            for (int i = 0; i < C; i++) acc += x[i] * wr[i];
            o[oc] = acc;
        }
    }
}

/* llm.c §1.6 matmul_backward: dinp += dout . W (over positions), then
 * dW[o,:] += dout[bt,o] * inp[bt,:] and dbias[o] += dout[bt,o] (over output
 * channels, positions in order). */
OR_EXPORT void or_matmul_backward(real* dinp, real* dW, real* dbias, const real* dout,
                                  const real* inp, const real* W, int B, int T, int C, int OC) {
    #pragma omp parallel for
    for (int bt = 0; bt < B * T; bt++) {
        const real* d = dout + (size_t)bt * OC;
        real* dx = dinp + (size_t)bt * C;
        for (int oc = 0; oc < OC; oc++) {
            const real* wr = W + (size_t)oc * C;
            real g = d[oc];
            for (int i = 0; i < C; i++) dx[i] += wr[i] * g;
        }
    }
    #pragma omp parallel for
    for (int oc = 0; oc < OC; oc++) {
        real* dwr = dW + (size_t)oc * C;
        for (int bt = 0; bt < B * T; bt++) {
            const real* x = inp + (size_t)bt * C;
            real g = dout[(size_t)bt * OC + oc];
            if (dbias) dbias[oc] += g;
            for (int i = 0; i < C; i++) dwr[i] += x[i] * g;
        }
    }
}

/* llm.c §1.7 attention_forward; picoGPT attention/mha with the causal mask.
 * inp is the (B,T,3C) qkv buffer: query at channel offset 0, key at +C, value
 * at +2C, head h owning channels [h*hs, (h+1)*hs) of each.  For each (b,t,h):
 * preatt[t2] = q.k_t2 / sqrt(hs) for t2 <= t; att = softmax over t2 <= t,
 * zero for t2 > t; out = sum_t2 att[t2] v_t2.  preatt and att are (B,NH,T,T). */
OR_EXPORT void or_attention_forward(real* out, real* preatt, real* att, const real* inp,
                                    int B, int T, int C, int NH) {
    const int C3 = 3 * C, hs = C / NH;
    const real scale = (real)1 / R_SQRT((real)hs);
    #pragma omp parallel for collapse(2)
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < NH; h++) {
            for (int t = 0; t < T; t++) {
                const real* q = inp + ((size_t)b * T + t) * C3 + h * hs;
                real* pre = preatt + (((size_t)b * NH + h) * T + t) * T;
                real* a = att + (((size_t)b * NH + h) * T + t) * T;
                real mx = -INFINITY;
                for (int t2 = 0; t2 <= t; t2++) {
                    const real* k = inp + ((size_t)b * T + t2) * C3 + h * hs + C;
                    real s = 0;
                    for (int i = 0; i < hs; i++) s += q[i] * k[i];
                    s *= scale;
                    if (s > mx) mx = s;
                    pre[t2] = s;
                }
                real sum = 0;
                for (int t2 = 0; t2 <= t; t2++) {
                    real e = R_EXP(pre[t2] - mx);
                    sum += e;
                    a[t2] = e;
                }
                real inv = sum == (real)0 ? (real)0 : (real)1 / sum;
                for (int t2 = 0; t2 < T; t2++) a[t2] = t2 <= t ? a[t2] * inv : (real)0;
                real* o = out + ((size_t)b * T + t) * C + h * hs;
                for (int i = 0; i < hs; i++) o[i] = 0;
                for (int t2 = 0; t2 <= t; t2++) {
                    const real* v = inp + ((size_t)b * T + t2) * C3 + h * hs + 2 * C;
                    for (int i = 0; i < hs; i++) o[i] += a[t2] * v[i];
                }
            }
        }
    }
}

/* llm.c §1.8 attention_backward: through the weighted value sum (datt, dv),
 * the softmax Jacobian dpreatt[t3] += att[t2]*(1[t2==t3] - att[t3])*datt[t2],
 * and the scaled dot product (dq, dk).  Loops over (b,h) are independent: each
 * pair writes its own channel slice of dinp and its own datt/dpreatt rows, and
 * inside a pair the t order is the listing's. */
OR_EXPORT void or_attention_backward(real* dinp, real* dpreatt, real* datt, const real* dout,
                                     const real* inp, const real* att, int B, int T, int C, int NH) {
    const int C3 = 3 * C, hs = C / NH;
    const real scale = (real)1 / R_SQRT((real)hs);
    #pragma omp parallel for collapse(2)
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < NH; h++) {
            for (int t = 0; t < T; t++) {
                const real* a = att + (((size_t)b * NH + h) * T + t) * T;
                real* da = datt + (((size_t)b * NH + h) * T + t) * T;
                real* dpre = dpreatt + (((size_t)b * NH + h) * T + t) * T;
                const real* q = inp + ((size_t)b * T + t) * C3 + h * hs;
                real* dq = dinp + ((size_t)b * T + t) * C3 + h * hs;
                const real* d = dout + ((size_t)b * T + t) * C + h * hs;
                for (int t2 = 0; t2 <= t; t2++) {
                    const real* v = inp + ((size_t)b * T + t2) * C3 + h * hs + 2 * C;
                    real* dv = dinp + ((size_t)b * T + t2) * C3 + h * hs + 2 * C;
                    for (int i = 0; i < hs; i++) {
                        da[t2] += v[i] * d[i];
                        dv[i] += a[t2] * d[i];
                    }
                }
                for (int t2 = 0; t2 <= t; t2++) {
                    for (int t3 = 0; t3 <= t; t3++) {
                        real ind = t2 == t3 ? (real)1 : (real)0;
                        dpre[t3] += a[t2] * (ind - a[t3]) * da[t2];
                    }
                }
                for (int t2 = 0; t2 <= t; t2++) {
                    const real* k = inp + ((size_t)b * T + t2) * C3 + h * hs + C;
                    real* dk = dinp + ((size_t)b * T + t2) * C3 + h * hs + C;
                    for (int i = 0; i < hs; i++) {
                        dq[i] += k[i] * dpre[t2] * scale;
                        dk[i] += q[i] * dpre[t2] * scale;
                    }
                }
            }
        }
    }
}

/* llm.c §1.9 gelu_forward; picoGPT gelu: the tanh approximation
 * 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))). */
OR_EXPORT void or_gelu_forward(real* out, const real* inp, size_t N) {
    const real k = R_SQRT((real)2 / (real)M_PI);
    for (size_t i = 0; i < N; i++) {
        real x = inp[i];
        real cube = (real)0.044715 * x * x * x;
        out[i] = (real)0.5 * x * ((real)1 + R_TANH(k * (x + cube)));
    }
}

/* llm.c §1.10 gelu_backward: derivative of the tanh form,
 * 0.5(1+tanh u) + x*0.5*sech^2(u)*sqrt(2/pi)*(1+3*0.044715 x^2), times dout,
 * added into dinp. */
OR_EXPORT void or_gelu_backward(real* dinp, const real* inp, const real* dout, size_t N) {
    const real k = R_SQRT((real)2 / (real)M_PI);
    for (size_t i = 0; i < N; i++) {
        real x = inp[i];
        real u = k * (x + (real)0.044715 * x * x * x);
        real th = R_TANH(u);
        real ch = R_COSH(u);
        real sech2 = (real)1 / (ch * ch);
        real local = (real)0.5 * ((real)1 + th) +
                     x * (real)0.5 * sech2 * k * ((real)1 + (real)3 * (real)0.044715 * x * x);
        dinp[i] += local * dout[i];
    }
}

/* llm.c §1.11 residual_forward. */
OR_EXPORT void or_residual_forward(real* out, const real* a, const real* b, size_t N) {
    for (size_t i = 0; i < N; i++) out[i] = a[i] + b[i];
}

/* llm.c §1.12 residual_backward. */
OR_EXPORT void or_residual_backward(real* da, real* db, const real* dout, size_t N) {
    for (size_t i = 0; i < N; i++) {
        da[i] += dout[i];
        db[i] += dout[i];
    }
}

/* llm.c §1.13 softmax_forward; picoGPT softmax (max-subtracted).  Rows of V. */
OR_EXPORT void or_softmax_forward(real* probs, const real* logits, int B, int T, int V) {
    #pragma omp parallel for
    for (int bt = 0; bt < B * T; bt++) {
        const real* l = logits + (size_t)bt * V;
        real* p = probs + (size_t)bt * V;
        real mx = -INFINITY;
        for (int i = 0; i < V; i++) if (l[i] > mx) mx = l[i];
        real sum = 0;
        for (int i = 0; i < V; i++) {
            p[i] = R_EXP(l[i] - mx);
            sum += p[i];
        }
        for (int i = 0; i < V; i++) p[i] /= sum;
    }
}

/* llm.c §1.14 crossentropy_forward: losses[bt] = -log(probs[bt, target]). */
OR_EXPORT void or_crossentropy_forward(real* losses, const real* probs, const int* targets,
                                       int B, int T, int V) {
    for (int bt = 0; bt < B * T; bt++) losses[bt] = -R_LOG(probs[(size_t)bt * V + targets[bt]]);
}

/* llm.c §1.15 crossentropy_softmax_backward: dlogits += (p - onehot) * dloss. */
OR_EXPORT void or_crossentropy_softmax_backward(real* dlogits, const real* dlosses, const real* probs,
                                                const int* targets, int B, int T, int V) {
    for (int bt = 0; bt < B * T; bt++) {
        const real* p = probs + (size_t)bt * V;
        real* dl = dlogits + (size_t)bt * V;
        real g = dlosses[bt];
        int ix = targets[bt];
        for (int i = 0; i < V; i++) {
            real ind = i == ix ? (real)1 : (real)0;
            dl[i] += (p[i] - ind) * g;
        }
    }
}

/* llm.c §1.26 gpt2_update, one element at a time over a flat buffer (AdamW as
 * in the PyTorch documentation the listing links): m and v moments, bias
 * correction with beta^t (t counted from 1), decoupled weight decay applied to
 * the value of the parameter before the update.  Returns -1 if t < 1. */
OR_EXPORT int or_adamw(real* p, const real* g, real* m, real* v, size_t n, real lr, real b1,
                       real b2, real eps, real wd, int t) {
    if (t < 1) return -1;
    const real c1 = (real)1 - R_POW(b1, (real)t);
    const real c2 = (real)1 - R_POW(b2, (real)t);
    for (size_t i = 0; i < n; i++) {
        real old = p[i];
        real mi = b1 * m[i] + ((real)1 - b1) * g[i];
        real vi = b2 * v[i] + ((real)1 - b2) * g[i] * g[i];
        real mhat = mi / c1;
        real vhat = vi / c2;
        m[i] = mi;
        v[i] = vi;
        p[i] -= lr * (mhat / (R_SQRT(vhat) + eps) + wd * old);
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* the model: one flat buffer per role (llm.c §1.16-§1.21)                    */
/* ------------------------------------------------------------------------- */

enum { NP = 16, NA = 23 };

typedef struct {
    real *wte, *wpe, *ln1w, *ln1b, *qkvw, *qkvb, *attprojw, *attprojb, *ln2w, *ln2b, *fcw, *fcb,
        *fcprojw, *fcprojb, *lnfw, *lnfb;
} Params;

typedef struct {
    real *encoded, *ln1, *ln1_mean, *ln1_rstd, *qkv, *atty, *preatt, *att, *attproj, *residual2,
        *ln2, *ln2_mean, *ln2_rstd, *fch, *fch_gelu, *fcproj, *residual3, *lnf, *lnf_mean,
        *lnf_rstd, *logits, *probs, *losses;
} Acts;

/* Normalisation of the model: GPT-2's LayerNorm (llm.c) or the microGPT variant's
 * RMSNorm.  The RMSNorm model keeps the GPT-2 parameter layout; the LayerNorm
 * shift tensors (ln1b, ln2b, lnfb) are carried but unused, so their gradients are 0. */
enum { OR_LAYERNORM = 0, OR_RMSNORM = 1 };

typedef struct {
    int L, C, NH, V, maxT, norm;
    size_t psize[NP], nparams;
    Params p, g;
    real *pmem, *gmem, *mmem, *vmem;
    size_t asize[NA], nacts;
    Acts a, ga;
    real *amem, *gamem;
    int B, T;
    int *inputs, *targets;
    int have_targets;
    real mean_loss;
} OracleModel;

/* llm.c §1.17: carve consecutive tensors out of one allocation. */
static real* carve(real** slots[], const size_t* sizes, int n, size_t* total_out) {
    size_t total = 0;
    for (int i = 0; i < n; i++) total += sizes[i];
    real* mem = (real*)calloc(total ? total : 1, sizeof(real));
    if (!mem) return NULL;
    real* it = mem;
    for (int i = 0; i < n; i++) {
        *slots[i] = it;
        it += sizes[i];
    }
    if (total_out) *total_out = total;
    return mem;
}

static real* carve_params(Params* p, const size_t* sizes) {
    real** s[NP] = {&p->wte, &p->wpe, &p->ln1w, &p->ln1b, &p->qkvw, &p->qkvb, &p->attprojw,
                    &p->attprojb, &p->ln2w, &p->ln2b, &p->fcw, &p->fcb, &p->fcprojw, &p->fcprojb,
                    &p->lnfw, &p->lnfb};
    return carve(s, sizes, NP, NULL);
}

static real* carve_acts(Acts* a, const size_t* sizes) {
    real** s[NA] = {&a->encoded, &a->ln1, &a->ln1_mean, &a->ln1_rstd, &a->qkv, &a->atty,
                    &a->preatt, &a->att, &a->attproj, &a->residual2, &a->ln2, &a->ln2_mean,
                    &a->ln2_rstd, &a->fch, &a->fch_gelu, &a->fcproj, &a->residual3, &a->lnf,
                    &a->lnf_mean, &a->lnf_rstd, &a->logits, &a->probs, &a->losses};
    return carve(s, sizes, NA, NULL);
}

/* llm.c §1.22 (sizes) without the checkpoint file: the caller uploads the
 * parameters with or_set_params. */
OR_EXPORT OracleModel* or_build_ex(int L, int C, int NH, int V, int maxT, int norm) {
    if (L <= 0 || C <= 0 || NH <= 0 || V <= 0 || maxT <= 0 || C % NH) return NULL;
    if (norm != OR_LAYERNORM && norm != OR_RMSNORM) return NULL;
    OracleModel* m = (OracleModel*)calloc(1, sizeof(OracleModel));
    if (!m) return NULL;
    m->L = L; m->C = C; m->NH = NH; m->V = V; m->maxT = maxT; m->norm = norm;
    size_t Ls = L, Cs = C;
    size_t sz[NP] = {(size_t)V * Cs, (size_t)maxT * Cs, Ls * Cs, Ls * Cs, Ls * 3 * Cs * Cs,
                     Ls * 3 * Cs, Ls * Cs * Cs, Ls * Cs, Ls * Cs, Ls * Cs, Ls * 4 * Cs * Cs,
                     Ls * 4 * Cs, Ls * Cs * 4 * Cs, Ls * Cs, Cs, Cs};
    m->nparams = 0;
    for (int i = 0; i < NP; i++) { m->psize[i] = sz[i]; m->nparams += sz[i]; }
    m->pmem = carve_params(&m->p, m->psize);
    if (!m->pmem) { free(m); return NULL; }
    m->mean_loss = -1;
    return m;
}

OR_EXPORT OracleModel* or_build(int L, int C, int NH, int V, int maxT) {
    return or_build_ex(L, C, NH, V, maxT, OR_LAYERNORM);
}

OR_EXPORT size_t or_num_params(const OracleModel* m) { return m->nparams; }
OR_EXPORT size_t or_num_acts(const OracleModel* m) { return m->nacts; }
OR_EXPORT void or_param_sizes(const OracleModel* m, size_t* out) {
    for (int i = 0; i < NP; i++) out[i] = m->psize[i];
}

OR_EXPORT void or_set_params(OracleModel* m, const real* src) {
    memcpy(m->pmem, src, m->nparams * sizeof(real));
}
OR_EXPORT void or_get_params(const OracleModel* m, real* dst) {
    memcpy(dst, m->pmem, m->nparams * sizeof(real));
}
OR_EXPORT int or_get_grads(const OracleModel* m, real* dst) {
    if (!m->gmem) return -1;
    memcpy(dst, m->gmem, m->nparams * sizeof(real));
    return 0;
}
OR_EXPORT int or_get_opt_state(const OracleModel* m, real* mdst, real* vdst) {
    if (!m->mmem) return -1;
    memcpy(mdst, m->mmem, m->nparams * sizeof(real));
    memcpy(vdst, m->vmem, m->nparams * sizeof(real));
    return 0;
}
/* (B,T,V) logits of the last forward. */
OR_EXPORT int or_get_logits(const OracleModel* m, real* dst) {
    if (!m->amem) return -1;
    memcpy(dst, m->a.logits, (size_t)m->B * m->T * m->V * sizeof(real));
    return 0;
}
/* (B,T) per-position losses of the last forward with targets. */
OR_EXPORT int or_get_losses(const OracleModel* m, real* dst) {
    if (!m->amem || !m->have_targets) return -1;
    memcpy(dst, m->a.losses, (size_t)m->B * m->T * sizeof(real));
    return 0;
}
/* Activation-gradient of the encoder output (B,T,C) after a backward. */
OR_EXPORT int or_get_dencoded(const OracleModel* m, real* dst) {
    if (!m->gamem) return -1;
    memcpy(dst, m->ga.encoded, (size_t)m->B * m->T * m->C * sizeof(real));
    return 0;
}

/* The model's normalisation (LayerNorm, or RMSNorm for the microGPT variant, whose
 * mean slot is set to 0 and whose shift is not read). */
static void norm_forward(const OracleModel* m, real* out, real* mean, real* rstd, const real* inp,
                         const real* w, const real* b, int B, int T, int C) {
    if (m->norm == OR_RMSNORM) {
        or_rmsnorm_forward(out, rstd, inp, w, B, T, C);
        for (int i = 0; i < B * T; i++) mean[i] = 0;
    } else {
        or_layernorm_forward(out, mean, rstd, inp, w, b, B, T, C);
    }
}

static void norm_backward(const OracleModel* m, real* dinp, real* dw, real* db, const real* dout,
                          const real* inp, const real* w, const real* mean, const real* rstd, int B,
                          int T, int C) {
    if (m->norm == OR_RMSNORM)
        or_rmsnorm_backward(dinp, dw, dout, inp, w, rstd, B, T, C);
    else
        or_layernorm_backward(dinp, dw, db, dout, inp, w, mean, rstd, B, T, C);
}

/* llm.c §1.23 gpt2_forward.  Returns 0, -1 on out-of-range ids, -2 if (B,T)
 * differs from the first call or T > maxT, -3 on allocation failure.  The mean
 * loss is stored in *mean_loss (or -1 without targets). */
OR_EXPORT int or_forward(OracleModel* m, const int* inputs, const int* targets, int B, int T,
                         real* mean_loss) {
    const int V = m->V, L = m->L, NH = m->NH, C = m->C;
    if (B <= 0 || T <= 0 || T > m->maxT) return -2;
    for (int i = 0; i < B * T; i++) {
        if (inputs[i] < 0 || inputs[i] >= V) return -1;
        if (targets && (targets[i] < 0 || targets[i] >= V)) return -1;
    }
    if (!m->amem) {
        m->B = B; m->T = T;
        size_t Ls = L, BT = (size_t)B * T, Cs = C;
        size_t sz[NA] = {BT * Cs, Ls * BT * Cs, Ls * BT, Ls * BT, Ls * BT * 3 * Cs, Ls * BT * Cs,
                         Ls * B * NH * (size_t)T * T, Ls * B * NH * (size_t)T * T, Ls * BT * Cs,
                         Ls * BT * Cs, Ls * BT * Cs, Ls * BT, Ls * BT, Ls * BT * 4 * Cs,
                         Ls * BT * 4 * Cs, Ls * BT * Cs, Ls * BT * Cs, BT * Cs, BT, BT,
                         BT * V, BT * V, BT};
        m->nacts = 0;
        for (int i = 0; i < NA; i++) { m->asize[i] = sz[i]; m->nacts += sz[i]; }
        m->amem = carve_acts(&m->a, m->asize);
        m->inputs = (int*)malloc((size_t)B * T * sizeof(int));
        m->targets = (int*)malloc((size_t)B * T * sizeof(int));
        if (!m->amem || !m->inputs || !m->targets) return -3;
    } else if (B != m->B || T != m->T) {
        return -2;
    }
    memcpy(m->inputs, inputs, (size_t)B * T * sizeof(int));
    if (targets) memcpy(m->targets, targets, (size_t)B * T * sizeof(int));

    Params p = m->p;
    Acts a = m->a;
    const size_t BTC = (size_t)B * T * C, BT = (size_t)B * T, BNTT = (size_t)B * NH * T * T;
    or_encoder_forward(a.encoded, inputs, p.wte, p.wpe, B, T, C);
    for (int l = 0; l < L; l++) {
        real* res = l == 0 ? a.encoded : a.residual3 + (size_t)(l - 1) * BTC;
        real* ln1 = a.ln1 + l * BTC;
        real* qkv = a.qkv + l * 3 * BTC;
        real* atty = a.atty + l * BTC;
        real* attproj = a.attproj + l * BTC;
        real* res2 = a.residual2 + l * BTC;
        real* ln2 = a.ln2 + l * BTC;
        real* fch = a.fch + l * 4 * BTC;
        real* fchg = a.fch_gelu + l * 4 * BTC;
        real* fcproj = a.fcproj + l * BTC;
        real* res3 = a.residual3 + l * BTC;
        norm_forward(m, ln1, a.ln1_mean + l * BT, a.ln1_rstd + l * BT, res, p.ln1w + l * C,
                             p.ln1b + l * C, B, T, C);
        or_matmul_forward(qkv, ln1, p.qkvw + (size_t)l * 3 * C * C, p.qkvb + l * 3 * C, B, T, C, 3 * C);
        or_attention_forward(atty, a.preatt + l * BNTT, a.att + l * BNTT, qkv, B, T, C, NH);
        or_matmul_forward(attproj, atty, p.attprojw + (size_t)l * C * C, p.attprojb + l * C, B, T, C, C);
        or_residual_forward(res2, res, attproj, BTC);
        norm_forward(m, ln2, a.ln2_mean + l * BT, a.ln2_rstd + l * BT, res2, p.ln2w + l * C,
                             p.ln2b + l * C, B, T, C);
        or_matmul_forward(fch, ln2, p.fcw + (size_t)l * 4 * C * C, p.fcb + l * 4 * C, B, T, C, 4 * C);
        or_gelu_forward(fchg, fch, 4 * BTC);
        or_matmul_forward(fcproj, fchg, p.fcprojw + (size_t)l * C * 4 * C, p.fcprojb + l * C, B, T,
                          4 * C, C);
        or_residual_forward(res3, res2, fcproj, BTC);
    }
    real* last = a.residual3 + (size_t)(L - 1) * BTC;
    norm_forward(m, a.lnf, a.lnf_mean, a.lnf_rstd, last, p.lnfw, p.lnfb, B, T, C);
    or_matmul_forward(a.logits, a.lnf, p.wte, NULL, B, T, C, V);
    or_softmax_forward(a.probs, a.logits, B, T, V);
    if (targets) {
        or_crossentropy_forward(a.losses, a.probs, targets, B, T, V);
        real s = 0;
        for (size_t i = 0; i < BT; i++) s += a.losses[i];
        m->mean_loss = s / (real)BT;
        m->have_targets = 1;
    } else {
        m->mean_loss = -1;
        m->have_targets = 0;
    }
    if (mean_loss) *mean_loss = m->mean_loss;
    return 0;
}

/* llm.c §1.24 gpt2_zero_grad. */
OR_EXPORT void or_zero_grad(OracleModel* m) {
    if (m->gmem) memset(m->gmem, 0, m->nparams * sizeof(real));
    if (m->gamem) memset(m->gamem, 0, m->nacts * sizeof(real));
}

/* llm.c §1.25 gpt2_backward.  Accumulates (+=) into the gradient buffers like
 * the listing; call or_zero_grad first for a fresh gradient.  Returns -1 if the
 * last forward had no targets, -3 on allocation failure. */
OR_EXPORT int or_backward(OracleModel* m) {
    if (!m->amem || !m->have_targets) return -1;
    /* gradient buffers on first use (the activation gradients again after
     * or_release_acts, which frees them with the activations); calloc leaves them zero */
    if (!m->gmem) m->gmem = carve_params(&m->g, m->psize);
    if (!m->gamem) m->gamem = carve_acts(&m->ga, m->asize);
    if (!m->gmem || !m->gamem) return -3;
    const int B = m->B, T = m->T, V = m->V, L = m->L, NH = m->NH, C = m->C;
    const size_t BTC = (size_t)B * T * C, BT = (size_t)B * T, BNTT = (size_t)B * NH * T * T;
    Params p = m->p, g = m->g;
    Acts a = m->a, ga = m->ga;

    real dmean = (real)1 / (real)BT;
    for (size_t i = 0; i < BT; i++) ga.losses[i] = dmean;
    or_crossentropy_softmax_backward(ga.logits, ga.losses, a.probs, m->targets, B, T, V);
    or_matmul_backward(ga.lnf, g.wte, NULL, ga.logits, a.lnf, p.wte, B, T, C, V);
    real* res = a.residual3 + (size_t)(L - 1) * BTC;
    real* dres = ga.residual3 + (size_t)(L - 1) * BTC;
    norm_backward(m, dres, g.lnfw, g.lnfb, ga.lnf, res, p.lnfw, a.lnf_mean, a.lnf_rstd, B, T, C);
    for (int l = L - 1; l >= 0; l--) {
        res = l == 0 ? a.encoded : a.residual3 + (size_t)(l - 1) * BTC;
        dres = l == 0 ? ga.encoded : ga.residual3 + (size_t)(l - 1) * BTC;
        or_residual_backward(ga.residual2 + l * BTC, ga.fcproj + l * BTC, ga.residual3 + l * BTC, BTC);
        or_matmul_backward(ga.fch_gelu + l * 4 * BTC, g.fcprojw + (size_t)l * C * 4 * C,
                           g.fcprojb + l * C, ga.fcproj + l * BTC, a.fch_gelu + l * 4 * BTC,
                           p.fcprojw + (size_t)l * C * 4 * C, B, T, 4 * C, C);
        or_gelu_backward(ga.fch + l * 4 * BTC, a.fch + l * 4 * BTC, ga.fch_gelu + l * 4 * BTC, 4 * BTC);
        or_matmul_backward(ga.ln2 + l * BTC, g.fcw + (size_t)l * 4 * C * C, g.fcb + l * 4 * C,
                           ga.fch + l * 4 * BTC, a.ln2 + l * BTC, p.fcw + (size_t)l * 4 * C * C, B,
                           T, C, 4 * C);
        norm_backward(m, ga.residual2 + l * BTC, g.ln2w + l * C, g.ln2b + l * C, ga.ln2 + l * BTC,
                              a.residual2 + l * BTC, p.ln2w + l * C, a.ln2_mean + l * BT,
                              a.ln2_rstd + l * BT, B, T, C);
        or_residual_backward(dres, ga.attproj + l * BTC, ga.residual2 + l * BTC, BTC);
        or_matmul_backward(ga.atty + l * BTC, g.attprojw + (size_t)l * C * C, g.attprojb + l * C,
                           ga.attproj + l * BTC, a.atty + l * BTC, p.attprojw + (size_t)l * C * C,
                           B, T, C, C);
        or_attention_backward(ga.qkv + l * 3 * BTC, ga.preatt + l * BNTT, ga.att + l * BNTT,
                              ga.atty + l * BTC, a.qkv + l * 3 * BTC, a.att + l * BNTT, B, T, C, NH);
        or_matmul_backward(ga.ln1 + l * BTC, g.qkvw + (size_t)l * 3 * C * C, g.qkvb + l * 3 * C,
                           ga.qkv + l * 3 * BTC, a.ln1 + l * BTC, p.qkvw + (size_t)l * 3 * C * C,
                           B, T, C, 3 * C);
        norm_backward(m, dres, g.ln1w + l * C, g.ln1b + l * C, ga.ln1 + l * BTC, res,
                              p.ln1w + l * C, a.ln1_mean + l * BT, a.ln1_rstd + l * BT, B, T, C);
    }
    or_encoder_backward(g.wte, g.wpe, ga.encoded, m->inputs, B, T, C);
    return 0;
}

/* llm.c §1.26 gpt2_update over the whole flat parameter buffer (moments are
 * created zeroed on first use).  Returns -1 without gradients or with t < 1. */
OR_EXPORT int or_update(OracleModel* m, real lr, real b1, real b2, real eps, real wd, int t) {
    if (!m->gmem || t < 1) return -1;
    if (!m->mmem) {
        m->mmem = (real*)calloc(m->nparams, sizeof(real));
        m->vmem = (real*)calloc(m->nparams, sizeof(real));
        if (!m->mmem || !m->vmem) return -3;
    }
    return or_adamw(m->pmem, m->gmem, m->mmem, m->vmem, m->nparams, lr, b1, b2, eps, wd, t);
}

/* ------------------------------------------------------------------------- */
/* generation (picoGPT "generate"; llm.c §1.35 sample_mult)                    */
/* ------------------------------------------------------------------------- */

/* Drop the activation buffers (and their gradients) so the next or_forward may use
 * a different (B,T).  Parameters, gradients and AdamW moments are kept. */
OR_EXPORT void or_release_acts(OracleModel* m) {
    free(m->amem); free(m->gamem); free(m->inputs); free(m->targets);
    m->amem = m->gamem = NULL;
    m->inputs = m->targets = NULL;
    m->nacts = 0;
    m->have_targets = 0;
    m->mean_loss = -1;
}

/* llm.c §1.35 sample_mult: walk the cumulative distribution of the n probabilities and
 * return the first index whose cumulative value exceeds coin (in [0,1)); the last index
 * if rounding leaves coin above every cumulative value. */
OR_EXPORT int or_sample_mult(const real* probs, int n, real coin) {
    real cdf = 0;
    for (int i = 0; i < n; i++) {
        cdf += probs[i];
        if (coin < cdf) return i;
    }
    return n - 1;
}

/* picoGPT "generate", the autoregressive decode loop: n_new times, run the whole
 * forward over the sequence so far and pick the next id from the logits of its last
 * position, then append it.  temperature <= 0: greedy, argmax of the logits (the first
 * index among equal maxima, as numpy's argmax); temperature > 0: sample_mult over
 * softmax(logits / temperature) with coins[b * n_new + step] (drawn by the caller).
 * prompt (B,T0) int32; out (B,n_new) receives the new ids.  No cache: every step
 * recomputes every position.  Returns 0, or or_forward's code (T0 + n_new - 1 > maxT
 * gives -2, an id outside [0,V) -1), -3 on allocation failure. */
OR_EXPORT int or_generate(OracleModel* m, const int* prompt, int B, int T0, int n_new, real temperature,
                          const real* coins, int* out) {
    if (B <= 0 || T0 <= 0 || n_new < 0) return -2;
    const int V = m->V, Tmax = T0 + n_new;
    int* seq = (int*)malloc((size_t)B * Tmax * sizeof(int));
    int* cur = (int*)malloc((size_t)B * Tmax * sizeof(int));
    real* probs = (real*)malloc((size_t)V * sizeof(real));
    if (!seq || !cur || !probs) { free(seq); free(cur); free(probs); return -3; }
    for (int b = 0; b < B; b++)
        for (int t = 0; t < T0; t++) seq[b * Tmax + t] = prompt[b * T0 + t];
    int rc = 0;
    for (int step = 0; step < n_new && rc == 0; step++) {
        const int T = T0 + step;
        for (int b = 0; b < B; b++)
            for (int t = 0; t < T; t++) cur[b * T + t] = seq[b * Tmax + t];
        or_release_acts(m);
        rc = or_forward(m, cur, NULL, B, T, NULL);
        if (rc) break;
        for (int b = 0; b < B; b++) {
            const real* l = m->a.logits + ((size_t)b * T + (T - 1)) * V;
            int next = 0;
            if (temperature <= 0) {
                for (int i = 1; i < V; i++)
                    if (l[i] > l[next]) next = i;
            } else {
                real mx = -INFINITY;
                for (int i = 0; i < V; i++) if (l[i] / temperature > mx) mx = l[i] / temperature;
                real sum = 0;
                for (int i = 0; i < V; i++) {
                    probs[i] = R_EXP(l[i] / temperature - mx);
                    sum += probs[i];
                }
                for (int i = 0; i < V; i++) probs[i] /= sum;
                next = or_sample_mult(probs, V, coins[(size_t)b * n_new + step]);
            }
            seq[b * Tmax + T] = next;
            out[(size_t)b * n_new + step] = next;
        }
    }
    free(seq); free(cur); free(probs);
    return rc;
}

/* llm.c §1.27 gpt2_free. */
OR_EXPORT void or_free(OracleModel* m) {
    if (!m) return;
    free(m->pmem); free(m->gmem); free(m->mmem); free(m->vmem);
    free(m->amem); free(m->gamem); free(m->inputs); free(m->targets);
    free(m);
}

OR_EXPORT int or_real_bytes(void) { return (int)sizeof(real); }

/* Threads of the OpenMP loops for later calls (n <= 0 keeps the setting); returns the
 * count now in force (1 without OpenMP).  No result depends on it: every parallel loop
 * gives each thread its own outputs (rows, output channels or (b, h) pairs), each
 * computed in the listing's order. */
OR_EXPORT int or_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
