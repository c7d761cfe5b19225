/*
 * gpt2.h — C ABI of the B300 GPT-2 training step (forward, backward, AdamW).
 *
 * The operation is the one the llm.c listing defines on the page
 * "llm.c 的中文注解-20240421" (sections 1.16-1.27: ParameterTensors, GPT2Config,
 * gpt2_forward, gpt2_zero_grad, gpt2_backward, gpt2_update, gpt2_free) and that the
 * picoGPT article ("60 行 NumPy 代码 ... 实现一个 GPT": gpt2, transformer_block, mha,
 * ffn, lm_loss) states a second time: token + position embedding, L pre-LayerNorm
 * blocks of causal multi-head attention and a tanh-GELU MLP with residuals, a final
 * LayerNorm, a vocabulary projection tied to the token embedding, and softmax
 * cross-entropy against the inputs shifted by one; AdamW over one flat buffer.
 *
 * Conventions shared by every entry point:
 *  - A handle owns all of its device memory: one allocation for parameters,
 *    gradients, AdamW moments (and the bf16 weight copy in GPT2_BF16 mode) made by
 *    gpt2_build_ex, one for activations made by the first forward.  Nothing else is
 *    allocated on the hot path.
 *  - Parameter order and shapes are those of the listing (section 1.16): wte (V,C),
 *    wpe (maxT,C), ln1w, ln1b (L,C), qkvw (L,3C,C), qkvb (L,3C), attprojw (L,C,C),
 *    attprojb (L,C), ln2w, ln2b (L,C), fcw (L,4C,C), fcb (L,4C), fcprojw (L,C,4C),
 *    fcprojb (L,C), lnfw, lnfb (C); weights are (out, in) row-major; fp32.  Host
 *    buffers exchanged with set/get use exactly that layout with the real vocabulary
 *    V; internally the vocabulary is padded to Vp (a multiple of 128) with zero rows
 *    that never receive gradient.
 *  - All work is ordered on the handle's CUDA stream (gpt2_set_stream; default: the
 *    legacy default stream).  Only the calls documented as synchronising wait for it.
 *  - Host pointers are read or written only during the call; the library keeps no
 *    reference to caller memory.  Device pointers must stay valid until the work
 *    queued by the call has run.
 *  - A handle is not thread-safe.  Errors never abort the process: calls return a
 *    negative gpt2_status and gpt2_last_error() describes the last failure.
 */
#ifndef GPT2_B300_H
#define GPT2_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gpt2 gpt2_t;

/* Status codes.  The listing exits the process on these conditions (bad model
 * state, ids out of range, B,T changing after the first forward, backward without
 * a forward with targets); this library returns them instead. */
enum gpt2_status {
    GPT2_OK = 0,
    GPT2_ERR_ARG = -1,       /* bad argument: NULL pointer, size mismatch, t < 1, ... */
    GPT2_ERR_OOM = -2,       /* device allocation failed; the handle stays freeable */
    GPT2_ERR_CUDA = -3,      /* a CUDA call failed; see gpt2_last_error */
    GPT2_ERR_TOKEN = -4,     /* an input id or target outside [0, V) */
    GPT2_ERR_SHAPE = -5,     /* (B,T) differs from the first forward, or T > maxT */
    GPT2_ERR_STATE = -6,     /* call order: backward before a forward with targets, ... */
    GPT2_ERR_NONFINITE = -7, /* the mean loss is NaN or infinite */
    GPT2_ERR_TIMEOUT = -8    /* a device-side bounded wait gave up (reported, never hangs) */
};

/* Arithmetic of the step.
 * GPT2_FP32: every tensor fp32, fp32 arithmetic everywhere (no TF32).
 * GPT2_TF32: every tensor fp32; the matrix products (llm.c §1.5 matmul_forward, §1.6
 *            matmul_backward) run on the tensor cores with their fp32 operands read as
 *            TF32 (10-bit mantissa) and fp32 accumulation; everything else as GPT2_FP32.
 *            Held to the bf16 tolerances, not the fp32 ones.
 * GPT2_BF16: bf16 activations and matrix operands, fp32 accumulation, fp32 master
 *            parameters, gradients and AdamW moments (mixed precision). */
enum gpt2_precision { GPT2_FP32 = 0, GPT2_TF32 = 1, GPT2_BF16 = 2 };

/* Where the id arrays of gpt2_forward_async live. */
enum gpt2_memory { GPT2_HOST = 0, GPT2_DEVICE = 1 };

/* Build a model (llm.c §1.20 GPT2Config, §1.22 sizes) and allocate its parameter
 * arena on the current CUDA device: parameters are zero until gpt2_set_params.
 * L layers, C channels, H heads (C % H == 0), V real vocabulary size, maxT maximum
 * sequence length.  Returns NULL on failure; *status (may be NULL) receives the code. */
gpt2_t* gpt2_build_ex(int L, int C, int H, int V, int maxT, int precision, int* status);
/* gpt2_build_ex(..., GPT2_BF16, NULL). */
gpt2_t* gpt2_build(int L, int C, int H, int V, int maxT);

/* Normalisation of the block.  GPT2_LAYERNORM: GPT-2's LayerNorm (llm.c §1.3, §1.4).
 * GPT2_RMSNORM: the microGPT variant (page "microGPT 3D", lesson 04: embedding ->
 * RMSNorm -> attention -> residual -> MLP -> residual -> logits): every LayerNorm
 * (ln1, ln2, lnf) becomes out = x / sqrt(mean(x^2) + 1e-5) * w with the same gains w;
 * the parameter layout is unchanged and the shift tensors (ln1b, ln2b, lnfb) are
 * carried but unused, so their gradients are 0. */
enum gpt2_norm { GPT2_LAYERNORM = 0, GPT2_RMSNORM = 1 };
/* gpt2_build_ex with a choice of normalisation; GPT2_ERR_ARG for another norm value.
 * gpt2_build_ex(...) = gpt2_build_norm(..., GPT2_LAYERNORM, status). */
gpt2_t* gpt2_build_norm(int L, int C, int H, int V, int maxT, int precision, int norm, int* status);
/* Release everything the handle owns (llm.c §1.27).  NULL is accepted. */
void gpt2_free(gpt2_t* m);

/* Number of parameters in the listing's layout with the real vocabulary V
 * (124,439,808 for L=12, C=768, V=50257, maxT=1024). */
size_t gpt2_num_params(const gpt2_t* m);
/* Vocabulary rows held on the device (V rounded up to a multiple of 128). */
int gpt2_padded_vocab(const gpt2_t* m);

/* Seeded initial parameters, drawn on the device (the listing's random_u32 / random_f32,
 * llm.c §1.33-§1.34, run as 65,536 xorshift64* lanes, lane j seeded with
 * splitmix64(seed + j); draw i of a tensor from lane i % 65536, whole rounds per tensor):
 * wte, wpe, qkvw, fcw ~ N(0, 0.02) and attprojw, fcprojw ~ N(0, 0.02/sqrt(2L)) by
 * Box-Muller in double (u1 >= 1e-7) rounded once to fp32, drawn in that order; LayerNorm
 * gains 1; biases, shifts and padded vocabulary rows 0.  Refreshes the bf16 weight copy;
 * the AdamW moments are left as they are.  The values equal those of the seeded input
 * generator the tests use (gpt_train_step_arena_b300.synth.init_params) up to the
 * last-ulp rounding of the double log, cos and sin of the two sides.  Asynchronous. */
int gpt2_init_params(gpt2_t* m, uint64_t seed);

/* Copy n = gpt2_num_params() fp32 values in, or out, in the layout above.  set also
 * refreshes the bf16 weight copy.  Synchronising.  GPT2_ERR_ARG if n differs. */
int gpt2_set_params(gpt2_t* m, const float* host, size_t n);
int gpt2_get_params(gpt2_t* m, float* host, size_t n);
/* Gradients of the last gpt2_backward (same layout).  GPT2_ERR_STATE before any. */
int gpt2_get_grads(gpt2_t* m, float* host, size_t n);
/* AdamW first and second moments (same layout; zero before the first update). */
int gpt2_get_opt_state(gpt2_t* m, float* m_host, float* v_host, size_t n);

/* Forward pass (llm.c §1.23).  tokens and targets are (B,T) int32 row-major host
 * arrays; targets may be NULL.  The first call fixes (B,T) and allocates the
 * activation arena; later calls must use the same (B,T) (GPT2_ERR_SHAPE); T <= maxT.
 * Returns the mean cross-entropy loss over all B*T positions, -1.0f when targets is
 * NULL (the listing's convention), or NaN on error (gpt2_last_status tells which).
 * Synchronising (one device-to-host read of the loss).  With targets, the logits
 * buffer is overwritten by the loss gradient for the following gpt2_backward. */
float gpt2_forward(gpt2_t* m, const int32_t* tokens, const int32_t* targets, int B, int T);
/* Same work without waiting: ids are read from host (copied on the stream) or device
 * memory per `where`.  Id range errors and a non-finite loss are reported by the
 * next gpt2_read_loss.  Returns a gpt2_status. */
int gpt2_forward_async(gpt2_t* m, const int32_t* tokens, const int32_t* targets, int B, int T,
                       int where);
/* Wait for the stream and read the mean loss of the last forward (-1.0f without
 * targets).  Returns GPT2_ERR_TOKEN / GPT2_ERR_NONFINITE if the forward saw bad ids
 * or a non-finite loss. */
int gpt2_read_loss(gpt2_t* m, float* loss_host);

/* Backward pass (llm.c §1.25).  Needs a forward with targets since the last
 * backward (GPT2_ERR_STATE otherwise).  Overwrites the gradient buffer (equivalent
 * to the listing's zero_grad followed by its accumulating backward).  Asynchronous. */
int gpt2_backward(gpt2_t* m);
/* Zero the gradient buffer (llm.c §1.24).  Asynchronous. */
int gpt2_zero_grad(gpt2_t* m);
/* AdamW (llm.c §1.26) over the whole flat parameter buffer, all tensors alike:
 * m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2; p -= lr (m/(1-b1^t) / (sqrt(v/(1-b2^t))
 * + eps) + wd p).  t counts updates from 1 (GPT2_ERR_ARG if t < 1).  Needs
 * gradients (GPT2_ERR_STATE).  Asynchronous. */
int gpt2_update(gpt2_t* m, float lr, float b1, float b2, float eps, float wd, int t);

/* Per-position losses (B,T) of the last forward with targets; n = B*T.  Synchronising. */
int gpt2_get_losses(gpt2_t* m, float* host, size_t n);
/* Logits (B,T,V) of the last forward WITHOUT targets (real columns, fp32); n = B*T*V.
 * Synchronising.  GPT2_ERR_STATE if the last forward had targets (its logits were
 * turned into the loss gradient in place). */
int gpt2_get_logits(gpt2_t* m, float* host, size_t n);

/* Autoregressive generation (picoGPT's "generate" decode loop; llm.c §1.35
 * sample_mult), with a key/value cache: the prompt's positions run through the model
 * once, then each new token only its own position, attending over the cached keys
 * and values of all earlier positions.  prompt: B*T0 host int32 ids (row-major
 * (B,T0), each in [0,V)); out: B*n_new host int32, receives the new ids (B,n_new).
 * temperature <= 0: greedy, the argmax of the last position's logits (the first
 * index among equal maxima); temperature > 0: the first id whose cumulative
 * softmax(logits / temperature) exceeds coins[b*n_new + step] (B*n_new host floats
 * in [0,1), drawn by the caller; NULL allowed when greedy).  Requires
 * T0 + n_new - 1 <= maxT (GPT2_ERR_SHAPE).  The first call for a batch size B
 * allocates the cache and working buffers for (B, maxT) in a separate device arena
 * (kept until gpt2_free or a call with another B); training buffers are untouched.
 * Stream-ordered on the handle's stream; synchronises once at the end. */
int gpt2_generate(gpt2_t* m, const int32_t* prompt, int B, int T0, int n_new, float temperature,
                  const float* coins, int32_t* out);
/* Logits (B,V) fp32 (real columns) from which the last gpt2_generate chose its last
 * ids; n = B*V.  GPT2_ERR_STATE before any generation.  Synchronising. */
int gpt2_get_gen_logits(gpt2_t* m, float* host, size_t n);

/* The device copies of the last forward's token ids and targets (B*T each; targets
 * may be NULL).  Synchronising. */
int gpt2_get_ids(gpt2_t* m, int32_t* tokens_host, int32_t* targets_host, size_t n);

/* Kernel classes of the step, for gpt2_profile_read. */
enum gpt2_kernel_class {
    GPT2_K_GEMM = 0,      /* all matrix products (forward, dgrad, wgrad): work = FLOPs */
    GPT2_K_ATTN_FWD = 1,  /* causal attention forward: work = FLOPs (QK^T and PV, t2 <= t) */
    GPT2_K_ATTN_BWD = 2,  /* attention backward: work = 2x the forward FLOPs */
    GPT2_K_LAYERNORM = 3, /* layernorm forward and backward: work = bytes */
    GPT2_K_XENT = 4,      /* fused softmax + cross-entropy and the loss mean: work = bytes */
    GPT2_K_ADAMW = 5,     /* AdamW over the flat buffer: work = bytes */
    GPT2_K_ENCODER = 6,   /* embedding forward and backward, id checks: work = bytes */
    GPT2_K_BIAS_GRAD = 7, /* bias-gradient column sums: work = bytes */
    GPT2_K_COUNT = 8
};
/* Per-class timing.  While enabled, every op the handle queues is bracketed by a CUDA
 * event pair on the handle's stream and its algorithmic work (read-once/write-once
 * bytes, or FLOPs) is booked to its class.  gpt2_profile_read synchronises, adds up
 * all pairs recorded since the last read or reset into the class totals, and returns
 * the totals (milliseconds, work units, number of ops).  Reset clears them. */
int gpt2_profile_enable(gpt2_t* m, int on);
int gpt2_profile_reset(gpt2_t* m);
int gpt2_profile_read(gpt2_t* m, int kernel_class, double* ms, double* work, uint64_t* calls);

/* Diagnostic of the device-side bounded waits every tensor-core kernel uses: runs, on the
 * handle's stream, a one-thread kernel that waits on an mbarrier nothing arrives at, with
 * the wait's limit shortened to timeout_us microseconds (1..1e6), no copy or MMA in
 * flight.  The wait gives up, raises the device timeout flag and returns; the call
 * synchronises, clears the flag and returns GPT2_ERR_TIMEOUT (the status any call that
 * reads the flags reports after a real timeout).  The handle stays usable.  Needs a
 * prior forward (the flags live in the activation arena): GPT2_ERR_STATE otherwise. */
int gpt2_check_bounded_wait(gpt2_t* m, unsigned timeout_us);

/* Run subsequent work on `stream` (a cudaStream_t; NULL = legacy default stream). */
int gpt2_set_stream(gpt2_t* m, void* stream);
/* Wait for all queued work; returns a gpt2_status for any pending CUDA error. */
int gpt2_sync(gpt2_t* m);
/* Last status and a human-readable description of the last failure. */
int gpt2_last_status(const gpt2_t* m);
const char* gpt2_last_error(const gpt2_t* m);
/* Message of the last gpt2_build_ex failure (process-wide). */
const char* gpt2_last_build_error(void);
/* Number of kernel launches the handle has queued since it was built. */
uint64_t gpt2_kernel_launches(const gpt2_t* m);
/* Device bytes held by the handle (parameter, activation and generation arenas). */
size_t gpt2_device_bytes(const gpt2_t* m);

#ifdef __cplusplus
}
#endif
#endif /* GPT2_B300_H */
