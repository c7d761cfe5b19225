// Kernels of autoregressive generation with a key/value cache: picoGPT's "generate"
// decode loop (greedy argmax, or sampling from the last position's distribution with
// a temperature), the sampling rule being llm.c §1.35 sample_mult.
//
// An "extend" step runs the forward of n new positions t0..t0+n-1 of each of the B
// sequences: the embedding at an offset, the usual layernorm / GEMM kernels on the
// B*n new rows, and, per layer, the new keys and values appended to the cache
// kv (B, maxT, 2C) [k | v] and the attention of the new queries over the cached
// positions 0..t.  The prompt is one extend with t0 = 0, n = T0; each further token
// one extend with n = 1.  Only the last position of each sequence reaches the LM head.
//
// The one-token steps read their position from device memory (dstate: t0, step, n_new,
// temperature bits) instead of kernel arguments, so one captured CUDA graph of a step
// replays for every token; gen_advance_k moves the position on at the end of a step.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace g2 {

static inline unsigned gcdiv(size_t a, size_t b) { return (unsigned)((a + b - 1) / b); }
static inline unsigned grid_for(size_t n, int threads) {
    return (unsigned)std::min<size_t>(gcdiv(n, threads), (size_t)148 * 16);
}

// x[r] = wte[ids[b, t0+i]] + wpe[t0+i] for row r = b*n + i (llm.c §1.1 at a position offset).
template <typename T>
__global__ void gen_embed_k(T* x, const int32_t* ids, const T* wte, const T* wpe, int B, int n, int t0,
                            int maxT, int C, const int* dstate) {
    G2_PDL_ENTRY();
    if (dstate) t0 = dstate[0];
    const size_t total = (size_t)B * n * C;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
        const size_t r = e / C;
        const int c = (int)(e - r * C);
        const int b = (int)(r / n), i = (int)(r - (size_t)b * n);
        const int t = t0 + i;
        const int tok = ids[(size_t)b * maxT + t];
        x[e] = from_f<T>(to_f(wte[(size_t)tok * C + c]) + to_f(wpe[(size_t)t * C + c]));
    }
}

// kv[b, t0+i, :] = the key and value parts of qkv row b*n + i.
template <typename T>
__global__ void gen_kv_append_k(T* kv, const T* qkv, int B, int n, int t0, int maxT, int C, const int* dstate) {
    G2_PDL_ENTRY();
    if (dstate) t0 = dstate[0];
    const size_t C2 = 2 * (size_t)C, total = (size_t)B * n * C2;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
        const size_t r = e / C2;
        const size_t j = e - r * C2;
        const int b = (int)(r / n), i = (int)(r - (size_t)b * n);
        kv[((size_t)b * maxT + t0 + i) * C2 + j] = qkv[r * 3 * C + C + j];
    }
}

// Fixed-order block reductions (warp shuffles, then the warps' values in warp order).
template <bool MAX>
__device__ float block_reduce(float v, float* red) {
    v = MAX ? warp_max(v) : warp_sum(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = red[0];
    for (int w = 1; w < nw; w++) r = MAX ? fmaxf(r, red[w]) : r + red[w];
    __syncthreads();
    return r;
}

// Attention of the new queries (llm.c §1.7 for one query row): one CTA per (b, h, new
// position i).  Scores q.k_j / sqrt(hs) for the cached positions j <= t = t0 + i go to
// shared memory, then the softmax (max, exponentials, sum in a fixed order) and the
// weighted sum of the cached values, split over groups of keys and added in group order.
constexpr int GA_THREADS = 128;

template <typename T>
__global__ void __launch_bounds__(GA_THREADS) gen_attn_k(T* out, const T* qkv, const T* kv, int n, int t0,
                                                         int maxT, int C, int NH, const int* dstate) {
    G2_PDL_ENTRY();
    extern __shared__ float gsh[];  // q[hs] | scores[t0 + n] | red[32] | part[GA_THREADS]
    if (dstate) t0 = dstate[0];
    const int hs = C / NH;
    const int b = blockIdx.x / NH, h = blockIdx.x - b * NH;
    const int i = blockIdx.y, t = t0 + i;
    const size_t r = (size_t)b * n + i;
    float* q = gsh;
    float* sc = q + hs;
    float* red = sc + (t0 + n);
    float* part = red + 32;
    for (int d = threadIdx.x; d < hs; d += GA_THREADS) q[d] = to_f(qkv[r * 3 * C + (size_t)h * hs + d]);
    __syncthreads();
    const float scale = 1.0f / sqrtf((float)hs);
    const size_t C2 = 2 * (size_t)C;
    const T* kbase = kv + (size_t)b * maxT * C2 + (size_t)h * hs;  // key j at kbase + j*C2, value at +C
    float mx = -INFINITY;
    for (int j = threadIdx.x; j <= t; j += GA_THREADS) {
        const T* k = kbase + (size_t)j * C2;
        float s = 0.f;
        for (int d = 0; d < hs; d++) s += q[d] * to_f(k[d]);
        s *= scale;
        sc[j] = s;
        mx = fmaxf(mx, s);
    }
    mx = block_reduce<true>(mx, red);
    float sum = 0.f;
    for (int j = threadIdx.x; j <= t; j += GA_THREADS) {
        const float e = expf(sc[j] - mx);
        sc[j] = e;
        sum += e;
    }
    sum = block_reduce<false>(sum, red);  // its barrier also publishes sc[]
    const float inv = 1.0f / sum;
    for (int dc = 0; dc < hs; dc += GA_THREADS) {
        const int w = min(GA_THREADS, hs - dc);
        const int G = GA_THREADS / w;
        const int d = dc + threadIdx.x % w, g = threadIdx.x / w;
        float acc = 0.f;
        if (g < G) {
            const T* v = kbase + C + d;
            for (int j = g; j <= t; j += G) acc += sc[j] * to_f(v[(size_t)j * C2]);
        }
        part[threadIdx.x] = acc;
        __syncthreads();
        if (threadIdx.x < w) {
            float a = 0.f;
            for (int gg = 0; gg < G; gg++) a += part[gg * w + threadIdx.x];
            out[r * C + (size_t)h * hs + d] = from_f<T>(a * inv);
        }
        __syncthreads();
    }
}

// last[b] = x[b*n + n-1]
template <typename T>
__global__ void gen_last_rows_k(T* last, const T* x, int B, int n, int C) {
    G2_PDL_ENTRY();
    const size_t total = (size_t)B * C;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
        const size_t b = e / C, c = e - b * C;
        last[e] = x[(b * n + n - 1) * C + c];
    }
}

// The next id of sequence b = blockIdx.x from its logits row (V real columns of Vp):
//  temperature <= 0: argmax, the first index among equal maxima (numpy's argmax);
//  temperature > 0: sample_mult over softmax(logit / temperature) with the coin
//  coins[b*n_new + step]: the first id whose cumulative probability exceeds the coin,
//  the last id if rounding leaves the coin above every cumulative value.  Each thread
//  owns one contiguous chunk of ids; thread 0 adds the chunk totals in id order and
//  walks the chunk holding the coin, so the cumulative sums follow id order.
// Writes ids[b, t_next] (when t_next < maxT) and out[b, step].
constexpr int GS_THREADS = 1024;

template <typename T>
__global__ void __launch_bounds__(GS_THREADS) gen_sample_k(int32_t* ids, int32_t* out, const T* logits, int V, int Vp,
                                                           float temperature, const float* coins, int step,
                                                           int n_new, int t_next, int maxT, const int* dstate) {
    G2_PDL_ENTRY();
    if (dstate) {
        t_next = dstate[0] + 1;
        step = dstate[1];
        n_new = dstate[2];
        temperature = __int_as_float(dstate[3]);
    }
    __shared__ float red[32];
    __shared__ int redi[32];
    __shared__ float csum[GS_THREADS];
    __shared__ int chosen;
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T* l = logits + (size_t)b * Vp;
    if (temperature <= 0.f) {
        float best = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = tid; i < V; i += GS_THREADS) {
            const float v = to_f(l[i]);
            if (v > best) {  // ids rise along a thread's walk: the first maximum stays
                best = v;
                bi = i;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > best || (ov == best && oi < bi)) {
                best = ov;
                bi = oi;
            }
        }
        if (lane == 0) {
            red[warp] = best;
            redi[warp] = bi;
        }
        __syncthreads();
        if (tid == 0) {
            float bv = red[0];
            int bx = redi[0];
            for (int w = 1; w < GS_THREADS / 32; w++)
                if (red[w] > bv || (red[w] == bv && redi[w] < bx)) {
                    bv = red[w];
                    bx = redi[w];
                }
            chosen = bx == 0x7fffffff ? 0 : bx;  // all -inf/NaN logits: id 0
        }
    } else {
        const int chunk = (V + GS_THREADS - 1) / GS_THREADS;
        const int lo = min(V, tid * chunk), hi = min(V, lo + chunk);
        float mx = -INFINITY;
        for (int i = lo; i < hi; i++) mx = fmaxf(mx, to_f(l[i]) / temperature);
        mx = block_reduce<true>(mx, red);
        float s = 0.f;
        for (int i = lo; i < hi; i++) s += expf(to_f(l[i]) / temperature - mx);
        csum[tid] = s;
        __syncthreads();
        if (tid == 0) {
            float total = 0.f;
            for (int k = 0; k < GS_THREADS; k++) total += csum[k];
            const float target = coins[(size_t)b * n_new + step] * total;
            int pick = V - 1;
            float acc = 0.f;
            for (int k = 0; k < GS_THREADS; k++) {
                if (target < acc + csum[k]) {
                    const int klo = min(V, k * chunk), khi = min(V, klo + chunk);
                    pick = khi - 1;
                    for (int i = klo; i < khi; i++) {
                        acc += expf(to_f(l[i]) / temperature - mx);
                        if (target < acc) {
                            pick = i;
                            break;
                        }
                    }
                    break;
                }
                acc += csum[k];
            }
            chosen = pick;
        }
    }
    __syncthreads();
    if (tid == 0) {
        if (t_next < maxT) ids[(size_t)b * maxT + t_next] = chosen;
        out[(size_t)b * n_new + step] = chosen;
    }
}

// End of a one-token step: the next step extends the following position.
__global__ void gen_advance_k(int* dstate) {
    G2_PDL_ENTRY();
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        dstate[0] += 1;
        dstate[1] += 1;
    }
}

// ------------------------------------------------------------------ launchers
cudaError_t gen_embed(ActType at, void* x, const int32_t* ids, const void* wte, const void* wpe, int B, int n, int t0,
                      int maxT, int C, const int* dstate, cudaStream_t s) {
    const unsigned g = grid_for((size_t)B * n * C, 256);
    if (at == ACT_BF16)
        ::g2::launch_k(gen_embed_k<bf16>, g, 256, 0, s, (bf16*)x, ids, (const bf16*)wte, (const bf16*)wpe, B, n, t0,
                                                     maxT, C, dstate);
    else
        ::g2::launch_k(gen_embed_k<float>, g, 256, 0, s, (float*)x, ids, (const float*)wte, (const float*)wpe, B, n,
                                                      t0, maxT, C, dstate);
    return cudaGetLastError();
}

cudaError_t gen_kv_append(ActType at, void* kv, const void* qkv, int B, int n, int t0, int maxT, int C,
                          const int* dstate, cudaStream_t s) {
    const unsigned g = grid_for((size_t)B * n * 2 * C, 256);
    if (at == ACT_BF16)
        ::g2::launch_k(gen_kv_append_k<bf16>, g, 256, 0, s, (bf16*)kv, (const bf16*)qkv, B, n, t0, maxT, C, dstate);
    else
        ::g2::launch_k(gen_kv_append_k<float>, g, 256, 0, s, (float*)kv, (const float*)qkv, B, n, t0, maxT, C,
                                                           dstate);
    return cudaGetLastError();
}

size_t gen_attn_smem_bytes(int C, int NH, int maxT) {
    return ((size_t)(C / NH) + (size_t)maxT + 32 + GA_THREADS) * sizeof(float);
}

cudaError_t gen_attention(ActType at, void* out, const void* qkv, const void* kv, int B, int n, int t0, int maxT,
                          int C, int NH, const int* dstate, cudaStream_t s) {
    // with the position in device memory the scores are sized for the longest cache
    const size_t smem = gen_attn_smem_bytes(C, NH, dstate ? maxT : t0 + n);
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    static bool attr_done[2] = {false, false};
    const int ti = at == ACT_BF16 ? 1 : 0;
    if (!attr_done[ti]) {
        cudaError_t e = at == ACT_BF16
                            ? cudaFuncSetAttribute(gen_attn_k<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   227 * 1024)
                            : cudaFuncSetAttribute(gen_attn_k<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   227 * 1024);
        if (e != cudaSuccess) return e;
        attr_done[ti] = true;
    }
    dim3 g((unsigned)(B * NH), (unsigned)n);
    if (at == ACT_BF16)
        ::g2::launch_k(gen_attn_k<bf16>, g, GA_THREADS, smem, s, (bf16*)out, (const bf16*)qkv, (const bf16*)kv, n, t0,
                                                              maxT, C, NH, dstate);
    else
        ::g2::launch_k(gen_attn_k<float>, g, GA_THREADS, smem, s, (float*)out, (const float*)qkv, (const float*)kv, n,
                                                               t0, maxT, C, NH, dstate);
    return cudaGetLastError();
}

cudaError_t gen_last_rows(ActType at, void* last, const void* x, int B, int n, int C, cudaStream_t s) {
    const unsigned g = grid_for((size_t)B * C, 256);
    if (at == ACT_BF16)
        ::g2::launch_k(gen_last_rows_k<bf16>, g, 256, 0, s, (bf16*)last, (const bf16*)x, B, n, C);
    else
        ::g2::launch_k(gen_last_rows_k<float>, g, 256, 0, s, (float*)last, (const float*)x, B, n, C);
    return cudaGetLastError();
}

cudaError_t gen_sample(ActType at, int32_t* ids, int32_t* out, const void* logits, int B, int V, int Vp,
                       float temperature, const float* coins, int step, int n_new, int t_next, int maxT,
                       const int* dstate, cudaStream_t s) {
    if (at == ACT_BF16)
        ::g2::launch_k(gen_sample_k<bf16>, B, GS_THREADS, 0, s, ids, out, (const bf16*)logits, V, Vp, temperature,
                                                             coins, step, n_new, t_next, maxT, dstate);
    else
        ::g2::launch_k(gen_sample_k<float>, B, GS_THREADS, 0, s, ids, out, (const float*)logits, V, Vp, temperature,
                                                              coins, step, n_new, t_next, maxT, dstate);
    return cudaGetLastError();
}

cudaError_t gen_advance(int* dstate, cudaStream_t s) {
    ::g2::launch_k(gen_advance_k, 1, 32, 0, s, dstate);
    return cudaGetLastError();
}

}  // namespace g2
