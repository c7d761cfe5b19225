// Causal multi-head attention, SIMT form (any head size, fp32 or bf16 storage, fp32 math).
//
// Forward (llm.c annotated listing §1.7; picoGPT attention with causal_mask): one warp
// per (b, t, h) query row.  Scores q.k/sqrt(hs) for keys t2 <= t are taken 32 keys at a
// time (lane j scores key t0+j), folded into a running max and sum (online softmax), and
// the value rows are accumulated with lanes owning output channels.  The row's
// log-sum-exp is kept so the backward can rebuild the softmax without storing it.
//
// Backward (llm.c §1.8): with P = exp(S - lse) rebuilt from the saved lse and
// D = rowsum(dO * O), dS = P * (dO.v - D) is the softmax-Jacobian product of the listing.
// dq is gathered per query row; dk and dv per key row (queries t >= t2).  No atomics.
#include "common.cuh"
#include "kernels.h"

namespace g2 {

static const int ATT_MAX_HS = 256;

template <typename T>
__global__ void attn_fwd_simt_k(T* out, float* lse, const T* qkv, int B, int Tn, int C, int NH) {
    G2_PDL_ENTRY();
    __shared__ float s_q[8][ATT_MAX_HS];
    int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    long long gid = (long long)blockIdx.x * 8 + warp;  // ((b*NH + h)*T + t)
    if (gid >= (long long)B * NH * Tn) return;
    int t = (int)(gid % Tn), h = (int)((gid / Tn) % NH), b = (int)(gid / ((long long)Tn * NH));
    int hs = C / NH, C3 = 3 * C;
    float scale = 1.0f / sqrtf((float)hs);
    const T* base = qkv + (size_t)b * Tn * C3;
    const T* q = base + (size_t)t * C3 + h * hs;
    for (int d = lane; d < hs; d += 32) s_q[warp][d] = to_f(q[d]);
    __syncwarp();
    const int ND = ATT_MAX_HS / 32;
    float acc[ND];
#pragma unroll
    for (int i = 0; i < ND; i++) acc[i] = 0.f;
    float m = -INFINITY, l = 0.f;
    for (int t0 = 0; t0 <= t; t0 += 32) {
        int t2 = t0 + lane;
        float sc = -INFINITY;
        if (t2 <= t) {
            const T* k = base + (size_t)t2 * C3 + C + h * hs;
            float dot = 0.f;
            for (int d = 0; d < hs; d++) dot += s_q[warp][d] * to_f(k[d]);
            sc = dot * scale;
        }
        float mnew = fmaxf(m, warp_max(sc));
        float p = t2 <= t ? expf(sc - mnew) : 0.f;
        float corr = expf(m - mnew);
        l = l * corr + warp_sum(p);
#pragma unroll
        for (int i = 0; i < ND; i++) acc[i] *= corr;
        int nk = min(32, t - t0 + 1);
        for (int j = 0; j < nk; j++) {
            float pj = __shfl_sync(0xffffffffu, p, j);
            const T* v = base + (size_t)(t0 + j) * C3 + 2 * C + h * hs;
#pragma unroll
            for (int i = 0; i < ND; i++) {
                int d = lane + 32 * i;
                if (d < hs) acc[i] += pj * to_f(v[d]);
            }
        }
        m = mnew;
    }
    T* o = out + ((size_t)b * Tn + t) * C + h * hs;
    float inv = 1.0f / l;
#pragma unroll
    for (int i = 0; i < ND; i++) {
        int d = lane + 32 * i;
        if (d < hs) o[d] = from_f<T>(acc[i] * inv);
    }
    if (lane == 0) lse[gid] = m + logf(l);
}

// D[b,h,t] = sum_d dO[b,t,h,d] * O[b,t,h,d]
template <typename T>
__global__ void attn_bwd_dot_k(float* D, const T* dout, const T* out, int B, int Tn, int C, int NH) {
    G2_PDL_ENTRY();
    int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    long long gid = (long long)blockIdx.x * 8 + warp;
    if (gid >= (long long)B * NH * Tn) return;
    int t = (int)(gid % Tn), h = (int)((gid / Tn) % NH), b = (int)(gid / ((long long)Tn * NH));
    int hs = C / NH;
    const T* a = dout + ((size_t)b * Tn + t) * C + h * hs;
    const T* o = out + ((size_t)b * Tn + t) * C + h * hs;
    float s = 0.f;
    for (int d = lane; d < hs; d += 32) s += to_f(a[d]) * to_f(o[d]);
    s = warp_sum(s);
    if (lane == 0) D[gid] = s;
}

// dq for query row t: sum over t2 <= t of dS[t,t2] * k[t2] * scale.
template <typename T>
__global__ void attn_bwd_dq_simt_k(T* dqkv, const T* dout, const T* qkv, const float* lse,
                                   const float* D, int B, int Tn, int C, int NH) {
    G2_PDL_ENTRY();
    __shared__ float s_q[8][ATT_MAX_HS];
    __shared__ float s_do[8][ATT_MAX_HS];
    int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    long long gid = (long long)blockIdx.x * 8 + warp;
    if (gid >= (long long)B * NH * Tn) return;
    int t = (int)(gid % Tn), h = (int)((gid / Tn) % NH), b = (int)(gid / ((long long)Tn * NH));
    int hs = C / NH, C3 = 3 * C;
    float scale = 1.0f / sqrtf((float)hs);
    const T* base = qkv + (size_t)b * Tn * C3;
    const T* q = base + (size_t)t * C3 + h * hs;
    const T* dO = dout + ((size_t)b * Tn + t) * C + h * hs;
    for (int d = lane; d < hs; d += 32) {
        s_q[warp][d] = to_f(q[d]);
        s_do[warp][d] = to_f(dO[d]);
    }
    __syncwarp();
    float L = lse[gid], Dt = D[gid];
    const int ND = ATT_MAX_HS / 32;
    float acc[ND];
#pragma unroll
    for (int i = 0; i < ND; i++) acc[i] = 0.f;
    for (int t0 = 0; t0 <= t; t0 += 32) {
        int t2 = t0 + lane;
        float ds = 0.f;
        if (t2 <= t) {
            const T* k = base + (size_t)t2 * C3 + C + h * hs;
            const T* v = base + (size_t)t2 * C3 + 2 * C + h * hs;
            float sdot = 0.f, pdot = 0.f;
            for (int d = 0; d < hs; d++) {
                sdot += s_q[warp][d] * to_f(k[d]);
                pdot += s_do[warp][d] * to_f(v[d]);
            }
            float p = expf(sdot * scale - L);
            ds = p * (pdot - Dt);
        }
        int nk = min(32, t - t0 + 1);
        for (int j = 0; j < nk; j++) {
            float dsj = __shfl_sync(0xffffffffu, ds, j);
            const T* k = base + (size_t)(t0 + j) * C3 + C + h * hs;
#pragma unroll
            for (int i = 0; i < ND; i++) {
                int d = lane + 32 * i;
                if (d < hs) acc[i] += dsj * to_f(k[d]);
            }
        }
    }
    T* dq = dqkv + ((size_t)b * Tn + t) * C3 + h * hs;
#pragma unroll
    for (int i = 0; i < ND; i++) {
        int d = lane + 32 * i;
        if (d < hs) dq[d] = from_f<T>(acc[i] * scale);
    }
}

// dk, dv for key row t2: sums over queries t >= t2.
template <typename T>
__global__ void attn_bwd_dkv_simt_k(T* dqkv, const T* dout, const T* qkv, const float* lse,
                                    const float* D, int B, int Tn, int C, int NH) {
    G2_PDL_ENTRY();
    __shared__ float s_k[8][ATT_MAX_HS];
    __shared__ float s_v[8][ATT_MAX_HS];
    int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    long long gid = (long long)blockIdx.x * 8 + warp;
    if (gid >= (long long)B * NH * Tn) return;
    int t2 = (int)(gid % Tn), h = (int)((gid / Tn) % NH), b = (int)(gid / ((long long)Tn * NH));
    int hs = C / NH, C3 = 3 * C;
    float scale = 1.0f / sqrtf((float)hs);
    const T* base = qkv + (size_t)b * Tn * C3;
    const T* k = base + (size_t)t2 * C3 + C + h * hs;
    const T* v = base + (size_t)t2 * C3 + 2 * C + h * hs;
    for (int d = lane; d < hs; d += 32) {
        s_k[warp][d] = to_f(k[d]);
        s_v[warp][d] = to_f(v[d]);
    }
    __syncwarp();
    const float* lse_bh = lse + ((size_t)b * NH + h) * Tn;
    const float* D_bh = D + ((size_t)b * NH + h) * Tn;
    const int ND = ATT_MAX_HS / 32;
    float dk[ND], dv[ND];
#pragma unroll
    for (int i = 0; i < ND; i++) dk[i] = dv[i] = 0.f;
    for (int t0 = t2; t0 < Tn; t0 += 32) {
        int t = t0 + lane;
        float p = 0.f, ds = 0.f;
        if (t < Tn) {
            const T* q = base + (size_t)t * C3 + h * hs;
            const T* dO = dout + ((size_t)b * Tn + t) * C + h * hs;
            float sdot = 0.f, pdot = 0.f;
            for (int d = 0; d < hs; d++) {
                sdot += to_f(q[d]) * s_k[warp][d];
                pdot += to_f(dO[d]) * s_v[warp][d];
            }
            p = expf(sdot * scale - lse_bh[t]);
            ds = p * (pdot - D_bh[t]);
        }
        int nq = min(32, Tn - t0);
        for (int j = 0; j < nq; j++) {
            float pj = __shfl_sync(0xffffffffu, p, j);
            float dsj = __shfl_sync(0xffffffffu, ds, j);
            const T* q = base + (size_t)(t0 + j) * C3 + h * hs;
            const T* dO = dout + ((size_t)b * Tn + t0 + j) * C + h * hs;
#pragma unroll
            for (int i = 0; i < ND; i++) {
                int d = lane + 32 * i;
                if (d < hs) {
                    dv[i] += pj * to_f(dO[d]);
                    dk[i] += dsj * to_f(q[d]);
                }
            }
        }
    }
    T* dkp = dqkv + ((size_t)b * Tn + t2) * C3 + C + h * hs;
    T* dvp = dkp + C;
#pragma unroll
    for (int i = 0; i < ND; i++) {
        int d = lane + 32 * i;
        if (d < hs) {
            dkp[d] = from_f<T>(dk[i] * scale);
            dvp[d] = from_f<T>(dv[i]);
        }
    }
}

static inline unsigned rows8(long long n) { return (unsigned)((n + 7) / 8); }

cudaError_t attention_forward_simt(ActType at, void* out, float* lse, const void* qkv, int B, int T,
                                   int C, int NH, cudaStream_t s) {
    if (C % NH || C / NH > ATT_MAX_HS) return cudaErrorInvalidValue;
    long long n = (long long)B * NH * T;
    if (n <= 0) return cudaSuccess;
    if (at == ACT_BF16)
        ::g2::launch_k(attn_fwd_simt_k<bf16>, rows8(n), 256, 0, s, (bf16*)out, lse, (const bf16*)qkv, B, T, C, NH);
    else
        ::g2::launch_k(attn_fwd_simt_k<float>, rows8(n), 256, 0, s, (float*)out, lse, (const float*)qkv, B, T, C, NH);
    return cudaGetLastError();
}

cudaError_t attention_bwd_dot(ActType at, float* D, const void* dout, const void* out, int B, int T,
                              int C, int NH, cudaStream_t s) {
    long long n = (long long)B * NH * T;
    if (n <= 0) return cudaSuccess;
    if (at == ACT_BF16)
        ::g2::launch_k(attn_bwd_dot_k<bf16>, rows8(n), 256, 0, s, D, (const bf16*)dout, (const bf16*)out, B, T, C, NH);
    else
        ::g2::launch_k(attn_bwd_dot_k<float>, rows8(n), 256, 0, s, D, (const float*)dout, (const float*)out, B, T, C, NH);
    return cudaGetLastError();
}

cudaError_t attention_backward_simt(ActType at, void* dqkv, const void* dout, const void* qkv,
                                    const void* out, const float* lse, int B, int T, int C, int NH,
                                    float* Dbuf, cudaStream_t s) {
    if (C % NH || C / NH > ATT_MAX_HS) return cudaErrorInvalidValue;
    long long n = (long long)B * NH * T;
    if (n <= 0) return cudaSuccess;
    if (at == ACT_BF16) {
        ::g2::launch_k(attn_bwd_dot_k<bf16>, rows8(n), 256, 0, s, Dbuf, (const bf16*)dout, (const bf16*)out, B, T, C, NH);
        ::g2::launch_k(attn_bwd_dq_simt_k<bf16>, rows8(n), 256, 0, s, (bf16*)dqkv, (const bf16*)dout,
                                                          (const bf16*)qkv, lse, Dbuf, B, T, C, NH);
        ::g2::launch_k(attn_bwd_dkv_simt_k<bf16>, rows8(n), 256, 0, s, (bf16*)dqkv, (const bf16*)dout,
                                                           (const bf16*)qkv, lse, Dbuf, B, T, C, NH);
    } else {
        ::g2::launch_k(attn_bwd_dot_k<float>, rows8(n), 256, 0, s, Dbuf, (const float*)dout, (const float*)out, B, T, C, NH);
        ::g2::launch_k(attn_bwd_dq_simt_k<float>, rows8(n), 256, 0, s, (float*)dqkv, (const float*)dout,
                                                           (const float*)qkv, lse, Dbuf, B, T, C, NH);
        ::g2::launch_k(attn_bwd_dkv_simt_k<float>, rows8(n), 256, 0, s, (float*)dqkv, (const float*)dout,
                                                            (const float*)qkv, lse, Dbuf, B, T, C, NH);
    }
    return cudaGetLastError();
}

}  // namespace g2
