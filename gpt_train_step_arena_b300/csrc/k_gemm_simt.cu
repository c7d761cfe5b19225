// SIMT GEMM with arbitrary operand strides and the fused epilogues of the train step.
//
// D[m,n] = epi( sum_k A(m,k) B(n,k) ).  This is the strict-fp32 contraction (every
// product and sum in fp32 FMA) used by the fp32 precision mode, and the fallback for
// shapes the tensor-core path does not take.  llm.c annotated listing §1.5/§1.6 define
// the three uses: forward out = inp . W^T + bias, dinp = dout . W, dW = dout^T . inp.
#include "common.cuh"
#include "kernels.h"

namespace g2 {

static const int SB_M = 64, SB_N = 64, SB_K = 16;

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_k(GemmArgs a) {
    G2_PDL_ENTRY();
    __shared__ float As[SB_K][SB_M + 4];
    __shared__ float Bs[SB_K][SB_N + 4];
    const T* A = (const T*)a.A;
    const T* Bm = (const T*)a.B;
    int tid = threadIdx.x;
    int m0 = blockIdx.y * SB_M, n0 = blockIdx.x * SB_N;
    int tm = (tid / 16) * 4, tn = (tid % 16) * 4;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = 0.f;
    // Loader mapping: 1024 elements per tile, 4 per thread.  When the operand is
    // contiguous along k, consecutive threads walk k; otherwise they walk m (or n).
    bool a_kfast = a.sAk == 1, b_kfast = a.sBk == 1;
    for (int k0 = 0; k0 < a.K; k0 += SB_K) {
#pragma unroll
        for (int r = 0; r < 4; r++) {
            int e = tid + r * 256;
            int mm, kk;
            if (a_kfast) { kk = e % SB_K; mm = e / SB_K; } else { mm = e % SB_M; kk = e / SB_M; }
            int gm = m0 + mm, gk = k0 + kk;
            As[kk][mm] = (gm < a.M && gk < a.K) ? to_f(A[(long long)gm * a.sAm + (long long)gk * a.sAk]) : 0.f;
            int nn;
            if (b_kfast) { kk = e % SB_K; nn = e / SB_K; } else { nn = e % SB_N; kk = e / SB_N; }
            int gn = n0 + nn;
            gk = k0 + kk;
            Bs[kk][nn] = (gn < a.N && gk < a.K) ? to_f(Bm[(long long)gn * a.sBn + (long long)gk * a.sBk]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < SB_K; kk++) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; i++) av[i] = As[kk][tm + i];
#pragma unroll
            for (int j = 0; j < 4; j++) bv[j] = Bs[kk][tn + j];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
    // epilogue
#pragma unroll
    for (int i = 0; i < 4; i++) {
        int gm = m0 + tm + i;
        if (gm >= a.M) continue;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            int gn = n0 + tn + j;
            if (gn >= a.N) continue;
            float v = acc[i][j];
            if (a.epi == EPI_GELU_BWD) {
                float pre = to_f(((const T*)a.P)[(long long)gm * a.ldp + gn]);
                v = v * gelu_tanh_grad(pre);
            } else {
                if (a.bias) v += a.bias[gn];
                if (a.R) v += to_f(((const T*)a.R)[(long long)gm * a.ldr + gn]);
            }
            if (a.d_f32)
                ((float*)a.D)[(long long)gm * a.ldd + gn] = v;
            else
                ((T*)a.D)[(long long)gm * a.ldd + gn] = from_f<T>(v);
            if (a.epi == EPI_GELU) ((T*)a.D2)[(long long)gm * a.ldd2 + gn] = from_f<T>(gelu_tanh(v));
        }
    }
}

cudaError_t gemm_simt(const GemmArgs& a, cudaStream_t s) {
    if (a.M <= 0 || a.N <= 0) return cudaSuccess;
    dim3 grid((a.N + SB_N - 1) / SB_N, (a.M + SB_M - 1) / SB_M);
    if (grid.y > 65535) return cudaErrorInvalidValue;
    if (a.in_type == ACT_BF16)
        ::g2::launch_k(gemm_simt_k<bf16>, grid, 256, 0, s, a);
    else
        ::g2::launch_k(gemm_simt_k<float>, grid, 256, 0, s, a);
    return cudaGetLastError();
}

}  // namespace g2
