// TF32 products around the tensor-core kernel: operands that are not K-major are packed
// K-major first (the TF32 MMA reads K-major operands here), and the epilogues the bf16
// kernel fuses (residual add, GELU, GELU') run as fp32 elementwise passes afterwards.
// The contraction itself is the llm.c annotated listing's matmul (§1.5 forward, §1.6
// backward) with TF32 operand rounding and fp32 accumulation.
#include <algorithm>

#include "common.cuh"
#include "dispatch.h"
#include "gemm_tc.h"
#include "kernels.h"

namespace g2 {

namespace {

// out (cols, rows) = in (rows, cols)^T, in row stride ld_in, out dense: 32x32 tiles
// through shared memory (padded against bank conflicts), reads and writes coalesced.
__global__ void __launch_bounds__(256) transpose_f32_k(float* out, const float* in, int rows, int cols,
                                                        long long ld_in) {
    G2_PDL_ENTRY();
    __shared__ float t[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int i = ty; i < 32; i += 8) {
        const int r = r0 + i, c = c0 + tx;
        if (r < rows && c < cols) t[i][tx] = in[(size_t)r * ld_in + c];
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int c = c0 + i, r = r0 + tx;
        if (r < rows && c < cols) out[(size_t)c * rows + r] = t[tx][i];
    }
}

// mode 0: D += R; mode 1: D2 = gelu(D); mode 2: D *= gelu'(P)
__global__ void tf32_epilogue_k(float* D, long long ldd, int M, int N, const float* R, long long ldr, float* D2,
                                long long ldd2, const float* P, long long ldp, int mode) {
    G2_PDL_ENTRY();
    const size_t n = (size_t)M * N;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t m = i / N, c = i % N;
        float* d = D + m * ldd + c;
        if (mode == 0)
            *d += R[m * ldr + c];
        else if (mode == 1)
            D2[m * ldd2 + c] = gelu_tanh(*d);
        else
            *d *= gelu_tanh_grad(P[m * ldp + c]);
    }
}

unsigned grid_for(size_t n) { return (unsigned)std::min<size_t>((n + 255) / 256, 148 * 16); }

}  // namespace

size_t gemm_tf32_pack_bytes(int M, int N, int K, bool a_kmajor, bool b_kmajor) {
    size_t f = (a_kmajor ? 0 : (size_t)M * K) + (b_kmajor ? 0 : (size_t)N * K);
    return f ? (f * 4 + 255) / 256 * 256 + 256 : 0;
}

cudaError_t gemm_dispatch_tf32(const GemmArgs& a0, float* ws, size_t ws_bytes, cudaStream_t s) {
    GemmArgs a = a0;
    float* pk = a0.tws;
    size_t left = a0.tws ? a0.tws_bytes : 0;
    auto pack = [&](const void* src, int rows_out, int K, long long ld_in, const void** dst) -> bool {
        // src holds the operand as (K, rows_out) with row stride ld_in; dst gets (rows_out, K)
        const size_t bytes = (size_t)rows_out * K * 4;
        if (!pk || left < bytes) return false;
        dim3 g((rows_out + 31) / 32, (K + 31) / 32);
        ::g2::launch_k(transpose_f32_k, g, 256, 0, s, pk, (const float*)src, K, rows_out, ld_in);
        *dst = pk;
        const size_t adv = (bytes + 255) / 256 * 256;
        pk = (float*)((char*)pk + adv);
        left = left > adv ? left - adv : 0;
        return true;
    };
    bool ok = true;
    if (a.sAk != 1 && a.sAm == 1) {
        ok = pack(a0.A, a0.M, a0.K, a0.sAk, &a.A);
        a.sAm = a.K;
        a.sAk = 1;
    }
    if (ok && a.sBk != 1 && a.sBn == 1) {
        ok = pack(a0.B, a0.N, a0.K, a0.sBk, &a.B);
        a.sBn = a.K;
        a.sBk = 1;
    }
    // the tensor-core kernel computes acc (+ bias) into fp32 D; the rest follows
    GemmArgs t = a;
    t.d_f32 = 1;
    t.R = nullptr;
    t.D2 = nullptr;
    t.P = nullptr;
    t.epi = EPI_STORE;
    if (a0.epi == EPI_GELU_BWD) t.bias = nullptr;
    if (!ok || !gemm_tc_supported(t)) {
        gemm_tc_note_variant("simt");
        return gemm_simt(a0, s);  // exact fp32 on the original operands
    }
    cudaError_t e = gemm_tc(t, ws, ws_bytes, a0.flags, s);
    if (e != cudaSuccess) return e;
    const size_t n = (size_t)a0.M * a0.N;
    if (a0.epi == EPI_STORE && a0.R)
        ::g2::launch_k(tf32_epilogue_k, grid_for(n), 256, 0, s, (float*)a0.D, a0.ldd, a0.M, a0.N, (const float*)a0.R,
                                                             a0.ldr, nullptr, 0, nullptr, 0, 0);
    else if (a0.epi == EPI_GELU)
        ::g2::launch_k(tf32_epilogue_k, grid_for(n), 256, 0, s, (float*)a0.D, a0.ldd, a0.M, a0.N, nullptr, 0,
                                                             (float*)a0.D2, a0.ldd2, nullptr, 0, 1);
    else if (a0.epi == EPI_GELU_BWD)
        ::g2::launch_k(tf32_epilogue_k, grid_for(n), 256, 0, s, (float*)a0.D, a0.ldd, a0.M, a0.N, nullptr, 0, nullptr,
                                                             0, (const float*)a0.P, a0.ldp, 2);
    else
        return cudaSuccess;
    return cudaGetLastError();
}

}  // namespace g2
