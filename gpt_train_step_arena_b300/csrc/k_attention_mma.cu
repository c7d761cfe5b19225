// Causal multi-head attention on tensor cores (bf16 in, fp32 accumulate), head size 64.
//
// Forward (llm.c annotated listing §1.7; picoGPT attention with causal_mask): one CTA
// of 4 warps per (64-query tile, b, h); each warp owns 16 query rows.  Key/value tiles
// of 64 rows stream through double-buffered shared memory (cp.async); S = Q K^T and
// O += P V are m16n8k16 bf16 MMAs; the softmax is online (running max and sum per row,
// exp2 with pre-scaled scores) and only the row log-sum-exp is stored.
//
// Backward (llm.c §1.8), without atomics: P is rebuilt from the saved log-sum-exp and
// D = rowsum(dO * O);
//   key-major CTA  (64 keys):    S^T = K Q^T, dP^T = V dO^T, dS^T = P^T (dP^T - D),
//                                dV += P^T dO,  dK += dS^T Q      over query tiles >= key tile
//   query-major CTA (64 queries): S = Q K^T, dP = dO V^T, dS = P (dP - D), dQ += dS K
// so every output element is summed by one thread in a fixed order.
//
// Shared tiles are [64 rows][64 bf16] with the 16-byte chunks of row r XOR-swizzled by
// (r & 7), which keeps ldmatrix conflict-free.
#include "common.cuh"
#include "kernels.h"

namespace g2 {
namespace fa {

constexpr int HS = 64, BQ = 64, BKV = 64, NW = 4, NT = NW * 32;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

G2_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// byte offset of element (row, col) in a swizzled [64][64] bf16 tile (col multiple of 8)
G2_DEV uint32_t swz(int row, int col) {
    return (uint32_t)(row * 128 + ((((col >> 3) ^ (row & 7)) & 7) << 4));
}

G2_DEV void cp_async16(uint32_t dst, const void* src, bool valid) {
    int n = valid ? 16 : 0;  // zero-fill rows past the sequence end
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
G2_DEV void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
G2_DEV void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

G2_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
G2_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
G2_DEV void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
G2_DEV uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Copy 64 rows x 64 bf16 (rows r0.. of a strided matrix) into a swizzled tile.
G2_DEV void load_tile(uint32_t tile, const bf16* base, long long ld, int r0, int nrows, int tid) {
#pragma unroll
    for (int i = 0; i < 4; i++) {
        int e = tid + i * NT;  // 512 chunks of 16 bytes
        int row = e >> 3, ch = e & 7;
        int gr = r0 + row;
        bool ok = gr < nrows;
        const bf16* src = base + (long long)(ok ? gr : 0) * ld + ch * 8;
        cp_async16(tile + swz(row, ch * 8), src, ok);
    }
}

// A fragments (16 rows x 64 cols -> 4 k-steps) of rows [r0, r0+16) of a swizzled tile.
G2_DEV void load_a_frags(uint32_t tile, int r0, int lane, uint32_t (&a)[4][4]) {
#pragma unroll
    for (int ks = 0; ks < 4; ks++) {
        int row = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
        int col = ks * 16 + (lane >> 4) * 8;
        ldsm_x4(tile + swz(row, col), a[ks][0], a[ks][1], a[ks][2], a[ks][3]);
    }
}

// acc[16 rows][64 cols] += A(16 x 64, fragments) . T^T where T is a [64 n][64 k] tile
// stored row-major (n rows, k contiguous): B operand without transpose.
G2_DEV void mma_abT(float (&acc)[8][4], const uint32_t (&a)[4][4], uint32_t tile, int lane) {
#pragma unroll
    for (int np = 0; np < 4; np++) {      // pairs of 8-wide n tiles
#pragma unroll
        for (int ks = 0; ks < 4; ks++) {
            int row = np * 16 + (lane & 7) + (lane >> 4) * 8;
            int col = ks * 16 + ((lane >> 3) & 1) * 8;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(tile + swz(row, col), b0, b1, b2, b3);
            mma16816(acc[2 * np], a[ks], b0, b1);
            mma16816(acc[2 * np + 1], a[ks], b2, b3);
        }
    }
}

// acc[16 rows][64 cols] += P(16 x 64, C-fragment layout) . T where T is a [64 k][64 n]
// tile stored row-major (k rows, n contiguous): B operand through ldmatrix.trans.
G2_DEV void mma_pv(float (&acc)[8][4], const float (&p)[8][4], uint32_t tile, int lane) {
#pragma unroll
    for (int ks = 0; ks < 4; ks++) {
        uint32_t a[4];
        a[0] = pack_bf16(p[2 * ks][0], p[2 * ks][1]);
        a[1] = pack_bf16(p[2 * ks][2], p[2 * ks][3]);
        a[2] = pack_bf16(p[2 * ks + 1][0], p[2 * ks + 1][1]);
        a[3] = pack_bf16(p[2 * ks + 1][2], p[2 * ks + 1][3]);
#pragma unroll
        for (int np = 0; np < 4; np++) {
            int row = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            int col = np * 16 + (lane >> 4) * 8;
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(tile + swz(row, col), b0, b1, b2, b3);
            mma16816(acc[2 * np], a, b0, b1);
            mma16816(acc[2 * np + 1], a, b2, b3);
        }
    }
}

G2_DEV void zero(float (&acc)[8][4]) {
#pragma unroll
    for (int i = 0; i < 8; i++) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
}

// Store a 16 x 64 fp32 C-fragment block (times `mul`) as bf16 rows of a strided matrix.
G2_DEV void store_rows(bf16* base, long long ld, int r0, int nrows, const float (&acc)[8][4], float mul,
                       int lane) {
    int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 8; nt++) {
        int col = nt * 8 + 2 * t;
        int ra = r0 + g, rb = r0 + g + 8;
        if (ra < nrows)
            *reinterpret_cast<__nv_bfloat162*>(base + (long long)ra * ld + col) =
                __floats2bfloat162_rn(acc[nt][0] * mul, acc[nt][1] * mul);
        if (rb < nrows)
            *reinterpret_cast<__nv_bfloat162*>(base + (long long)rb * ld + col) =
                __floats2bfloat162_rn(acc[nt][2] * mul, acc[nt][3] * mul);
    }
}

// ------------------------------------------------------------------ forward
__global__ void __launch_bounds__(NT) attn_fwd_mma_k(bf16* out, float* lse, const bf16* qkv, int T, int C,
                                                      int NH) {
    __shared__ __align__(128) uint8_t sm[5 * 8192];
    const int nqt = gridDim.x;
    const int qt = nqt - 1 - blockIdx.x;  // heaviest (latest) query tiles first
    const int bh = blockIdx.y, b = bh / NH, h = bh % NH;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long ld = 3LL * C;
    const bf16* q_base = qkv + (long long)b * T * ld + h * HS;
    const bf16* k_base = q_base + C;
    const bf16* v_base = q_base + 2 * C;
    const uint32_t sQ = smem_u32(sm), sK0 = sQ + 8192, sV0 = sQ + 16384;  // K,V double buffers
    const int q0 = qt * BQ;
    const float sl2 = LOG2E / sqrtf((float)HS);  // scores to log2 units

    load_tile(sQ, q_base, ld, q0, T, tid);
    load_tile(sK0, k_base, ld, 0, T, tid);
    load_tile(sV0, v_base, ld, 0, T, tid);
    cp_commit();

    float o[8][4];
    zero(o);
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    uint32_t qa[4][4];
    const int g = lane >> 2, t4 = lane & 3;
    const int nkv = qt + 1;
    for (int j = 0; j < nkv; j++) {
        const int buf = j & 1;
        if (j + 1 < nkv) {
            const int nb = buf ^ 1;
            load_tile(sK0 + nb * 16384, k_base, ld, (j + 1) * BKV, T, tid);
            load_tile(sV0 + nb * 16384, v_base, ld, (j + 1) * BKV, T, tid);
        }
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        if (j == 0) load_a_frags(sQ, warp * 16, lane, qa);
        const uint32_t sK = sK0 + buf * 16384, sV = sV0 + buf * 16384;
        float s[8][4];
        zero(s);
        mma_abT(s, qa, sK, lane);
        // scale, causal mask on the diagonal tile, online softmax (rows g and g+8)
        const int qa_row = q0 + warp * 16 + g, qb_row = qa_row + 8;
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
            int key = j * BKV + nt * 8 + 2 * t4;
#pragma unroll
            for (int e = 0; e < 4; e++) {
                int kk = key + (e & 1);
                int qq = e < 2 ? qa_row : qb_row;
                float v = s[nt][e] * sl2;
                if (j == qt && kk > qq) v = -INFINITY;
                s[nt][e] = v;
                mx[e >> 1] = fmaxf(mx[e >> 1], v);
            }
        }
#pragma unroll
        for (int r = 0; r < 2; r++) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        }
        float mnew[2], corr[2], rs[2] = {0.f, 0.f};
#pragma unroll
        for (int r = 0; r < 2; r++) {
            mnew[r] = fmaxf(mrow[r], mx[r]);
            corr[r] = exp2f(mrow[r] - mnew[r]);  // 0 on the first tile (mrow = -inf)
        }
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                float p = exp2f(s[nt][e] - mnew[e >> 1]);
                s[nt][e] = p;
                rs[e >> 1] += p;
            }
        }
#pragma unroll
        for (int r = 0; r < 2; r++) {
            rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 1);
            rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 2);
            lrow[r] = lrow[r] * corr[r] + rs[r];
            mrow[r] = mnew[r];
        }
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
            o[nt][0] *= corr[0];
            o[nt][1] *= corr[0];
            o[nt][2] *= corr[1];
            o[nt][3] *= corr[1];
        }
        mma_pv(o, s, sV, lane);
        __syncthreads();  // this buffer is refilled two iterations on
    }
    // normalise and store
    const int r0 = q0 + warp * 16;
    bf16* obase = out + (long long)b * T * C + h * HS;
#pragma unroll
    for (int nt = 0; nt < 8; nt++) {
        o[nt][0] /= lrow[0];
        o[nt][1] /= lrow[0];
        o[nt][2] /= lrow[1];
        o[nt][3] /= lrow[1];
    }
    store_rows(obase, C, r0, T, o, 1.0f, lane);
    if (t4 == 0) {
        float* lb = lse + (long long)bh * T;
        if (r0 + g < T) lb[r0 + g] = (mrow[0] + log2f(lrow[0])) * LN2;
        if (r0 + g + 8 < T) lb[r0 + g + 8] = (mrow[1] + log2f(lrow[1])) * LN2;
    }
}

// ------------------------------------------------------------------ backward: dK, dV
__global__ void __launch_bounds__(NT) attn_bwd_dkv_mma_k(bf16* dqkv, const bf16* dout, const bf16* qkv,
                                                          const float* lse, const float* Dv, int T, int C,
                                                          int NH) {
    __shared__ __align__(128) uint8_t sm[6 * 8192];
    const int nkt = gridDim.x;
    const int kt = blockIdx.x;  // key tile; the lightest (last) tiles finish first anyway
    const int bh = blockIdx.y, b = bh / NH, h = bh % NH;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long ld = 3LL * C;
    const bf16* q_base = qkv + (long long)b * T * ld + h * HS;
    const bf16* k_base = q_base + C;
    const bf16* v_base = q_base + 2 * C;
    const bf16* do_base = dout + (long long)b * T * C + h * HS;
    const float* lse_bh = lse + (long long)bh * T;
    const float* D_bh = Dv + (long long)bh * T;
    // sK, sV: this CTA's keys; sQ/sdO double buffered
    const uint32_t sK = smem_u32(sm), sV = sK + 8192, sQ0 = sK + 16384, sO0 = sK + 32768;
    const int k0 = kt * BKV;
    const float scale = 1.0f / sqrtf((float)HS), sl2 = scale * LOG2E;
    (void)nkt;

    load_tile(sK, k_base, ld, k0, T, tid);
    load_tile(sV, v_base, ld, k0, T, tid);
    load_tile(sQ0, q_base, ld, k0, T, tid);
    load_tile(sO0, do_base, C, k0, T, tid);
    cp_commit();

    uint32_t ka[4][4], va[4][4];
    float dk[8][4], dv[8][4];
    zero(dk);
    zero(dv);
    const int g = lane >> 2, t4 = lane & 3;
    const int nqt = (T + BQ - 1) / BQ;
    const int key_a = k0 + warp * 16 + g, key_b = key_a + 8;  // this thread's key rows
    for (int i = kt, it = 0; i < nqt; i++, it++) {
        const int buf = it & 1;
        if (i + 1 < nqt) {
            load_tile(sQ0 + (buf ^ 1) * 8192, q_base, ld, (i + 1) * BQ, T, tid);
            load_tile(sO0 + (buf ^ 1) * 8192, do_base, C, (i + 1) * BQ, T, tid);
        }
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        if (it == 0) {
            load_a_frags(sK, warp * 16, lane, ka);
            load_a_frags(sV, warp * 16, lane, va);
        }
        const uint32_t sQ = sQ0 + buf * 8192, sO = sO0 + buf * 8192;
        float st[8][4], dpt[8][4];
        zero(st);
        zero(dpt);
        mma_abT(st, ka, sQ, lane);   // S^T = K Q^T   (keys x queries)
        mma_abT(dpt, va, sO, lane);  // dP^T = V dO^T
        const int qbase = i * BQ;
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
            int qc = qbase + nt * 8 + 2 * t4;
#pragma unroll
            for (int e = 0; e < 4; e++) {
                int qq = qc + (e & 1);
                int kk = e < 2 ? key_a : key_b;
                float L = qq < T ? lse_bh[qq] : 0.f;
                float Dq = qq < T ? D_bh[qq] : 0.f;
                float p = (qq < T && qq >= kk) ? exp2f(st[nt][e] * sl2 - L * LOG2E) : 0.f;
                st[nt][e] = p;                         // P^T
                dpt[nt][e] = p * (dpt[nt][e] - Dq);    // dS^T (unscaled)
            }
        }
        mma_pv(dv, st, sO, lane);   // dV += P^T dO
        mma_pv(dk, dpt, sQ, lane);  // dK += dS^T Q
        __syncthreads();
    }
    bf16* dk_base = dqkv + (long long)b * T * ld + C + h * HS;
    bf16* dv_base = dk_base + C;
    store_rows(dk_base, ld, k0 + warp * 16, T, dk, scale, lane);
    store_rows(dv_base, ld, k0 + warp * 16, T, dv, 1.0f, lane);
}

// ------------------------------------------------------------------ backward: dQ
__global__ void __launch_bounds__(NT) attn_bwd_dq_mma_k(bf16* dqkv, const bf16* dout, const bf16* qkv,
                                                         const float* lse, const float* Dv, int T, int C,
                                                         int NH) {
    __shared__ __align__(128) uint8_t sm[6 * 8192];
    const int nqt = gridDim.x;
    const int qt = nqt - 1 - blockIdx.x;
    const int bh = blockIdx.y, b = bh / NH, h = bh % NH;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long ld = 3LL * C;
    const bf16* q_base = qkv + (long long)b * T * ld + h * HS;
    const bf16* k_base = q_base + C;
    const bf16* v_base = q_base + 2 * C;
    const bf16* do_base = dout + (long long)b * T * C + h * HS;
    const uint32_t sQ = smem_u32(sm), sO = sQ + 8192, sK0 = sQ + 16384, sV0 = sQ + 32768;
    const int q0 = qt * BQ;
    const float scale = 1.0f / sqrtf((float)HS), sl2 = scale * LOG2E;

    load_tile(sQ, q_base, ld, q0, T, tid);
    load_tile(sO, do_base, C, q0, T, tid);
    load_tile(sK0, k_base, ld, 0, T, tid);
    load_tile(sV0, v_base, ld, 0, T, tid);
    cp_commit();

    const int g = lane >> 2, t4 = lane & 3;
    const int qa_row = q0 + warp * 16 + g, qb_row = qa_row + 8;
    const float* lse_bh = lse + (long long)bh * T;
    const float* D_bh = Dv + (long long)bh * T;
    const float La = qa_row < T ? lse_bh[qa_row] * LOG2E : 0.f, Lb = qb_row < T ? lse_bh[qb_row] * LOG2E : 0.f;
    const float Da = qa_row < T ? D_bh[qa_row] : 0.f, Db = qb_row < T ? D_bh[qb_row] : 0.f;
    uint32_t qa[4][4], oa[4][4];
    float dq[8][4];
    zero(dq);
    const int nkv = qt + 1;
    for (int j = 0; j < nkv; j++) {
        const int buf = j & 1;
        if (j + 1 < nkv) {
            load_tile(sK0 + (buf ^ 1) * 8192, k_base, ld, (j + 1) * BKV, T, tid);
            load_tile(sV0 + (buf ^ 1) * 8192, v_base, ld, (j + 1) * BKV, T, tid);
        }
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        if (j == 0) {
            load_a_frags(sQ, warp * 16, lane, qa);
            load_a_frags(sO, warp * 16, lane, oa);
        }
        const uint32_t sK = sK0 + buf * 8192, sV = sV0 + buf * 8192;
        float s[8][4], dp[8][4];
        zero(s);
        zero(dp);
        mma_abT(s, qa, sK, lane);   // S = Q K^T
        mma_abT(dp, oa, sV, lane);  // dP = dO V^T
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
            int key = j * BKV + nt * 8 + 2 * t4;
#pragma unroll
            for (int e = 0; e < 4; e++) {
                int kk = key + (e & 1);
                int qq = e < 2 ? qa_row : qb_row;
                float L = e < 2 ? La : Lb, Dq = e < 2 ? Da : Db;
                float p = (kk <= qq && qq < T) ? exp2f(s[nt][e] * sl2 - L) : 0.f;
                s[nt][e] = p * (dp[nt][e] - Dq);  // dS (unscaled)
            }
        }
        mma_pv(dq, s, sK, lane);  // dQ += dS K
        __syncthreads();
    }
    bf16* dq_base = dqkv + (long long)b * T * ld + h * HS;
    store_rows(dq_base, ld, q0 + warp * 16, T, dq, scale, lane);
}

}  // namespace fa

bool attention_mma_supported(ActType at, int C, int NH) {
    return at == ACT_BF16 && C % NH == 0 && C / NH == fa::HS && (C % 8) == 0;
}

cudaError_t attention_forward_mma(void* out, float* lse, const void* qkv, int B, int T, int C, int NH,
                                  cudaStream_t s) {
    dim3 grid((T + fa::BQ - 1) / fa::BQ, B * NH);
    if (grid.y > 65535) return cudaErrorInvalidValue;
    G2_LAUNCH fa::attn_fwd_mma_k<<<grid, fa::NT, 0, s>>>((bf16*)out, lse, (const bf16*)qkv, T, C, NH);
    return cudaGetLastError();
}

cudaError_t attention_backward_mma(void* dqkv, const void* dout, const void* qkv, const void* out,
                                   const float* lse, int B, int T, int C, int NH, float* Dbuf,
                                   cudaStream_t s) {
    cudaError_t e = attention_bwd_dot(ACT_BF16, Dbuf, dout, out, B, T, C, NH, s);
    if (e != cudaSuccess) return e;
    dim3 grid((T + fa::BQ - 1) / fa::BQ, B * NH);
    if (grid.y > 65535) return cudaErrorInvalidValue;
    G2_LAUNCH fa::attn_bwd_dkv_mma_k<<<grid, fa::NT, 0, s>>>((bf16*)dqkv, (const bf16*)dout, (const bf16*)qkv,
                                                             lse, Dbuf, T, C, NH);
    G2_LAUNCH fa::attn_bwd_dq_mma_k<<<grid, fa::NT, 0, s>>>((bf16*)dqkv, (const bf16*)dout, (const bf16*)qkv,
                                                            lse, Dbuf, T, C, NH);
    return cudaGetLastError();
}

}  // namespace g2
