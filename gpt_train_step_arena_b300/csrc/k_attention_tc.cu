// Causal multi-head attention forward on the 5th-generation tensor cores (tcgen05),
// head size 64, bf16 operands, fp32 accumulation in tensor memory.
//
// What it computes is llm.c's attention_forward (annotated listing §1.7) and picoGPT's
// attention with its causal mask: for every (b, h) and query t, softmax over keys
// t2 <= t of q.k / sqrt(hs), times v.  Only the row log-sum-exp is kept for the
// backward, not the (T, T) probabilities.
//
// One CTA per (128-query tile, b, h), two CTAs resident per SM, 192 threads:
//   warp 0     TMA: the Q tile once, then K_j and V_j (128 keys x 64 bf16 each) into
//              two-stage rings, read straight from the (B, T, 3C) qkv buffer; a K stage
//              is refilled once its S product is done, a V stage once its PV product is;
//              all of the CTA's K and V tiles are prefetched into L2 at the start.
//   warp 1     owns 256 columns of tensor memory (S: 128 x 128 fp32 at column 0,
//              O: 128 x 64 fp32 at column 128); one lane issues S = Q K_j^T and
//              O += P_{j-1} V_{j-1} (tcgen05.mma kind::f16, M = 128).
//   warps 2-5  softmax, one query row per thread: the row max of S_j (tcgen05.ld),
//              P_j = 2^(s * log2e / sqrt(hs) - m) rounded to bf16 into shared memory
//              (the A operand of the PV product, K-major with the 128-byte swizzle),
//              the running sum l, and a rescale of O in tensor memory when the row max
//              grows by more than 2^8 (lazy rescaling: the result is unchanged, the
//              stale max only lets terms reach 2^8).  At the end: O / l and the row
//              log-sum-exp, natural-log units.
// S_{j+1} is issued as soon as the softmax has released S_j, so the product P_j V_j
// and the next S overlap the softmax; the second resident CTA fills the remaining
// gaps.  Every mbarrier wait is bounded; on expiry the kernel raises the timeout flag,
// drains what it issued and returns.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace g2 {
namespace atc {
using namespace tc;

constexpr int HS = 64, BQ = 128, BKV = 128, NTH = 192;
constexpr int TILE = 128 * 64 * 2;  // 16 KB: 128 rows of one head, 128-byte rows
constexpr int OFF_Q = 0, OFF_K = TILE, OFF_V = 3 * TILE, OFF_P = 5 * TILE, OFF_BAR = 7 * TILE;
constexpr uint32_t TMEM_COLS = 256, TM_S = 0, TM_O = 128;
constexpr float LOG2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;
constexpr float RESCALE_LOG2 = 8.0f;

struct FwdBars {
    uint64_t q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full, s_free, p_full, o_done, drain;
    uint32_t tmem_slot;
    int abort;
};
constexpr int FWD_SMEM = OFF_BAR + (int)sizeof(FwdBars);

// 2^x, the hardware approximation (relative error about 2^-22; results below 2^-126
// flush to zero, far below what a bf16 probability or an fp32 row sum resolves).
G2_DEV float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

G2_DEV uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(NTH, 2)
    attn_fwd_tc_k(const __grid_constant__ CUtensorMap tm_qkv, bf16* out, float* lse, int T, int C, int NH,
                  int* flags) {
    extern __shared__ __align__(1024) uint8_t smem[];
    FwdBars* bar = reinterpret_cast<FwdBars*>(smem + OFF_BAR);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The swizzled tiles need a 1024-byte aligned base (the dynamic window starts there
    // when the kernel has no static shared memory); refuse to run otherwise.
    if (smem_u32(smem) & 1023) {
        if (threadIdx.x == 0 && flags) atomicOr(flags, G2_FLAG_TIMEOUT);
        return;
    }
    const int nqt = gridDim.x, qt = nqt - 1 - (int)blockIdx.x;  // heaviest query tiles first
    const int bh = blockIdx.y, b = bh / NH, h = bh % NH;
    const int q0 = qt * BQ, nkv = qt + 1, row0 = b * T;

    if (threadIdx.x == 0) {
        bar->abort = 0;
        mbar_init(&bar->q_full, 1);
        for (int i = 0; i < 2; i++) {
            mbar_init(&bar->k_full[i], 1);
            mbar_init(&bar->k_empty[i], 1);
            mbar_init(&bar->v_full[i], 1);
            mbar_init(&bar->v_empty[i], 1);
        }
        mbar_init(&bar->s_full, 1);
        mbar_init(&bar->s_free, 4);
        mbar_init(&bar->p_full, 4);
        mbar_init(&bar->o_done, 1);
        mbar_init(&bar->drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
        tma_prefetch_desc(&tm_qkv);
    }
    if (warp == 1) tmem_alloc(&bar->tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar->tmem_slot;
    volatile int* abort_flag = &bar->abort;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            mbar_expect_tx(&bar->q_full, TILE);
            tma_load_2d(&tm_qkv, &bar->q_full, smem + OFF_Q, h * HS, row0 + q0);
            // every K and V tile this CTA will read, into L2 ahead of the loads
            for (int j = 2; j < nkv; j++) {
                tma_prefetch_l2(&tm_qkv, C + h * HS, row0 + j * BKV);
                tma_prefetch_l2(&tm_qkv, 2 * C + h * HS, row0 + j * BKV);
            }
            // K_j goes as soon as S_{j-2} has consumed its stage, V_j once P_{j-2} V_{j-2} has
            int issued_k[2] = {-1, -1}, issued_v[2] = {-1, -1};
            bool ok = true;
            for (int j = 0; j < nkv; j++) {
                const int s = j & 1;
                const uint32_t ph = (j >> 1) & 1;
                if (!mbar_wait(&bar->k_empty[s], ph ^ 1, abort_flag, flags)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&bar->k_full[s], TILE);
                tma_load_2d(&tm_qkv, &bar->k_full[s], smem + OFF_K + s * TILE, C + h * HS, row0 + j * BKV);
                issued_k[s] = (int)ph;
                if (!mbar_wait(&bar->v_empty[s], ph ^ 1, abort_flag, flags)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&bar->v_full[s], TILE);
                tma_load_2d(&tm_qkv, &bar->v_full[s], smem + OFF_V + s * TILE, 2 * C + h * HS, row0 + j * BKV);
                issued_v[s] = (int)ph;
            }
            if (!ok) {  // wait (bounded) for the copies still in flight before leaving
                unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(&bar->q_full, 0) && globaltimer() - t0 < TIMEOUT_NS) {
                }
                for (int s = 0; s < 2; s++) {
                    if (issued_k[s] >= 0) {
                        t0 = globaltimer();
                        while (!mbar_try_wait(&bar->k_full[s], (uint32_t)issued_k[s]) && globaltimer() - t0 < TIMEOUT_NS) {
                        }
                    }
                    if (issued_v[s] >= 0) {
                        t0 = globaltimer();
                        while (!mbar_try_wait(&bar->v_full[s], (uint32_t)issued_v[s]) && globaltimer() - t0 < TIMEOUT_NS) {
                        }
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_S = make_idesc(BKV, false, false);  // S: N = 128 keys
            constexpr uint32_t ID_PV = make_idesc(HS, false, true);   // O: N = 64, V is MN-major
            const uint32_t sQ = smem_u32(smem + OFF_Q), sP = smem_u32(smem + OFF_P);
            bool ok = mbar_wait(&bar->q_full, 0, abort_flag, flags);
            bool issued_any = false;
            for (int j = 0; ok && j <= nkv; j++) {
                if (j < nkv) {
                    // S_j once K_j has landed and the softmax has read S_{j-1} out
                    const int s = j & 1;
                    if (!mbar_wait(&bar->k_full[s], (j >> 1) & 1, abort_flag, flags) ||
                        (j > 0 && !mbar_wait(&bar->s_free, (j - 1) & 1, abort_flag, flags))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sK = smem_u32(smem + OFF_K + s * TILE);
#pragma unroll
                    for (int k = 0; k < HS / 16; k++)
                        umma_bf16(tmem + TM_S, sdesc(sQ + k * 32, 16, 1024), sdesc(sK + k * 32, 16, 1024), ID_S,
                                  k > 0 ? 1u : 0u);
                    umma_commit(&bar->s_full);
                    umma_commit(&bar->k_empty[s]);
                    issued_any = true;
                }
                // P_{j-1} V_{j-1} once the softmax has written P_{j-1}
                if (j > 0) {
                    if (!mbar_wait(&bar->p_full, (j - 1) & 1, abort_flag, flags) ||
                        !mbar_wait(&bar->v_full[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, flags)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                if (j > 0) {
                    const int pj = j - 1, ps = pj & 1;
                    const uint32_t sV = smem_u32(smem + OFF_V + ps * TILE);
#pragma unroll
                    for (int k = 0; k < BKV / 16; k++) {
                        // keys [16k, 16k+16): 64-key block k/4 of P, 32 bytes per step inside it
                        const uint64_t ad = sdesc(sP + (k >> 2) * TILE + (k & 3) * 32, 16, 1024);
                        const uint64_t bd = sdesc(sV + k * 16 * 128, 8192, 1024);
                        umma_bf16(tmem + TM_O, ad, bd, ID_PV, (pj > 0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit(&bar->o_done);
                    umma_commit(&bar->v_empty[ps]);
                    issued_any = true;
                }
            }
            if (!ok && issued_any) {
                umma_commit(&bar->drain);
                unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(&bar->drain, 0) && globaltimer() - t0 < TIMEOUT_NS) {
                }
            }
        }
    } else {
        // ---------------- softmax warps 2..5
        const int quarter = warp & 3, r = quarter * 32 + lane;  // TMEM lane = row of the tile
        const int q = q0 + r;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const float sl2 = LOG2E / sqrtf((float)HS);
        uint8_t* prow = smem + OFF_P + r * 128;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkv; j++) {
            ok = mbar_wait(&bar->s_full, j & 1, abort_flag, flags);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const bool diag = j == qt;
            // the whole row of S_j into registers, then S is released for S_{j+1}
            uint32_t sv[BKV];
#pragma unroll
            for (int c = 0; c < BKV / 32; c++) tmem_ld32_raw(lane_base + TM_S + c * 32, sv + c * 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->s_free);
            // causal mask on the diagonal tile: key j*128 + i is visible to row r iff i <= r
            if (diag) {
#pragma unroll
                for (int i = 0; i < BKV; i++)
                    if (i > r) sv[i] = __float_as_uint(-INFINITY);
            }
            float m8[8];
#pragma unroll
            for (int e = 0; e < 8; e++) m8[e] = __uint_as_float(sv[e]);
#pragma unroll
            for (int i = 8; i < BKV; i++) m8[i & 7] = fmaxf(m8[i & 7], __uint_as_float(sv[i]));
            const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * sl2;
            bool resc = false;
            float corr = 1.f;
            if (j == 0) {
                m_used = mx;
            } else if (mx > m_used + RESCALE_LOG2) {
                corr = ex2(m_used - mx);
                m_used = mx;
                l *= corr;
                resc = true;
            }
            // P = 2^(s * sl2 - m) packed to bf16 in registers (S dies as P grows)
            const float mneg = -m_used;
            float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            uint32_t pk[BKV / 2];
#pragma unroll
            for (int i = 0; i < BKV; i += 2) {
                const float p0 = ex2(fmaf(__uint_as_float(sv[i]), sl2, mneg));
                const float p1 = ex2(fmaf(__uint_as_float(sv[i + 1]), sl2, mneg));
                l8[i & 7] += p0;
                l8[(i & 7) + 1] += p1;
                pk[i >> 1] = pack_bf16x2(p0, p1);
            }
            l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
            if (j > 0) {
                // O and the P buffer are free once P_{j-1} V_{j-1} has completed
                ok = mbar_wait(&bar->o_done, (j - 1) & 1, abort_flag, flags);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
                    for (int c = 0; c < 2; c++) {
                        float o[32];
                        tmem_ld32(lane_base + TM_O + c * 32, o);
#pragma unroll
                        for (int i = 0; i < 32; i++) o[i] *= corr;
                        tmem_st32(lane_base + TM_O + c * 32, o);
                    }
                    tmem_wait_st();
                }
            }
            // 16-byte chunk ch (keys 8ch..8ch+7): 64-key block ch/8, chunk ch%8 of this row,
            // XOR-swizzled by the row (the layout TMA's 128-byte swizzle produces)
#pragma unroll
            for (int ch = 0; ch < BKV / 8; ch++)
                *reinterpret_cast<uint4*>(prow + (ch >> 3) * TILE + (((ch & 7) ^ (r & 7)) << 4)) =
                    make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->p_full);
        }
        if (ok) {
            ok = mbar_wait(&bar->o_done, (nkv - 1) & 1, abort_flag, flags);
            if (__all_sync(0xffffffffu, ok)) {
                tc_fence_after();
                float o[64];
                tmem_ld32(lane_base + TM_O, o);
                tmem_ld32(lane_base + TM_O + 32, o + 32);
                if (q < T) {
                    const float inv = 1.0f / l;
                    bf16* dst = out + (size_t)(row0 + q) * C + h * HS;
#pragma unroll
                    for (int i = 0; i < HS; i += 8) {
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 8; e++) y[e] = o[i + e] * inv;
                        Vec8<bf16>::store(dst + i, y);
                    }
                    lse[(size_t)bh * T + q] = (m_used + log2f(l)) * LN2;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace atc

bool attention_tc_supported(ActType at, int C, int NH, const void* qkv) {
    return at == ACT_BF16 && C % NH == 0 && C / NH == atc::HS && (C % 8) == 0 &&
           ((uintptr_t)qkv & 15) == 0 && tc::encode_fn() != nullptr;
}

cudaError_t attention_forward_tc(void* out, float* lse, const void* qkv, int B, int T, int C, int NH, int* flags,
                                 cudaStream_t s) {
    CUtensorMap tm;
    if (!tc::make_map(&tm, qkv, 3ull * C, (uint64_t)B * T, 3ull * C, 64, 128)) return cudaErrorNotSupported;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(atc::attn_fwd_tc_k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             atc::FWD_SMEM);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    dim3 grid((T + atc::BQ - 1) / atc::BQ, B * NH);
    if (grid.y > 65535) return cudaErrorInvalidValue;
    G2_LAUNCH atc::attn_fwd_tc_k<<<grid, atc::NTH, atc::FWD_SMEM, s>>>(tm, (bf16*)out, lse, T, C, NH, flags);
    return cudaGetLastError();
}

}  // namespace g2
