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
constexpr int NTH_BWD = 320;  // backward: TMA warp, MMA warp, 8 softmax warps
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


// ------------------------------------------------------------------ backward
// llm.c §1.8 attention_backward, without atomics and without the (T, T) buffers: P is
// rebuilt from the forward's log-sum-exp L and D = rowsum(dO * O), dS = P * (dP - D).
// Two kernels of one template, 320 threads (TMA warp, MMA warp, 8 softmax warps: two per
// tensor-memory lane quarter, each taking 32 of a half's 64 columns), two CTAs per SM:
//   DQ = true   (query-major, runs first): the CTA owns 128 queries of one head and
//               streams K_j and V_j for j <= the query tile.  Its softmax threads first
//               compute D for their own rows (and store it for the other kernel); then
//               S = Q K^T, dP = dO V^T, dS = P (dP - D), dQ += dS K.
//   DQ = false  (key-major): the CTA owns 128 keys and streams Q_i and dO_i for i >= the
//               key tile; S^T = K Q^T, dP^T = V dO^T, P^T and dS^T = P^T (dP^T - D) with
//               L and D of the query columns staged in shared memory; dV += P^T dO,
//               dK += dS^T Q.
// Each streamed 128-row tile is processed in two 64-column halves through one tensor-
// memory buffer (S at column 0, dP at 64); P and dS are written back (bf16) over the
// columns each thread read and are the A operand of the accumulation products, which the
// tensor core runs before the next half's S and dP overwrite the buffer.  A CTA's chain
// (products -> softmax -> products) is serial; the second CTA on the SM fills the gaps:
// one CTA per SM issues these 64-column products at about 85 clocks each, two reach
// about 58 (the tensor core's own rate is 45-48).
// Tensor memory (256 columns): the half buffer at 0-127, dQ (or dV) at 128, dK at 192; the
// query-major CTA's own rows Q and dO (A operands of S and dP) at 192 and 224.  The key-
// major CTA keeps K and V in shared memory instead.
struct BwdBars {
    uint64_t row_full, st_full[2], st_empty[2], sdp_full, pds_full, stats[2], acc_done, drain;
    uint32_t tmem_slot;
    int abort;
};
constexpr int B_ROWS = 0;                 // key-major: K, V tiles (32 KB)
constexpr int B_ST = 2 * TILE;            // streamed stages: 2 x (A 16 KB + B 16 KB)
constexpr int B_STATS = B_ST + 4 * TILE;  // key-major: L, D of 2 x 128 query columns
constexpr int B_BAR = B_STATS + 2 * 2 * 128 * 4;
constexpr int BWD_SMEM = B_BAR + (int)sizeof(BwdBars);
constexpr uint32_t TB_COLS = 256, TB_ACC1 = 128, TB_ACC2 = 192, TB_RA = 192, TB_RB = 224;

template <bool DQ>
__global__ void __launch_bounds__(NTH_BWD, 2)
    attn_bwd_tc_k(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                  bf16* dqkv, const bf16* qkv, const bf16* dout, const bf16* outp, const float* lse, float* Dbuf,
                  int T, int C, int NH, int* flags) {
    extern __shared__ __align__(1024) uint8_t smem[];
    BwdBars* bar = reinterpret_cast<BwdBars*>(smem + B_BAR);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (smem_u32(smem) & 1023) {
        if (threadIdx.x == 0 && flags) atomicOr(flags, G2_FLAG_TIMEOUT);
        return;
    }
    const int ntiles_t = gridDim.x;
    // the row tile: queries (heaviest = last first) or keys (heaviest = first first)
    const int rt = DQ ? ntiles_t - 1 - (int)blockIdx.x : (int)blockIdx.x;
    const int bh = blockIdx.y, b = bh / NH, h = bh % NH;
    const int row0 = b * T, r0 = rt * 128;
    // streamed tiles: keys 0..rt (DQ) or queries rt..ntiles_t-1 (key-major)
    const int st0 = DQ ? 0 : rt, nst = DQ ? rt + 1 : ntiles_t - rt;
    const int xa_st = DQ ? C + h * HS : h * HS;      // K or Q (qkv map)
    const int xb_st = DQ ? 2 * C + h * HS : h * HS;  // V (qkv map) or dO (its own map)
    const CUtensorMap* map_b_st = DQ ? &tm_qkv : &tm_do;

    if (threadIdx.x == 0) {
        bar->abort = 0;
        mbar_init(&bar->row_full, DQ ? 8 : 1);  // softmax warps' tensor-memory rows, or TMA
        for (int i = 0; i < 2; i++) {
            mbar_init(&bar->st_full[i], 1);
            mbar_init(&bar->st_empty[i], 1);
            mbar_init(&bar->stats[i], 256);
        }
        mbar_init(&bar->sdp_full, 1);
        mbar_init(&bar->pds_full, 8);
        mbar_init(&bar->acc_done, 1);
        mbar_init(&bar->drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
        tma_prefetch_desc(&tm_qkv);
        tma_prefetch_desc(&tm_do);
    }
    if (warp == 1) tmem_alloc(&bar->tmem_slot, TB_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar->tmem_slot;
    volatile int* abort_flag = &bar->abort;

    if (warp == 0) {
        // ---------------- TMA producer: the key-major CTA's K and V, then the streamed tiles
        if (lane == 0) {
            if (!DQ) {
                mbar_expect_tx(&bar->row_full, 2 * TILE);
                tma_load_2d(&tm_qkv, &bar->row_full, smem + B_ROWS, C + h * HS, row0 + r0);
                tma_load_2d(&tm_qkv, &bar->row_full, smem + B_ROWS + TILE, 2 * C + h * HS, row0 + r0);
            }
            for (int n = 2; n < nst; n++) {
                tma_prefetch_l2(&tm_qkv, xa_st, row0 + (st0 + n) * 128);
                tma_prefetch_l2(map_b_st, xb_st, row0 + (st0 + n) * 128);
            }
            int issued[2] = {-1, -1};
            bool ok = true;
            for (int n = 0; n < nst; n++) {
                const int s = n & 1;
                const uint32_t ph = (n >> 1) & 1;
                if (!mbar_wait(&bar->st_empty[s], ph ^ 1, abort_flag, flags)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&bar->st_full[s], 2 * TILE);
                uint8_t* st = smem + B_ST + s * 2 * TILE;
                tma_load_2d(&tm_qkv, &bar->st_full[s], st, xa_st, row0 + (st0 + n) * 128);
                tma_load_2d(map_b_st, &bar->st_full[s], st + TILE, xb_st, row0 + (st0 + n) * 128);
                issued[s] = (int)ph;
            }
            if (!ok) {
                unsigned long long t0 = globaltimer();
                if (!DQ) {
                    while (!mbar_try_wait(&bar->row_full, 0) && globaltimer() - t0 < TIMEOUT_NS) {
                    }
                }
                for (int s = 0; s < 2; s++) {
                    if (issued[s] < 0) continue;
                    t0 = globaltimer();
                    while (!mbar_try_wait(&bar->st_full[s], (uint32_t)issued[s]) && globaltimer() - t0 < TIMEOUT_NS) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_SDP = make_idesc(64, false, false);  // N = 64 streamed rows
            constexpr uint32_t ID_ACC = make_idesc(HS, false, true);   // N = 64, streamed operand MN-major
            const uint32_t sbase = smem_u32(smem);
            const int nhalves = 2 * nst;
            bool ok = mbar_wait(&bar->row_full, 0, abort_flag, flags);
            bool issued_any = false;
            // S and dP of half g (tile g/2, columns 64 (g%2) ..): A = the CTA's rows (tensor
            // memory, or shared memory for K and V), B = the streamed rows of the half
            auto issue_sdp = [&](int g) -> bool {
                const int n = g >> 1, hh = g & 1, s = n & 1;
                if (hh == 0 && !mbar_wait(&bar->st_full[s], (n >> 1) & 1, abort_flag, flags)) return false;
                tc_fence_after();
                const uint32_t sA = sbase + B_ST + s * 2 * TILE + hh * 8192, sB = sA + TILE;
#pragma unroll
                for (int k = 0; k < HS / 16; k++) {
                    const uint64_t bd = sdesc(sA + k * 32, 16, 1024);
                    if (DQ)
                        umma_bf16_ts(tmem, tmem + TB_RA + k * 8, bd, ID_SDP, k > 0 ? 1u : 0u);
                    else
                        umma_bf16(tmem, sdesc(sbase + B_ROWS + k * 32, 16, 1024), bd, ID_SDP, k > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int k = 0; k < HS / 16; k++) {
                    const uint64_t bd = sdesc(sB + k * 32, 16, 1024);
                    if (DQ)
                        umma_bf16_ts(tmem + 64, tmem + TB_RB + k * 8, bd, ID_SDP, k > 0 ? 1u : 0u);
                    else
                        umma_bf16(tmem + 64, sdesc(sbase + B_ROWS + TILE + k * 32, 16, 1024), bd, ID_SDP,
                                  k > 0 ? 1u : 0u);
                }
                umma_commit(&bar->sdp_full);
                issued_any = true;
                return true;
            };
            if (ok) ok = issue_sdp(0);
            for (int g = 0; ok && g < nhalves; g++) {
                const int n = g >> 1, hh = g & 1, s = n & 1;
                if (!mbar_wait(&bar->pds_full, g & 1, abort_flag, flags)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // accumulation of half g: A = P or dS in tensor memory (column group c of the
                // half at 32c, 16 columns = 32 rows of the contraction each), B = the
                // streamed rows of the half read N-major (64 hs wide)
                const uint32_t sA = sbase + B_ST + s * 2 * TILE + hh * 8192, sB = sA + TILE;
#pragma unroll
                for (int k = 0; k < 64 / 16; k++) {
                    const uint32_t acc = (g > 0 || k > 0) ? 1u : 0u;
                    const uint32_t a_off = (k >> 1) * 32 + (k & 1) * 8;
                    const uint64_t bA = sdesc(sA + k * 2048, 8192, 1024);
                    if (DQ) {
                        umma_bf16_ts(tmem + TB_ACC1, tmem + 64 + a_off, bA, ID_ACC, acc);  // dQ += dS K
                    } else {
                        const uint64_t bB = sdesc(sB + k * 2048, 8192, 1024);
                        umma_bf16_ts(tmem + TB_ACC1, tmem + a_off, bB, ID_ACC, acc);       // dV += P^T dO
                        umma_bf16_ts(tmem + TB_ACC2, tmem + 64 + a_off, bA, ID_ACC, acc);  // dK += dS^T Q
                    }
                }
                issued_any = true;
                if (hh == 1) umma_commit(&bar->st_empty[s]);
                if (g == nhalves - 1) umma_commit(&bar->acc_done);
                // the next half's S and dP follow this accumulation on the tensor core
                if (g + 1 < nhalves && !issue_sdp(g + 1)) ok = false;
            }
            if (!ok && issued_any) {
                umma_commit(&bar->drain);
                unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(&bar->drain, 0) && globaltimer() - t0 < TIMEOUT_NS) {
                }
            }
        }
    } else {
        // ---------------- softmax warps 2..9: thread = row of the CTA's tile; warps 2-5
        // take columns 0-31 of each half, warps 6-9 columns 32-63
        const int quarter = warp & 3, r = quarter * 32 + lane, sub = (warp - 2) >> 2;
        const int grow = r0 + r;  // query (DQ) or key position of this thread's row
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float sl2 = LOG2E / sqrtf((float)HS);
        float L2_row = 0.f, D_row = 0.f;
        float* Ls = reinterpret_cast<float*>(smem + B_STATS);  // [2][128] (key-major only)
        float* Dsm = Ls + 2 * 128;
        float nL = 0.f, nD = 0.f;  // key-major: this thread's query column of the next tile
        if (DQ) {
            // this row's Q (group 0) or dO (group 1) into tensor memory: the A operands of S
            // and dP, 64 bf16 = 32 packed columns
            {
                uint32_t rv[32];
                const bf16* src = sub == 0 ? qkv + (size_t)(row0 + grow) * 3 * C + h * HS
                                           : dout + (size_t)(row0 + grow) * C + h * HS;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const uint4 u = grow < T ? reinterpret_cast<const uint4*>(src)[i] : make_uint4(0, 0, 0, 0);
                    rv[4 * i] = u.x;
                    rv[4 * i + 1] = u.y;
                    rv[4 * i + 2] = u.z;
                    rv[4 * i + 3] = u.w;
                }
                tmem_st32u(tmem + lane_off + (sub == 0 ? TB_RA : TB_RB), rv);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar->row_full);
            }
            // D = rowsum(dO * O) for this row (both column groups need it; group 0 stores
            // it for the key-major kernel)
            if (grow < T) {
                const bf16* dor = dout + (size_t)(row0 + grow) * C + h * HS;
                const bf16* orr = outp + (size_t)(row0 + grow) * C + h * HS;
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < HS; i += 8) {
                    float a8[8], c8[8];
                    Vec8<bf16>::load(dor + i, a8);
                    Vec8<bf16>::load(orr + i, c8);
#pragma unroll
                    for (int e = 0; e < 8; e++) acc += a8[e] * c8[e];
                }
                D_row = acc;
                if (sub == 0) Dbuf[(size_t)bh * T + grow] = acc;
                L2_row = lse[(size_t)bh * T + grow] * LOG2E;
            }
        } else if (sub == 0) {
            const int q = st0 * 128 + r;
            nL = q < T ? lse[(size_t)bh * T + q] * LOG2E : INFINITY;  // absent queries: P = 0
            nD = q < T ? Dbuf[(size_t)bh * T + q] : 0.f;
        }
        bool ok = true;
        for (int n = 0; n < nst && ok; n++) {
            const int slot = n & 1;
            if (!DQ) {
                // column group 0 writes one query column's L and D each; everyone waits
                // (bounded) until all have: slot n&1 was last read in tile n-2, which every
                // thread finished before arriving for tile n-1
                if (sub == 0) {
                    Ls[slot * 128 + r] = nL;
                    Dsm[slot * 128 + r] = nD;
                }
                mbar_arrive(&bar->stats[slot]);
                ok = mbar_wait(&bar->stats[slot], (n >> 1) & 1, abort_flag, flags);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                if (sub == 0 && n + 1 < nst) {
                    const int q = (st0 + n + 1) * 128 + r;
                    nL = q < T ? lse[(size_t)bh * T + q] * LOG2E : INFINITY;
                    nD = q < T ? Dbuf[(size_t)bh * T + q] : 0.f;
                }
            }
            const bool diag = (st0 + n) == rt;
            for (int hh = 0; hh < 2; hh++) {
                const int g = 2 * n + hh;
                ok = mbar_wait(&bar->sdp_full, g & 1, abort_flag, flags);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // 32 columns in two rounds of 16: S and dP in, P and dS (8 packed columns
                // each) written back over the first half of what this thread read
#pragma unroll
                for (int rd = 0; rd < 2; rd++) {
                    uint32_t sv[16], dv[16];
                    const uint32_t tS = tmem + lane_off + sub * 32 + rd * 16;
                    tmem_ld16_raw(tS, sv);
                    tmem_ld16_raw(tS + 64, dv);
                    tmem_wait_ld();
                    uint32_t pk[8], dk[8];
                    const int cbase = hh * 64 + sub * 32 + rd * 16;  // column within the streamed tile
#pragma unroll
                    for (int c4 = 0; c4 < 16; c4 += 4) {
                        float Lc[4], Dc[4];
                        if (DQ) {
#pragma unroll
                            for (int e = 0; e < 4; e++) {
                                Lc[e] = L2_row;
                                Dc[e] = D_row;
                            }
                        } else {
                            const float4 l4 = *reinterpret_cast<const float4*>(Ls + slot * 128 + cbase + c4);
                            const float4 d4 = *reinterpret_cast<const float4*>(Dsm + slot * 128 + cbase + c4);
                            Lc[0] = l4.x; Lc[1] = l4.y; Lc[2] = l4.z; Lc[3] = l4.w;
                            Dc[0] = d4.x; Dc[1] = d4.y; Dc[2] = d4.z; Dc[3] = d4.w;
                        }
                        float pv[4], dsv[4];
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const int c = cbase + c4 + e;
                            // causal: key <= query; DQ rows are queries, key-major rows are keys
                            const bool vis = !diag || (DQ ? c <= r : r <= c);
                            const float pr = vis ? ex2(fmaf(__uint_as_float(sv[c4 + e]), sl2, -Lc[e])) : 0.f;
                            pv[e] = pr;
                            dsv[e] = pr * (__uint_as_float(dv[c4 + e]) - Dc[e]);
                        }
                        pk[c4 >> 1] = pack_bf16x2(pv[0], pv[1]);
                        pk[(c4 >> 1) + 1] = pack_bf16x2(pv[2], pv[3]);
                        dk[c4 >> 1] = pack_bf16x2(dsv[0], dsv[1]);
                        dk[(c4 >> 1) + 1] = pack_bf16x2(dsv[2], dsv[3]);
                    }
                    // packed columns 8 rd .. 8 rd + 7 of this group's 16 (all already read)
                    const uint32_t tP = tmem + lane_off + sub * 32 + rd * 8;
                    if (!DQ) tmem_st8(tP, pk);
                    tmem_st8(tP + 64, dk);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar->pds_full);
            }
        }
        if (ok) {
            ok = mbar_wait(&bar->acc_done, 0, abort_flag, flags);
            if (__all_sync(0xffffffffu, ok)) {
                tc_fence_after();
                const float scale = 1.0f / sqrtf((float)HS);
                bf16* base = dqkv + (size_t)(row0 + grow) * 3 * C + h * HS;
                // DQ: group g stores dQ columns 32g..32g+31; key-major: group 0 dV, group 1 dK
                const int ncol = DQ ? 32 : 64;
                bf16* dst = DQ ? base + sub * 32 : (sub ? base + C : base + 2 * C);
                const float mul = (DQ || sub) ? scale : 1.0f;
                const uint32_t t0 = tmem + lane_off + (DQ ? TB_ACC1 + sub * 32 : (sub ? TB_ACC2 : TB_ACC1));
                for (int c0 = 0; c0 < ncol; c0 += 32) {
                    float a[32];
                    tmem_ld32(t0 + c0, a);
                    if (grow < T) {
#pragma unroll
                        for (int i = 0; i < 32; i += 8) {
                            float y[8];
#pragma unroll
                            for (int e = 0; e < 8; e++) y[e] = a[i + e] * mul;
                            Vec8<bf16>::store(dst + c0 + i, y);
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TB_COLS);
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

cudaError_t attention_backward_tc(void* dqkv, const void* dout, const void* qkv, const void* out, const float* lse,
                                  int B, int T, int C, int NH, float* Dbuf, int* flags, cudaStream_t s) {
    CUtensorMap tq, td;
    if (((uintptr_t)dout & 15) || ((uintptr_t)out & 15) || ((uintptr_t)dqkv & 15) || (C % 8))
        return cudaErrorNotSupported;
    if (!tc::make_map(&tq, qkv, 3ull * C, (uint64_t)B * T, 3ull * C, 64, 128) ||
        !tc::make_map(&td, dout, (uint64_t)C, (uint64_t)B * T, (uint64_t)C, 64, 128))
        return cudaErrorNotSupported;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(atc::attn_bwd_tc_k<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             atc::BWD_SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(atc::attn_bwd_tc_k<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     atc::BWD_SMEM);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    dim3 grid((T + 127) / 128, B * NH);
    if (grid.y > 65535) return cudaErrorInvalidValue;
    // the query-major kernel also writes D = rowsum(dO * O), which the key-major one reads
    G2_LAUNCH atc::attn_bwd_tc_k<true><<<grid, atc::NTH_BWD, atc::BWD_SMEM, s>>>(
        tq, td, (bf16*)dqkv, (const bf16*)qkv, (const bf16*)dout, (const bf16*)out, lse, Dbuf, T, C, NH, flags);
    G2_LAUNCH atc::attn_bwd_tc_k<false><<<grid, atc::NTH_BWD, atc::BWD_SMEM, s>>>(
        tq, td, (bf16*)dqkv, (const bf16*)qkv, (const bf16*)dout, (const bf16*)out, lse, Dbuf, T, C, NH, flags);
    return cudaGetLastError();
}

}  // namespace g2
