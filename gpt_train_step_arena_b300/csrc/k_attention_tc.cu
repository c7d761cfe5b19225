// Causal multi-head attention forward on the 5th-generation tensor cores (tcgen05),
// head size 64, bf16 operands, fp32 accumulation in tensor memory.
//
// What it computes is llm.c's attention_forward (annotated listing §1.7) and picoGPT's
// attention with its causal mask: for every (b, h) and query t, softmax over keys
// t2 <= t of q.k / sqrt(hs), times v.  Only the row log-sum-exp is kept for the
// backward, not the (T, T) probabilities.
//
// Persistent: two CTAs per SM, each looping over work items (a 128-query tile of one
// (b, h), heaviest first), 192 threads:
//   warp 0     TMA: each item's Q tile into one of two Q buffers (the next item's Q
//              loads while the current item runs), then K_j and V_j (128 keys x 64 bf16)
//              into two-stage rings, straight from the (B, T, 3C) qkv buffer; a K stage
//              is refilled once its S product is done, a V stage once its PV product is;
//              each item's K and V tiles are prefetched into L2 when it starts.
//   warp 1     owns 256 columns of tensor memory (S: 128 x 128 fp32 at column 0,
//              O: 128 x 64 fp32 at column 128, P: 128 x 128 bf16 packed at column 192);
//              one lane issues S = Q K_j^T and O += P_{j-1} V_{j-1} (tcgen05.mma
//              kind::f16, M = 128; P read from tensor memory), tile after tile across
//              items, so an item's last PV runs behind the next item's first S.
//   warps 2-5  softmax, one query row per thread: the row max of S_j (tcgen05.ld),
//              P_j = 2^(s * log2e / sqrt(hs) - m) rounded to bf16 into tensor memory
//              (tcgen05.st), the running sum l, and a rescale of O in tensor memory when
//              the row max grows by more than 2^8 (lazy rescaling: the result is
//              unchanged, the stale max only lets terms reach 2^8).  At the end of an
//              item: O / l and the row log-sum-exp, natural-log units; then O is released
//              for the next item's first PV.
// Every mbarrier wait is bounded; on expiry the kernel raises the timeout flag, drains
// what it issued and returns.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace g2 {
namespace atc {
using namespace tc;

constexpr int HS = 64, BQ = 128, BKV = 128, NTH = 192;
constexpr int NTH_BWD = 576;  // backward: TMA warp, MMA warp, two softmax groups of 8 warps
constexpr int TILE = 128 * 64 * 2;  // 16 KB: 128 rows of one head, 128-byte rows
constexpr int OFF_Q = 0, OFF_K = 2 * TILE, OFF_V = 4 * TILE, OFF_BAR = 6 * TILE;  // Q, K, V: 2 buffers each
constexpr uint32_t TMEM_COLS = 256, TM_S = 0, TM_O = 128, TM_P = 192;
constexpr float LOG2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;
constexpr float RESCALE_LOG2 = 8.0f;

struct FwdBars {
    uint64_t q_full[2], q_empty[2], k_full[2], k_empty[2], v_full[2], v_empty[2], s_full, s_free, p_full, o_done,
        o_free, drain;
    uint32_t tmem_slot;
    int abort;
};
// Work item w: query tile qt of (b, h) = bh, heaviest tiles first.
struct FwdItem {
    int qt, bh, nkv;
};
// The k-th work item of CTA c among G persistent CTAs: items are listed heaviest first and
// handed out in rounds of G whose direction alternates (a snake), so that every CTA's
// total stays within one item of the mean.  Which CTA runs an item changes nothing in
// its arithmetic.
G2_DEV int item_of(int k, int c, int G) { return k * G + ((k & 1) ? G - 1 - c : c); }

G2_DEV FwdItem fwd_item(int w, int nbh, int ntq) {
    FwdItem it;
    it.qt = ntq - 1 - w / nbh;
    it.bh = w % nbh;
    it.nkv = it.qt + 1;
    return it;
}
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
    attn_fwd_tc_k(const __grid_constant__ CUtensorMap tm_qkv, bf16* out, float* lse, int T, int C, int NH, int nbh,
                  int* flags) {
    G2_PDL_ENTRY();
    extern __shared__ __align__(1024) uint8_t smem[];
    FwdBars* bar = reinterpret_cast<FwdBars*>(smem + OFF_BAR);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The swizzled tiles need a 1024-byte aligned base (the dynamic window starts there
    // when the kernel has no static shared memory); refuse to run otherwise.
    if (smem_u32(smem) & 1023) {
        if (threadIdx.x == 0 && flags) atomicOr(flags, G2_FLAG_TIMEOUT);
        return;
    }
    const int ntq = (T + BQ - 1) / BQ, nitems = ntq * nbh;

    if (threadIdx.x == 0) {
        bar->abort = 0;
        for (int i = 0; i < 2; i++) {
            mbar_init(&bar->q_full[i], 1);
            mbar_init(&bar->q_empty[i], 1);
            mbar_init(&bar->k_full[i], 1);
            mbar_init(&bar->k_empty[i], 1);
            mbar_init(&bar->v_full[i], 1);
            mbar_init(&bar->v_empty[i], 1);
        }
        mbar_init(&bar->s_full, 1);
        mbar_init(&bar->s_free, 4);
        mbar_init(&bar->p_full, 4);
        mbar_init(&bar->o_done, 1);
        mbar_init(&bar->o_free, 4);
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
        // ---------------- TMA producer: per item its Q (buffer k % 2, free once the item
        // two back has issued its last S), then its K and V tiles through the rings; the
        // ring position g counts tiles over all of this CTA's items
        if (lane == 0) {
            int issued_q[2] = {-1, -1}, issued_k[2] = {-1, -1}, issued_v[2] = {-1, -1};
            bool ok = true;
            int g = 0;
            for (int k = 0, w = item_of(0, blockIdx.x, gridDim.x); ok && w < nitems;
                 k++, w = item_of(k, blockIdx.x, gridDim.x)) {
                const FwdItem it = fwd_item(w, nbh, ntq);
                const int row0 = (it.bh / NH) * T, h = it.bh % NH;
                const int qb = k & 1;
                const uint32_t qph = (k >> 1) & 1;
                if (!mbar_wait(&bar->q_empty[qb], qph ^ 1, abort_flag, flags)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&bar->q_full[qb], TILE);
                tma_load_2d(&tm_qkv, &bar->q_full[qb], smem + OFF_Q + qb * TILE, h * HS, row0 + it.qt * BQ);
                issued_q[qb] = (int)qph;
                // the item's K and V tiles past the first two, into L2 ahead of their loads
                for (int j = 2; j < it.nkv; j++) {
                    tma_prefetch_l2(&tm_qkv, C + h * HS, row0 + j * BKV);
                    tma_prefetch_l2(&tm_qkv, 2 * C + h * HS, row0 + j * BKV);
                }
                for (int j = 0; j < it.nkv; j++, g++) {
                    const int s = g & 1;
                    const uint32_t ph = (g >> 1) & 1;
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
            }
            if (!ok) {  // wait (bounded) for the copies still in flight before leaving
                auto drain = [&](uint64_t* b, int parity) {
                    if (parity < 0) return;
                    const unsigned long long t0 = globaltimer();
                    while (!mbar_try_wait(b, (uint32_t)parity) && globaltimer() - t0 < TIMEOUT_NS) {
                    }
                };
#pragma unroll
                for (int s = 0; s < 2; s++) {
                    drain(&bar->q_full[s], issued_q[s]);
                    drain(&bar->k_full[s], issued_k[s]);
                    drain(&bar->v_full[s], issued_v[s]);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: the whole warp runs the loop converged, one elected
        // lane issues (see umma_bf16_w); tiles are numbered g over all of this CTA's items
        {
            auto wait_all = [&](uint64_t* b, uint32_t par) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(b, par, abort_flag, flags));
            };
            constexpr uint32_t ID_S = make_idesc(BKV, false, false);  // S: N = 128 keys
            constexpr uint32_t ID_PV = make_idesc(HS, false, true);   // O: N = 64, V is MN-major
            bool ok = true, issued_any = false;
            // O += P_g V_g once the softmax has written P_g into tensor memory: 8 products of 16
            // keys (8 packed columns of P each); an item's first one overwrites O, after the
            // softmax has read out the item before's (o_free)
            auto issue_pv = [&](int g, bool first, int k) -> bool {
                if (!wait_all(&bar->p_full, g & 1) || !wait_all(&bar->v_full[g & 1], (g >> 1) & 1)) return false;
                if (first && k > 0 && !wait_all(&bar->o_free, (k - 1) & 1)) return false;
                tc_fence_after();
                const uint32_t sV = smem_u32(smem + OFF_V + (g & 1) * TILE);
#pragma unroll
                for (int kk = 0; kk < BKV / 16; kk++)
                    umma_bf16_ts_w(tmem + TM_O, tmem + TM_P + kk * 8, sdesc(sV + kk * 16 * 128, 8192, 1024), ID_PV,
                                   (!first || kk > 0) ? 1u : 0u);
                umma_commit_w(&bar->o_done);
                umma_commit_w(&bar->v_empty[g & 1]);
                return true;
            };
            int g = 0;                                        // S products issued so far
            int pend_g = -1, pend_k = 0;                      // the tile whose PV is still to issue
            bool pend_first = false;
            for (int k = 0, w = item_of(0, blockIdx.x, gridDim.x); ok && w < nitems;
                 k++, w = item_of(k, blockIdx.x, gridDim.x)) {
                const FwdItem it = fwd_item(w, nbh, ntq);
                const int qb = k & 1;
                if (!wait_all(&bar->q_full[qb], (k >> 1) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t sQ = smem_u32(smem + OFF_Q + qb * TILE);
                for (int j = 0; j < it.nkv; j++, g++) {
                    // S_g once K_g has landed and the softmax has read S_{g-1} out
                    const int s = g & 1;
                    if (!wait_all(&bar->k_full[s], (g >> 1) & 1) || (g > 0 && !wait_all(&bar->s_free, (g - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sK = smem_u32(smem + OFF_K + s * TILE);
#pragma unroll
                    for (int kk = 0; kk < HS / 16; kk++)
                        umma_bf16_w(tmem + TM_S, sdesc(sQ + kk * 32, 16, 1024), sdesc(sK + kk * 32, 16, 1024), ID_S,
                                    kk > 0 ? 1u : 0u);
                    umma_commit_w(&bar->s_full);
                    umma_commit_w(&bar->k_empty[s]);
                    if (j == it.nkv - 1) umma_commit_w(&bar->q_empty[qb]);  // the item's Q is done with
                    issued_any = true;
                    // the previous tile's PV (perhaps the item before's last) behind this S
                    if (pend_g >= 0 && !issue_pv(pend_g, pend_first, pend_k)) {
                        ok = false;
                        break;
                    }
                    pend_g = g;
                    pend_first = j == 0;
                    pend_k = k;
                }
            }
            if (ok && pend_g >= 0 && !issue_pv(pend_g, pend_first, pend_k)) ok = false;
            if (!ok && issued_any) {
                umma_commit_w(&bar->drain);
                if (lane == 0) {
                    unsigned long long t0 = globaltimer();
                    while (!mbar_try_wait(&bar->drain, 0) && globaltimer() - t0 < TIMEOUT_NS) {
                    }
                }
                __syncwarp();
            }
        }
    } else {
        // ---------------- softmax warps 2..5
        const int quarter = warp & 3, r = quarter * 32 + lane;  // TMEM lane = row of the tile
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const float sl2 = LOG2E / sqrtf((float)HS);
        bool ok = true;
        int g = 0;  // tiles over all of this CTA's items (the barriers' phase count)
        for (int k = 0, w = item_of(0, blockIdx.x, gridDim.x); ok && w < nitems;
             k++, w = item_of(k, blockIdx.x, gridDim.x)) {
            const int qt = fwd_item(w, nbh, ntq).qt;
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j <= qt; j++, g++) {
                ok = mbar_wait(&bar->s_full, g & 1, abort_flag, flags);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const bool diag = j == qt;
                // the whole row of S_g into registers, then S is released for S_{g+1}
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
                // row maximum: a tree of three-input maxima (43 + 15 + 5 + 2 + 1 instructions)
                float t43[43];
#pragma unroll
                for (int i = 0; i < 42; i++)
                    t43[i] = max3f(__uint_as_float(sv[3 * i]), __uint_as_float(sv[3 * i + 1]),
                                   __uint_as_float(sv[3 * i + 2]));
                t43[42] = fmaxf(__uint_as_float(sv[126]), __uint_as_float(sv[127]));
                float t15[15];
#pragma unroll
                for (int i = 0; i < 14; i++) t15[i] = max3f(t43[3 * i], t43[3 * i + 1], t43[3 * i + 2]);
                t15[14] = t43[42];
                const float t5[5] = {max3f(t15[0], t15[1], t15[2]), max3f(t15[3], t15[4], t15[5]),
                                     max3f(t15[6], t15[7], t15[8]), max3f(t15[9], t15[10], t15[11]),
                                     max3f(t15[12], t15[13], t15[14])};
                const float mx = max3f(max3f(t5[0], t5[1], t5[2]), t5[3], t5[4]) * sl2;
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
                // P = 2^(s * sl2 - m) packed to bf16 in registers (S dies as P grows); the
                // scale and the row sum run two columns per instruction
                const float2 sl2x2 = make_float2(sl2, sl2), mneg = make_float2(-m_used, -m_used);
                float2 l4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
                uint32_t pk[BKV / 2];
#pragma unroll
                for (int i = 0; i < BKV; i += 2) {
                    const float2 a = fma2(make_float2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), sl2x2, mneg);
                    const float2 p = make_float2(ex2(a.x), ex2(a.y));
                    l4[(i >> 1) & 3] = add2(l4[(i >> 1) & 3], p);
                    pk[i >> 1] = pack_bf16x2(p.x, p.y);
                }
                const float2 l2 = add2(add2(l4[0], l4[1]), add2(l4[2], l4[3]));
                l += l2.x + l2.y;
                if (j > 0) {
                    // O and the P columns are free once P_{g-1} V_{g-1} has completed (an
                    // item's first tile: the item before's end already waited for it)
                    ok = mbar_wait(&bar->o_done, (g - 1) & 1, abort_flag, flags);
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
                    }
                }
                // P_g into tensor memory: key pair i of this row in column TM_P + i (the A
                // operand of the PV product, 8 columns per 16 keys)
                tmem_st32u(lane_base + TM_P, pk);
                tmem_st32u(lane_base + TM_P + 32, pk + 32);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar->p_full);
            }
            if (!ok) break;
            // the item's O once its last PV is done; then O is free for the next item
            ok = mbar_wait(&bar->o_done, (g - 1) & 1, abort_flag, flags);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float o[64];
            tmem_ld32(lane_base + TM_O, o);
            tmem_ld32(lane_base + TM_O + 32, o + 32);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->o_free);
            const int bh = w % nbh, q = qt * BQ + r;
            if (q < T) {
                const int row0 = (bh / NH) * T, h = bh % NH;
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}


// ------------------------------------------------------------------ backward
// llm.c §1.8 attention_backward, without atomics and without the (T, T) buffers: P is
// rebuilt from the forward's log-sum-exp L and D = rowsum(dO * O), dS = P * (dP - D).
// Two persistent kernels of one template, one CTA per SM, 576 threads (a TMA warp, an MMA
// warp, two softmax groups of 8 warps), each CTA looping over work items (a 128-row tile
// of one (b, h)), heaviest first:
//   DQ = true   (query-major, runs first): an item is 128 queries; it streams K_j and V_j
//               for j <= the query tile: S = Q K^T, dP = dO V^T, dS = P (dP - D),
//               dQ += dS K.  D of the item's rows is computed here and stored for the
//               other kernel.
//   DQ = false  (key-major): an item is 128 keys; it streams Q_i and dO_i for i >= the key
//               tile, with L and D of the tile's queries copied next to them: S^T = K Q^T,
//               dP^T = V dO^T, P^T and dS^T = P^T (dP^T - D); dV += P^T dO, dK += dS^T Q.
// The item's own rows (Q and dO, or K and V) come by TMA into shared memory and are moved
// by the first softmax group into tensor memory, where they are the A operand of S and
// dP; P and dS are written back there as the A operand of the accumulation products, so
// every MMA reads only its B operand from shared memory (64-column MMAs with A in shared
// memory measured twice as long).  Each streamed 128-row tile is processed as two
// 64-column halves; half g goes to tensor-memory buffer g % 2 (S at its column 0, dP at
// 64) and to softmax group g % 2, whose 8 warps take 32 columns of a row each.  The MMA
// warp keeps two halves' S and dP ahead of the softmax, and the work of consecutive items
// overlaps: the TMA warp streams the next item's tiles as stages free up, the first group
// moves the next item's rows into the second row buffer before the current item's
// accumulators are drained, and the next item's S and dP start as soon as its rows are
// in; only its first accumulation waits for the drain.
// Tensor memory (512 columns): buffers at 0 and 128; accumulators at 256 (dQ, or dV) and
// 320 (dK); two row buffers of 64 columns (the two A operands, 32 packed columns each) at
// 384 and 448, by item parity.
constexpr int BW_NS = 4;  // streamed-tile stages
struct BwdBars {
    uint64_t rt_full, rt_empty, rows_full[2], st_full[BW_NS], st_empty[BW_NS], sdp_full[2], pds_full[2], acc_done,
        acc_free, drain;
    uint32_t tmem_slot;
    int abort;
};
constexpr int BW_ST = 0;                                // stages: A 16 KB + B 16 KB each
constexpr int BW_RT = BW_ST + BW_NS * 2 * TILE;         // the item's row tiles: Q|K, dO|V, O (query-major)
constexpr int BW_STATS = BW_RT + 3 * TILE;              // key-major: per stage L[128], D[128] (raw L)
constexpr int BW_RSTAT = BW_STATS + BW_NS * 2 * 128 * 4;  // query-major: the item's L slice [128] (raw)
constexpr int BW_LD = BW_RSTAT + 128 * 4;               // query-major: [2 row sets][L2 128, D 128]
constexpr int BW_BAR = BW_LD + 2 * 2 * 128 * 4;
constexpr int BWD_SMEM = BW_BAR + (int)sizeof(BwdBars);
constexpr uint32_t TB_COLS = 512, TB_ACC = 256, TB_ACC2 = 320, TB_ROWS = 384;

struct BwdItem {
    int rt, bh, b, h, row0, r0, st0, nst;
};
G2_DEV BwdItem bwd_item(bool dq, int w, int nbh, int ntiles, int T, int NH) {
    BwdItem it;
    const int rank = w / nbh;  // items of the heaviest row tile first
    it.bh = w % nbh;
    it.rt = dq ? ntiles - 1 - rank : rank;
    it.b = it.bh / NH;
    it.h = it.bh % NH;
    it.row0 = it.b * T;
    it.r0 = it.rt * 128;
    it.st0 = dq ? 0 : it.rt;
    it.nst = dq ? it.rt + 1 : ntiles - it.rt;
    return it;
}

template <bool DQ>
__global__ void __launch_bounds__(NTH_BWD, 1)
    attn_bwd_tc_k(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_o, bf16* dqkv, const float* lse, float* Dbuf, int T, int C,
                  int NH, int nbh, int* flags) {
    G2_PDL_ENTRY();
    extern __shared__ __align__(1024) uint8_t smem[];
    BwdBars* bar = reinterpret_cast<BwdBars*>(smem + BW_BAR);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (smem_u32(smem) & 1023) {
        if (threadIdx.x == 0 && flags) atomicOr(flags, G2_FLAG_TIMEOUT);
        return;
    }
    const int ntiles = (T + 127) / 128, nitems = ntiles * nbh;
    const uint32_t rt_bytes = (DQ ? 3 : 2) * TILE;

    if (threadIdx.x == 0) {
        bar->abort = 0;
        mbar_init(&bar->rt_full, 1);
        mbar_init(&bar->rt_empty, 8);       // the first group's warps, done with the row tiles
        for (int i = 0; i < 2; i++) {
            mbar_init(&bar->rows_full[i], 8);  // the first group's warps: rows in tensor memory
            mbar_init(&bar->sdp_full[i], 1);
            mbar_init(&bar->pds_full[i], 8);
        }
        for (int i = 0; i < BW_NS; i++) {
            mbar_init(&bar->st_full[i], 1);
            mbar_init(&bar->st_empty[i], 1);
        }
        mbar_init(&bar->acc_done, 1);
        mbar_init(&bar->acc_free, DQ ? 8 : 16);  // the warps that drain accumulators
        mbar_init(&bar->drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
        tma_prefetch_desc(&tm_qkv);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_o);
    }
    if (warp == 1) tmem_alloc(&bar->tmem_slot, TB_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar->tmem_slot;
    volatile int* abort_flag = &bar->abort;

    if (warp == 0) {
        // ---------------- TMA producer: per item its row tiles, then its streamed tiles
        // through the stage ring (lane 0 issues; all lanes copy statistics that a bulk
        // copy cannot take: a ragged last tile or an unaligned slice)
        int nt = 0;  // streamed tiles issued so far (stage ring position)
        int iss_st[BW_NS];
        for (int i = 0; i < BW_NS; i++) iss_st[i] = -1;
        int iss_rt = -1;
        bool ok = true;
        for (int k = 0, w = item_of(0, blockIdx.x, gridDim.x); ok && w < nitems;
             k++, w = item_of(k, blockIdx.x, gridDim.x)) {
            const BwdItem it = bwd_item(DQ, w, nbh, ntiles, T, NH);
            const int xa = DQ ? C + it.h * HS : it.h * HS;      // streamed K or Q
            const int xb = DQ ? 2 * C + it.h * HS : it.h * HS;  // streamed V (qkv) or dO (dout map)
            const CUtensorMap* mb = DQ ? &tm_qkv : &tm_do;
            // the item's rows, once the first group has released the previous item's
            bool wt = true;
            if (lane == 0) wt = mbar_wait(&bar->rt_empty, (k & 1) ^ 1, abort_flag, flags);
            if (!__shfl_sync(0xffffffffu, wt, 0)) {
                ok = false;
                break;
            }
            const size_t lrow = (size_t)it.bh * T + it.r0;  // first L of the item's rows
            // a bulk copy needs a whole tile inside T and 16-byte aligned addresses
            const bool rt_bulk = DQ && it.r0 + 128 <= T && ((uintptr_t)(lse + lrow) & 15) == 0;
            if (DQ && !rt_bulk) {
                float* rs = reinterpret_cast<float*>(smem + BW_RSTAT);
                for (int i = lane; i < 128; i += 32) rs[i] = it.r0 + i < T ? lse[lrow + i] : INFINITY;
                __syncwarp();
            }
            if (lane == 0) {
                mbar_expect_tx(&bar->rt_full, rt_bytes + (rt_bulk ? 512u : 0u));
                if (DQ) {
                    tma_load_2d(&tm_qkv, &bar->rt_full, smem + BW_RT, it.h * HS, it.row0 + it.r0);          // Q
                    tma_load_2d(&tm_do, &bar->rt_full, smem + BW_RT + TILE, it.h * HS, it.row0 + it.r0);    // dO
                    tma_load_2d(&tm_o, &bar->rt_full, smem + BW_RT + 2 * TILE, it.h * HS, it.row0 + it.r0); // O
                    if (rt_bulk) bulk_load_1d(smem + BW_RSTAT, lse + lrow, 512, &bar->rt_full);
                } else {
                    tma_load_2d(&tm_qkv, &bar->rt_full, smem + BW_RT, C + it.h * HS, it.row0 + it.r0);        // K
                    tma_load_2d(&tm_qkv, &bar->rt_full, smem + BW_RT + TILE, 2 * C + it.h * HS, it.row0 + it.r0);  // V
                }
                iss_rt = k & 1;
                for (int n = BW_NS; n < it.nst; n++) {
                    tma_prefetch_l2(&tm_qkv, xa, it.row0 + (it.st0 + n) * 128);
                    tma_prefetch_l2(mb, xb, it.row0 + (it.st0 + n) * 128);
                }
            }
            for (int n = 0; n < it.nst; n++, nt++) {
                const int s = nt % BW_NS;
                const uint32_t ph = (nt / BW_NS) & 1;
                bool w2 = true;
                if (lane == 0) w2 = mbar_wait(&bar->st_empty[s], ph ^ 1, abort_flag, flags);
                if (!__shfl_sync(0xffffffffu, w2, 0)) {
                    ok = false;
                    break;
                }
                const int q0 = (it.st0 + n) * 128;
                const size_t qrow = (size_t)it.bh * T + q0;
                const bool st_bulk = !DQ && q0 + 128 <= T && ((uintptr_t)(lse + qrow) & 15) == 0 &&
                                     ((uintptr_t)(Dbuf + qrow) & 15) == 0;
                float* Ls = reinterpret_cast<float*>(smem + BW_STATS) + s * 256;
                if (!DQ && !st_bulk) {
                    // L and D of the tile's queries; absent ones get L = +inf (P = 0)
                    for (int i = lane; i < 128; i += 32) {
                        Ls[i] = q0 + i < T ? lse[qrow + i] : INFINITY;
                        Ls[128 + i] = q0 + i < T ? Dbuf[qrow + i] : 0.f;
                    }
                    __syncwarp();  // the statistics are written before lane 0 arrives
                }
                if (lane == 0) {
                    mbar_expect_tx(&bar->st_full[s], 2 * TILE + (st_bulk ? 1024u : 0u));
                    uint8_t* st = smem + BW_ST + s * 2 * TILE;
                    tma_load_2d(&tm_qkv, &bar->st_full[s], st, xa, it.row0 + q0);
                    tma_load_2d(mb, &bar->st_full[s], st + TILE, xb, it.row0 + q0);
                    if (st_bulk) {
                        bulk_load_1d(Ls, lse + qrow, 512, &bar->st_full[s]);
                        bulk_load_1d(Ls + 128, Dbuf + qrow, 512, &bar->st_full[s]);
                    }
                    iss_st[s] = (int)ph;
                }
            }
        }
        if (!ok && lane == 0) {  // wait (bounded) for the copies still in flight before leaving
            unsigned long long t0 = globaltimer();
            if (iss_rt >= 0) {
                while (!mbar_try_wait(&bar->rt_full, (uint32_t)iss_rt) && globaltimer() - t0 < TIMEOUT_NS) {
                }
            }
            for (int s = 0; s < BW_NS; s++) {
                if (iss_st[s] < 0) continue;
                t0 = globaltimer();
                while (!mbar_try_wait(&bar->st_full[s], (uint32_t)iss_st[s]) && globaltimer() - t0 < TIMEOUT_NS) {
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: the whole warp runs the loop converged, one elected
        // lane issues (see umma_bf16_ts_w)
        {
            constexpr uint32_t ID_SDP = make_idesc(64, false, false);  // N = 64 streamed rows
            constexpr uint32_t ID_ACC = make_idesc(HS, false, true);   // N = 64, streamed operand MN-major
            const uint32_t sbase = smem_u32(smem);
            bool ok = true, issued_any = false;
            // every lane waits; a failure in any lane fails the warp
            auto wait_all = [&](uint64_t* b, uint32_t par) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(b, par, abort_flag, flags));
            };
            int nt = 0;  // streamed tiles before this item
            for (int k = 0, w = item_of(0, blockIdx.x, gridDim.x); ok && w < nitems;
                 k++, w = item_of(k, blockIdx.x, gridDim.x)) {
                const BwdItem it = bwd_item(DQ, w, nbh, ntiles, T, NH);
                const int nh = 2 * it.nst;
                const uint32_t rows = tmem + TB_ROWS + (uint32_t)(k & 1) * 64;
                if (!wait_all(&bar->rows_full[k & 1], (k >> 1) & 1)) {
                    ok = false;
                    break;
                }
                // S and dP of half g (tile g/2, its 64 rows from 64 (g%2)) into buffer g%2:
                // A = the item's rows in tensor memory, B = the half's rows (K-major)
                auto issue_sdp = [&](int g) -> bool {
                    const int tn = nt + (g >> 1), hh = g & 1, s = tn % BW_NS;
                    const uint32_t buf = tmem + (uint32_t)(g & 1) * 128;
                    if (hh == 0 && !wait_all(&bar->st_full[s], (tn / BW_NS) & 1)) return false;
                    tc_fence_after();
                    const uint32_t sA = sbase + BW_ST + s * 2 * TILE + hh * 8192, sB = sA + TILE;
#pragma unroll
                    for (int kk = 0; kk < HS / 16; kk++)
                        umma_bf16_ts_w(buf, rows + kk * 8, sdesc(sA + kk * 32, 16, 1024), ID_SDP, kk > 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < HS / 16; kk++)
                        umma_bf16_ts_w(buf + 64, rows + 32 + kk * 8, sdesc(sB + kk * 32, 16, 1024), ID_SDP,
                                       kk > 0 ? 1u : 0u);
                    umma_commit_w(&bar->sdp_full[g & 1]);
                    issued_any = true;
                    return true;
                };
                // the half counter of sdp_full / pds_full phases runs on across items: every
                // item has an even number of halves, so half g of any item uses buffer g % 2
                const int G = 2 * nt;
                ok = issue_sdp(0) && issue_sdp(1);
                for (int g = 0; ok && g < nh; g++) {
                    const int tn = nt + (g >> 1), hh = g & 1, s = tn % BW_NS;
                    if (!wait_all(&bar->pds_full[g & 1], ((G + g) >> 1) & 1) ||
                        (g == 0 && k > 0 && !wait_all(&bar->acc_free, (k - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // accumulation of half g: A = P or dS in the buffer (8 packed columns = 16
                    // rows of the contraction per MMA), B = the half's rows read N-major
                    const uint32_t buf = tmem + (uint32_t)(g & 1) * 128;
                    const uint32_t sA = sbase + BW_ST + s * 2 * TILE + hh * 8192, sB = sA + TILE;
#pragma unroll
                    for (int kk = 0; kk < 64 / 16; kk++) {
                        const uint32_t acc = (g > 0 || kk > 0) ? 1u : 0u;
                        const uint32_t a_off = (kk >> 1) * 32 + (kk & 1) * 8;  // column group kk/2, packed 8 (kk%2)
                        const uint64_t bA = sdesc(sA + kk * 2048, 8192, 1024);
                        if (DQ) {
                            umma_bf16_ts_w(tmem + TB_ACC, buf + 64 + a_off, bA, ID_ACC, acc);  // dQ += dS K
                        } else {
                            const uint64_t bB = sdesc(sB + kk * 2048, 8192, 1024);
                            umma_bf16_ts_w(tmem + TB_ACC, buf + a_off, bB, ID_ACC, acc);        // dV += P^T dO
                            umma_bf16_ts_w(tmem + TB_ACC2, buf + 64 + a_off, bA, ID_ACC, acc);  // dK += dS^T Q
                        }
                    }
                    if (hh == 1) umma_commit_w(&bar->st_empty[s]);  // both halves of the tile are done with it
                    if (g == nh - 1) umma_commit_w(&bar->acc_done);
                    // the buffer of half g+2 is that of half g, whose accumulation was issued just now
                    if (g + 2 < nh && !issue_sdp(g + 2)) ok = false;
                }
                nt += it.nst;
            }
            if (!ok && issued_any) {
                umma_commit_w(&bar->drain);
                if (lane == 0) {
                    unsigned long long t0 = globaltimer();
                    while (!mbar_try_wait(&bar->drain, 0) && globaltimer() - t0 < TIMEOUT_NS) {
                    }
                }
                __syncwarp();
            }
        }
    } else {
        // ---------------- softmax groups: warps 2-9 take the first 64 columns of every
        // streamed tile (even halves), warps 10-17 the second (odd halves); thread = row,
        // sub = which 32 of the half's 64 columns
        const int grp = (warp - 2) >> 3, sub = ((warp - 2) >> 2) & 1;
        const int quarter = warp & 3, r = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float sl2 = LOG2E / sqrtf((float)HS);
        float* LDs = reinterpret_cast<float*>(smem + BW_LD);  // [set][L2 | D][128]
        bool ok = true;
        // The first group moves item k's rows into row buffer k%2 (and, query-major, computes
        // L and D of the rows), then releases the row tiles and announces the rows.
        auto prep_rows = [&](int w, int k) -> bool {
            const BwdItem it = bwd_item(DQ, w, nbh, ntiles, T, NH);
            bool okp = mbar_wait(&bar->rt_full, k & 1, abort_flag, flags);
            if (!__all_sync(0xffffffffu, okp)) return false;
            const uint8_t* src = smem + BW_RT + sub * TILE + r * 128;  // row r of tile sub, 128-byte swizzle
            uint32_t rv[32];
#pragma unroll
            for (int c = 0; c < 8; c++) {
                const uint4 u = *reinterpret_cast<const uint4*>(src + ((c ^ (r & 7)) << 4));
                rv[4 * c] = u.x;
                rv[4 * c + 1] = u.y;
                rv[4 * c + 2] = u.z;
                rv[4 * c + 3] = u.w;
            }
            tmem_st32u(tmem + lane_off + TB_ROWS + (uint32_t)(k & 1) * 64 + sub * 32, rv);
            if (DQ) {
                // D = rowsum(dO * O) of row r from the staged rows (both subs of the row
                // compute it: no exchange, so no barrier a stalled warp could hold up)
                const uint8_t* dor = smem + BW_RT + TILE + r * 128;
                const uint8_t* orr = smem + BW_RT + 2 * TILE + r * 128;
                float D = 0.f;
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    float a8[8], c8[8];
                    Vec8<bf16>::load(reinterpret_cast<const bf16*>(dor + ((c ^ (r & 7)) << 4)), a8);
                    Vec8<bf16>::load(reinterpret_cast<const bf16*>(orr + ((c ^ (r & 7)) << 4)), c8);
#pragma unroll
                    for (int e = 0; e < 8; e++) D += a8[e] * c8[e];
                }
                const float Lraw = reinterpret_cast<const float*>(smem + BW_RSTAT)[r];
                const int q = it.r0 + r;
                if (sub == 0) {
                    float* ld = LDs + (k & 1) * 256;
                    ld[r] = q < T ? Lraw * LOG2E : INFINITY;  // rows past T: P = 0
                    ld[128 + r] = q < T ? D : 0.f;
                    if (q < T) Dbuf[(size_t)it.bh * T + q] = D;
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bar->rt_empty);
                mbar_arrive(&bar->rows_full[k & 1]);
            }
            return true;
        };
        if (grp == 0 && blockIdx.x < nitems) ok = prep_rows(blockIdx.x, 0);
        int nt = 0;
        for (int k = 0, w = item_of(0, blockIdx.x, gridDim.x); w < nitems;
             k++, w = item_of(k, blockIdx.x, gridDim.x)) {
            if (!__all_sync(0xffffffffu, ok)) break;
            const BwdItem it = bwd_item(DQ, w, nbh, ntiles, T, NH);
            const int nh = 2 * it.nst, G = 2 * nt;
            float L2_row = INFINITY, D_row = 0.f;  // query-major: this row's L (log2 units) and D
            if (DQ) {
                ok = mbar_wait(&bar->rows_full[k & 1], (k >> 1) & 1, abort_flag, flags);
                if (!__all_sync(0xffffffffu, ok)) break;
                L2_row = LDs[(k & 1) * 256 + r];
                D_row = LDs[(k & 1) * 256 + 128 + r];
            }
            for (int g = grp; g < nh; g += 2) {
                const int n = g >> 1, tn = nt + n, s = tn % BW_NS;
                ok = mbar_wait(&bar->sdp_full[g & 1], ((G + g) >> 1) & 1, abort_flag, flags);
                // key-major: the stage's statistics (already complete; the wait orders the reads)
                if (!DQ && ok) ok = mbar_wait(&bar->st_full[s], (tn / BW_NS) & 1, abort_flag, flags);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const bool diag = (it.st0 + n) == it.rt;
                const uint32_t tb = tmem + lane_off + (uint32_t)(g & 1) * 128 + sub * 32;
                const float* Ls = reinterpret_cast<const float*>(smem + BW_STATS) + s * 256 + grp * 64 + sub * 32;
                const float* Ds = Ls + 128;
                // 32 columns in two rounds of 16: S and dP in, P and dS (8 packed columns
                // each) written back over the first half of what this thread read
#pragma unroll
                for (int rd = 0; rd < 2; rd++) {
                    uint32_t v[32];  // [0, 16) S, [16, 32) dP
                    tmem_ld16_raw(tb + rd * 16, v);
                    tmem_ld16_raw(tb + 64 + rd * 16, v + 16);
                    tmem_wait_ld_tied32(v);
                    uint32_t pk[8], dk[8];
                    const int cbase = grp * 64 + sub * 32 + rd * 16;  // column within the streamed tile
#pragma unroll
                    for (int c4 = 0; c4 < 16; c4 += 4) {
                        // this column pair's -L (log2 units) and D
                        float2 nL[2], Dc[2];
                        if (DQ) {
                            nL[0] = nL[1] = make_float2(-L2_row, -L2_row);
                            Dc[0] = Dc[1] = make_float2(D_row, D_row);
                        } else {
                            const float4 l4 = *reinterpret_cast<const float4*>(Ls + rd * 16 + c4);
                            const float4 d4 = *reinterpret_cast<const float4*>(Ds + rd * 16 + c4);
                            const float2 nl2e = make_float2(-LOG2E, -LOG2E);
                            nL[0] = mul2(make_float2(l4.x, l4.y), nl2e);
                            nL[1] = mul2(make_float2(l4.z, l4.w), nl2e);
                            Dc[0] = make_float2(d4.x, d4.y);
                            Dc[1] = make_float2(d4.z, d4.w);
                        }
#pragma unroll
                        for (int h = 0; h < 2; h++) {
                            const int e = c4 + 2 * h;
                            const float2 a = fma2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                                                  make_float2(sl2, sl2), nL[h]);
                            float2 p = make_float2(ex2(a.x), ex2(a.y));
                            if (diag) {  // causal: key <= query; DQ rows are queries, key-major rows are keys
                                const int c = cbase + e;
                                if (!(DQ ? c <= r : r <= c)) p.x = 0.f;
                                if (!(DQ ? c + 1 <= r : r <= c + 1)) p.y = 0.f;
                            }
                            const float2 ds = mul2(p, sub2(make_float2(__uint_as_float(v[16 + e]), __uint_as_float(v[17 + e])), Dc[h]));
                            pk[e >> 1] = pack_bf16x2(p.x, p.y);
                            dk[e >> 1] = pack_bf16x2(ds.x, ds.y);
                        }
                    }
                    // packed columns 8 rd .. 8 rd + 7 of this thread's 32: already read
                    if (!DQ) tmem_st8(tb + 8 * rd, pk);
                    tmem_st8(tb + 64 + 8 * rd, dk);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar->pds_full[g & 1]);
            }
            if (!__all_sync(0xffffffffu, ok)) break;
            // the next item's rows go into the other row buffer now (its S and dP can start
            // while this item's accumulators drain); that buffer's last reader was the item
            // before this one, all of whose products completed before its drain
            const int w_next = item_of(k + 1, blockIdx.x, gridDim.x);
            if (grp == 0 && w_next < nitems) {
                ok = prep_rows(w_next, k + 1);
                if (!__all_sync(0xffffffffu, ok)) break;
            }
            ok = mbar_wait(&bar->acc_done, k & 1, abort_flag, flags);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            // DQ: group 0 stores dQ (32 columns per sub); key-major: group 0 dV, group 1 dK
            if (!DQ || grp == 0) {
                const int grow = it.r0 + r;
                const float scale = 1.0f / sqrtf((float)HS);
                bf16* base = dqkv + (size_t)(it.row0 + grow) * 3 * C + it.h * HS;
                bf16* dst = DQ ? base : (grp ? base + C : base + 2 * C);
                const float mul = (DQ || grp) ? scale : 1.0f;
                const uint32_t t0 = tmem + lane_off + (DQ ? TB_ACC : (grp ? TB_ACC2 : TB_ACC)) + sub * 32;
                float a[32];
                tmem_ld32(t0, a);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar->acc_free);  // the accumulator columns are read
                if (grow < T) {
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 8; e++) y[e] = a[i + e] * mul;
                        Vec8<bf16>::store(dst + sub * 32 + i, y);
                    }
                }
            }
            nt += it.nst;
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
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 148;
    }
    const int nbh = B * NH, items = ((T + atc::BQ - 1) / atc::BQ) * nbh;
    const int grid = items < 2 * sms ? items : 2 * sms;  // persistent: two CTAs per SM
    ::g2::launch_k(atc::attn_fwd_tc_k, grid, atc::NTH, atc::FWD_SMEM, s, tm, (bf16*)out, lse, T, C, NH, nbh, flags);
    return cudaGetLastError();
}

cudaError_t attention_backward_tc(void* dqkv, const void* dout, const void* qkv, const void* out, const float* lse,
                                  int B, int T, int C, int NH, float* Dbuf, int* flags, cudaStream_t s) {
    CUtensorMap tq, td, to;
    if (((uintptr_t)dout & 15) || ((uintptr_t)out & 15) || ((uintptr_t)dqkv & 15) || (C % 8))
        return cudaErrorNotSupported;
    if (!tc::make_map(&tq, qkv, 3ull * C, (uint64_t)B * T, 3ull * C, 64, 128) ||
        !tc::make_map(&td, dout, (uint64_t)C, (uint64_t)B * T, (uint64_t)C, 64, 128) ||
        !tc::make_map(&to, out, (uint64_t)C, (uint64_t)B * T, (uint64_t)C, 64, 128))
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
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 148;
    }
    const int nbh = B * NH, items = ((T + 127) / 128) * nbh;
    const int grid = items < sms ? items : sms;  // persistent: one CTA per SM
    // the query-major kernel also writes D = rowsum(dO * O), which the key-major one reads
    ::g2::launch_k(atc::attn_bwd_tc_k<true>, grid, atc::NTH_BWD, atc::BWD_SMEM, s, tq, td, to, (bf16*)dqkv, lse, Dbuf, T,
                                                                                 C, NH, nbh, flags);
    ::g2::launch_k(atc::attn_bwd_tc_k<false>, grid, atc::NTH_BWD, atc::BWD_SMEM, s, tq, td, to, (bf16*)dqkv, lse, Dbuf,
                                                                                  T, C, NH, nbh, flags);
    return cudaGetLastError();
}

}  // namespace g2
