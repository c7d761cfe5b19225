// Tensor-core GEMM for sm_103a: D = epi(A . B^T) with bf16 operands and fp32
// accumulation in tensor memory (tcgen05), operands staged by TMA.
//
// The three products of a linear layer (llm.c annotated listing §1.5 matmul_forward,
// §1.6 matmul_backward) all run here:
//   forward  X.W^T   A K-major, B K-major      (+bias, +residual, or GELU epilogue)
//   dgrad    dY.W    A K-major, B N-major      (optionally times GELU'(pre-activation))
//   wgrad    dY^T.X  A M-major, B N-major      (fp32 out; split-K with a fixed-order sum)
//
// Structure (one persistent CTA per SM, 320 threads).  A tile is 256 rows x BN columns:
// two 128-row halves that share every B stage, so each SM receives 64 KB of operands per
// 1024 clocks of BN = 256 tensor work -- the rate its TMA ingress sustains (about 64
// bytes per clock); 128-row tiles would need 1.5 x that.
//   warp 0    TMA producer: one elected lane streams the 256 x 64 (A) and BN x 64 (B)
//             bf16 tiles of each K block into a ring of shared-memory stages (128-byte
//             swizzle).
//   warp 1    allocates all 512 tensor-memory columns; one lane issues tcgen05.mma
//             (M = 128 per half, N = BN, K = 16) into the tile's two fp32 accumulator
//             halves (2 x BN columns; two such buffers when BN = 128) and commits to
//             mbarriers that free the stage / publish the accumulator.
//   warps 2-9 epilogue, warps 2-5 for the first half and 6-9 for the second (each warp one
//             32-lane quarter): tcgen05.ld, fused epilogue math, bf16/fp32 stores; then
//             release the accumulator.
// Every mbarrier wait is bounded (about 2 s): on expiry the kernel raises a flag, drains
// what it issued and returns instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "gemm_tc.h"
#include "tc_ptx.cuh"

namespace g2 {
namespace tc {

constexpr int BM = 128, BK = 64, UMMA_K = 16;  // rows per MMA (one accumulator half)
// With fp32 operands (TF32 products) a K block is the same 128 bytes per row: 32
// elements, four MMAs of K = 8.
template <bool TF> struct OperandT {
    static constexpr int BKE = TF ? 32 : 64;   // elements per K block
    static constexpr int UK = TF ? 8 : 16;     // K per MMA instruction
};
constexpr int GROUP_M = 8;     // tile order: m fastest within groups of GROUP_M row tiles

// epilogues: bf16 store (+bias), GELU (two bf16 outputs), times GELU' of the pre-activation,
// fp32 split-K partial, fp32 store, bf16 store of + bias + residual
enum { E_STORE = 0, E_GELU = 1, E_GELU_BWD = 2, E_PARTIAL = 3, E_STORE_F32 = 4, E_STORE_RES = 5 };
template <int EPI> struct EpiOut {
    static constexpr bool F32 = EPI == E_PARTIAL || EPI == E_STORE_F32;
    static constexpr int CW = F32 ? 32 : 64;           // columns per 128-byte staged row
    static constexpr int NOUT = EPI == E_GELU ? 2 : 1;  // staged outputs per chunk
    // a bf16 (M,N) input read per chunk (pre-activation or residual): TMA-loaded one chunk
    // ahead into two staging buffers
    static constexpr bool IN = EPI == E_GELU_BWD || EPI == E_STORE_RES;
};

struct Params {
    int M, N, K;
    int tiles_m, tiles_n, splits, kb_per_split, num_kb, num_units;  // units: (row tile, col tile, split)
    void* D;
    long long ldd;
    int d_f32;
    const float* bias;
    const bf16* R;
    long long ldr;
    bf16* D2;
    long long ldd2;
    const bf16* P;
    long long ldp;
    float* ws;  // split-K partials: [splits][M][N] fp32
    float* cs_part;  // GELU' epilogue: column sums of the stored output per 32-row group, or null
    int* flags;
};

// PAIR: the tile is computed by a cluster of two CTAs on two SMs (cta_group::2): each CTA
// holds 128 rows of A and BN/2 rows of B per stage and receives its 128 accumulator rows.
template <int BN, int BMT, int EPI, bool PAIR = false>
struct Cfg {
    static constexpr int HALVES = BMT / BM;                 // 128-row accumulator halves per tile
    // The GELU' epilogue (FC-projection input gradient) is latency-bound with one epilogue
    // warp per SM sub-partition: on 128-row tiles it gets two warps per 32-lane quarter,
    // each draining half of the tile's columns, with one staged-input buffer each so the
    // pipeline keeps three stages (measured: 186 -> 162 us per layer at B=32, T=1024;
    // two input buffers and two stages: 189 us).  The residual epilogue gains nothing.
    // Pair tiles finish a K = 768 mainloop in about 6,000 clocks, so their bias + GELU and
    // residual epilogues get the column split too.
    static constexpr int COLSPLIT =
        (HALVES == 1 && (EPI == E_GELU_BWD || (PAIR && (EPI == E_GELU || EPI == E_STORE_RES)))) ? 2 : 1;
    static constexpr int EPI_WARPS = 4 * HALVES * COLSPLIT;  // per 32-lane quarter, per half, per column part
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;     // + TMA warp + MMA warp
    static constexpr int NIN = COLSPLIT == 2 ? 1 : 2;       // staged-input buffers per warp
    static constexpr int A_BYTES = BMT * BK * 2;
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;     // rows of B this CTA stages
    static constexpr int B_BYTES = B_ROWS * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // each epilogue warp stages 32 rows x 128 bytes per output for the TMA store
    // output staging: two sets on 128-row tiles (a chunk's stores need not have finished
    // reading before the next chunk is staged), one set on 256-row tiles (their 8
    // epilogue warps would otherwise take the shared memory of a pipeline stage)
    static constexpr int STG_BUFS = (HALVES == 1 && COLSPLIT == 1) ? 2 : 1;
    static constexpr int EPI_WARP_BYTES = (EpiOut<EPI>::NOUT * STG_BUFS + (EpiOut<EPI>::IN ? NIN : 0)) * 4096;
    static constexpr int EPI_BYTES = EPI_WARPS * EPI_WARP_BYTES;
    static constexpr int SMEM_LIMIT = 227 * 1024 - 1024 /*align*/ - 512 /*barriers*/;
    static constexpr int STAGES_FIT = (SMEM_LIMIT - EPI_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
    static constexpr int ACC_COLS = HALVES * BN;
    static constexpr int ACC_BUFS = (512 / ACC_COLS) >= 2 ? 2 : 1;
    static constexpr int TMEM_COLS = 512;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + 1024 /*align*/ + 512 /*barriers*/;
    static_assert(STAGES >= 2, "shared memory too small for the pipeline");
};

// Work unit u: row tile m_blk (BMT rows), column tile n_blk, K split `split`.  Row tiles
// run fastest within groups of GROUP_M, so concurrently running CTAs share B tiles in L2.
G2_DEV void unit_coords(const Params& p, int u, int& m_blk, int& n_blk, int& split) {
    int per = p.tiles_m * p.tiles_n;
    split = u / per;
    int t = u % per;
    int group_size = GROUP_M * p.tiles_n;
    int group = t / group_size;
    int first_m = group * GROUP_M;
    int gsz = min(p.tiles_m - first_m, GROUP_M);
    int r = t % group_size;
    m_blk = first_m + r % gsz;
    n_blk = r / gsz;
}

// ------------------------------------------------------------------ epilogue
// One chunk of CW columns of this thread's row (gm): the fused math on the fp32
// accumulator values, then the row written into the warp's staging buffer (32 rows x 128
// bytes, the 128-byte swizzle a TMA store expects).  Columns past N carry garbage the
// store does not write.
// this thread's row (64 bf16) of a staged input buffer, unswizzled
G2_DEV void unstage_row_bf16(const uint8_t* buf, int lane, float* x) {
    const uint8_t* row = buf + lane * 128;
#pragma unroll
    for (int c = 0; c < 8; c++) {
        const uint4 u = *reinterpret_cast<const uint4*>(row + ((c ^ (lane & 7)) << 4));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float2 f = __bfloat1622float2(h[i]);
            x[8 * c + 2 * i] = f.x;
            x[8 * c + 2 * i + 1] = f.y;
        }
    }
}

template <int EPI>
G2_DEV void epilogue_math(const Params& p, float* v, const uint8_t* in_row_buf, int lane, int gn0) {
    constexpr int CW = EpiOut<EPI>::CW;
    const int N = p.N;
    const bool full = gn0 + CW <= N;
    if (EPI == E_PARTIAL) return;
    if (EPI == E_GELU_BWD) {
        float x[CW];
        unstage_row_bf16(in_row_buf, lane, x);
#pragma unroll
        for (int i = 0; i < CW; i += 2) {
            const float2 g = gelu_grad2(make_float2(x[i], x[i + 1]));
            v[i] *= g.x;
            v[i + 1] *= g.y;
        }
        return;
    }
    if (p.bias) {
        if (full) {
#pragma unroll
            for (int i = 0; i < CW; i += 4) {
                float4 b = *reinterpret_cast<const float4*>(p.bias + gn0 + i);
                v[i] += b.x; v[i + 1] += b.y; v[i + 2] += b.z; v[i + 3] += b.w;
            }
        } else {
            for (int i = 0; i < CW; i++)
                if (gn0 + i < N) v[i] += p.bias[gn0 + i];
        }
    }
    if (EPI == E_STORE_RES) {
        float x[CW];
        unstage_row_bf16(in_row_buf, lane, x);
#pragma unroll
        for (int i = 0; i < CW; i++) v[i] += x[i];
    }
}

// this thread's row of a staging buffer: 8 chunks of 16 bytes, chunk c at (c ^ (row & 7))
template <bool F32>
G2_DEV void stage_row(uint8_t* buf, int lane, const float* v) {
    uint8_t* row = buf + lane * 128;
#pragma unroll
    for (int c = 0; c < 8; c++) {
        uint4 u;
        if (F32) {
            u = make_uint4(__float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]), __float_as_uint(v[4 * c + 2]),
                           __float_as_uint(v[4 * c + 3]));
        } else {
            __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * c], v[8 * c + 1]);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * c + 2], v[8 * c + 3]);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * c + 4], v[8 * c + 5]);
            __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * c + 6], v[8 * c + 7]);
            u = make_uint4(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1),
                           *reinterpret_cast<uint32_t*>(&h2), *reinterpret_cast<uint32_t*>(&h3));
        }
        *reinterpret_cast<uint4*>(row + ((c ^ (lane & 7)) << 4)) = u;
    }
}

// ------------------------------------------------------------------ the kernel
template <int BN, int BMT, bool A_MN, bool B_MN, int EPI, bool TF = false, bool PAIR = false>
__global__ void __launch_bounds__(Cfg<BN, BMT, EPI, PAIR>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD2,
                   const __grid_constant__ CUtensorMap tmX, const Params p) {
    G2_PDL_ENTRY();
    using CF = Cfg<BN, BMT, EPI, PAIR>;
    using EO = EpiOut<EPI>;
    using OT = OperandT<TF>;
    static_assert(!TF || (!A_MN && !B_MN), "TF32 products take K-major operands only");
    static_assert(!PAIR || (BMT == BM && !TF && BN == 256), "CTA pairs: 128 rows per CTA, bf16, BN = 256");
    // a work unit covers TILE_M rows: a CTA pair splits them 128 / 128 by cluster rank
    constexpr int TILE_M = PAIR ? 2 * BM : BMT;
    const uint32_t rank = PAIR ? cluster_rank() : 0u;
    const int u0 = PAIR ? (int)cluster_id_x() : (int)blockIdx.x;
    const int ustep = PAIR ? (int)num_clusters_x() : (int)gridDim.x;
    constexpr int S = CF::STAGES, NB = CF::ACC_BUFS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* epi_smem = smem + S * CF::STAGE_BYTES;  // staging for the TMA stores
    uint64_t* bars = (uint64_t*)(epi_smem + CF::EPI_BYTES);
    uint64_t* full_bar = bars;                  // [S]
    uint64_t* empty_bar = bars + S;             // [S]
    uint64_t* tfull_bar = bars + 2 * S;         // [NB]
    uint64_t* tempty_bar = bars + 2 * S + NB;   // [NB]
    uint64_t* drain_bar = bars + 2 * S + 2 * NB;
    uint64_t* in_bar = drain_bar + 1;  // [EPI_WARPS][2]: staged epilogue inputs
    uint32_t* tmem_slot = (uint32_t*)(in_bar + 2 * CF::EPI_WARPS);
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        s_abort = 0;
        // a pair's leader: both CTAs' epilogue warps release an accumulator
        const bool lead = PAIR && rank == 0;
        for (int i = 0; i < S; i++) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], 1);
        }
        for (int i = 0; i < NB; i++) {
            mbar_init(&tfull_bar[i], 1);
            mbar_init(&tempty_bar[i], lead ? 2 * CF::EPI_WARPS : CF::EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        for (int i = 0; i < 2 * CF::EPI_WARPS; i++) mbar_init(&in_bar[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmD);
    }
    if (warp == 1) {
        if constexpr (PAIR)
            tmem_alloc_pair(tmem_slot, CF::TMEM_COLS);
        else
            tmem_alloc(tmem_slot, CF::TMEM_COLS);
    }
    tc_fence_before();
    if (PAIR)
        cluster_sync();  // both CTAs' barriers and tensor memory exist before any cross-CTA signal
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    volatile int* abort_flag = &s_abort;

    if (warp == 0) {
        // ---------------- TMA producer (a pair: each CTA loads its halves; both halves of a
        // stage complete on the leader's barrier, which expects the bytes of both)
        if (lane == 0) {
            const uint32_t lead_full = PAIR ? mapa_rank(smem_u32(full_bar), 0) : 0u;
            int stage = 0;
            uint32_t phase = 0;
            int issued_phase[S];
            for (int i = 0; i < S; i++) issued_phase[i] = -1;
            bool ok = true;
            for (int u = u0; u < p.num_units && ok; u += ustep) {
                int mb, nb, sp;
                unit_coords(p, u, mb, nb, sp);
                int kb0 = sp * p.kb_per_split, kb1 = min(p.num_kb, kb0 + p.kb_per_split);
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, p.flags)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * CF::STAGE_BYTES;
                    uint8_t* sb = sa + CF::A_BYTES;
                    if (!PAIR || rank == 0) mbar_expect_tx(&full_bar[stage], (PAIR ? 2 : 1) * CF::STAGE_BYTES);
                    const int k0 = kb * OT::BKE;
                    const int arow = mb * TILE_M + (int)rank * BM;           // this CTA's A rows
                    const int bcol = nb * BN + (int)rank * CF::B_ROWS;      // and its B rows (N)
                    auto load = [&](const CUtensorMap* tm, void* dst, int x, int y) {
                        if constexpr (PAIR)
                            tma_load_2d_pair(tm, lead_full + (uint32_t)stage * 8u, dst, x, y);
                        else
                            tma_load_2d(tm, &full_bar[stage], dst, x, y);
                    };
                    if (!A_MN) {
                        load(&tmA, sa, k0, arow);
                    } else {
#pragma unroll
                        for (int j = 0; j < BMT / 64; j++) load(&tmA, sa + j * 64 * BK * 2, arow + 64 * j, k0);
                    }
                    if (!B_MN) {
                        load(&tmB, sb, k0, bcol);
                    } else {
#pragma unroll
                        for (int j = 0; j < CF::B_ROWS / 64; j++) load(&tmB, sb + j * 64 * BK * 2, bcol + 64 * j, k0);
                    }
                    issued_phase[stage] = (int)phase;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok && (!PAIR || rank == 0)) {
                // drain: wait (bounded) for every load still in flight before returning (the
                // leader's barriers also count the second CTA's loads)
                for (int i = 0; i < S; i++) {
                    if (issued_phase[i] < 0) continue;
                    unsigned long long t0 = globaltimer();
                    while (!mbar_try_wait(&full_bar[i], (uint32_t)issued_phase[i]) &&
                           globaltimer() - t0 < TIMEOUT_NS) {
                    }
                }
            } else if (!ok) {
                // the second CTA cannot observe its loads: give those issued time to land
                const unsigned long long t0 = globaltimer();
                while (globaltimer() - t0 < 100000ull) {
                }
            }
        }
    } else if (warp == 1 && PAIR && rank != 0) {
        // ---------------- the pair's second CTA issues no MMAs
    } else if (warp == 1) {
        // ---------------- MMA issuer (the leader of a pair issues for both CTAs)
        if (lane == 0) {
            constexpr uint32_t IDESC = TF ? make_idesc_tf32(BN) : make_idesc(BN, A_MN, B_MN, PAIR ? 2 * BM : BM);
            // completion of the MMAs issued so far, as an arrive on this CTA's barrier and, for
            // a pair, on the same barrier of the second CTA
            auto commit_both = [&](uint64_t* b) {
                if constexpr (PAIR) {
                    umma_commit_pair(smem_u32(b));
                    umma_commit_pair(mapa_rank(smem_u32(b), 1));
                } else {
                    umma_commit(b);
                }
            };
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            bool issued_any = false;
            for (int u = u0; u < p.num_units && ok; u += ustep) {
                int mb, nb, sp;
                unit_coords(p, u, mb, nb, sp);
                int kb0 = sp * p.kb_per_split, kb1 = min(p.num_kb, kb0 + p.kb_per_split);
                if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1, abort_flag, p.flags)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * CF::ACC_COLS);
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!mbar_wait(&full_bar[stage], phase, abort_flag, p.flags)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * CF::STAGE_BYTES);
                    const uint32_t sb = sa + CF::A_BYTES;
#pragma unroll
                    for (int hh = 0; hh < CF::HALVES; hh++) {
                        // rows 128 hh.. of the tile: 16 KB into the A stage in either layout
                        const uint32_t sah = sa + hh * (BM * BK * 2);
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; k++) {
                            uint64_t ad, bd;
                            if (!A_MN)
                                ad = sdesc(sah + k * UMMA_K * 2, 16, 1024);
                            else
                                ad = sdesc(sah + k * UMMA_K * 128, 64 * BK * 2, 1024);
                            if (!B_MN)
                                bd = sdesc(sb + k * UMMA_K * 2, 16, 1024);
                            else
                                bd = sdesc(sb + k * UMMA_K * 128, 64 * BK * 2, 1024);
                            // K-major: the k-th MMA's operands start 32 bytes further along the
                            // 128-byte row (16 bf16 or 8 fp32)
                            if constexpr (TF)
                                umma_tf32(d_tmem + hh * BN, ad, bd, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
                            else if constexpr (PAIR)
                                umma_bf16_pair(d_tmem + hh * BN, ad, bd, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
                            else
                                umma_bf16(d_tmem + hh * BN, ad, bd, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
                        }
                    }
                    issued_any = true;
                    commit_both(&empty_bar[stage]);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                commit_both(&tfull_bar[acc]);
                if (++acc == NB) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            if (!ok && issued_any) {
                // drain: all MMAs issued so far complete before this commit arrives
                if constexpr (PAIR)
                    umma_commit_pair(smem_u32(drain_bar));
                else
                    umma_commit(drain_bar);
                unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(drain_bar, 0) && globaltimer() - t0 < TIMEOUT_NS) {
                }
            }
        }
    } else {
        // ---------------- epilogue warps: warps 2-5 drain the first 128-row half of the tile,
        // warps 6-9 the second (256-row tiles) or the second half of the columns (split
        // columns); each warp its 32-lane quarter
        const int ew = warp - 2;
        const int quarter = warp & 3;  // TMEM lanes [32*quarter, 32*quarter + 32)
        const int hh = CF::COLSPLIT == 1 ? (ew >> 2) : 0;
        const int col0 = CF::COLSPLIT == 1 ? 0 : (ew >> 2) * (BN / CF::COLSPLIT);  // first column of this warp
        const int row_in_tile = hh * BM + quarter * 32 + lane;
        uint8_t* stg0 = epi_smem + ew * CF::EPI_WARP_BYTES;            // this warp's staging sets
        uint8_t* inb = stg0 + EO::NOUT * CF::STG_BUFS * 4096;          // its input buffers
        int sbuf = 0;       // staging set of the next chunk
        int newest_set = -1;  // (lane 0) set read by the most recently committed store group
        uint64_t* ibar = in_bar + 2 * ew;
        uint32_t in_par = 0;  // bit b: parity of input buffer b's next completion
        int acc = 0;
        uint32_t acc_phase = 0;
        // staged inputs: with NIN buffers, buffer b holds chunks b, b+NIN, ... of a tile; a
        // chunk's load is issued NIN chunks ahead (the first NIN before the accumulator is ready)
        constexpr int NIN = CF::NIN;
        int pend = 0;  // bit b: a load into input buffer b is in flight, not yet consumed
        auto issue_in = [&](int b, int gcol, int grow) {
            if (lane == 0) {
                mbar_expect_tx(&ibar[b], 4096);
                tma_load_2d(&tmX, &ibar[b], inb + b * 4096, gcol, grow);
            }
            pend |= 1 << b;
        };
        auto drain_in = [&]() {  // let issued loads land before the warp leaves (bounded)
            if (lane == 0) {
                for (int b = 0; b < NIN; b++) {
                    if (!((pend >> b) & 1)) continue;
                    unsigned long long t0 = globaltimer();
                    while (!mbar_try_wait(&ibar[b], (in_par >> b) & 1) && globaltimer() - t0 < TIMEOUT_NS) {
                    }
                }
            }
            __syncwarp();
        };
        for (int u = u0; u < p.num_units; u += ustep) {
            int mb, nb, sp;
            unit_coords(p, u, mb, nb, sp);
            const int gm = mb * TILE_M + (int)rank * BM + row_in_tile;
            const int gm0 = gm - lane;  // first row of this warp's 32
            constexpr int NCH = BN / EO::CW / CF::COLSPLIT;  // chunks of this warp
            if (EO::IN) {
                __syncwarp();  // the input buffers were read by the previous tile's chunks
#pragma unroll
                for (int b = 0; b < NIN && b < NCH; b++) issue_in(b, nb * BN + col0 + b * EO::CW, gm0);
            }
            bool ok = mbar_wait(&tfull_bar[acc], acc_phase, abort_flag, p.flags);
            if (!__all_sync(0xffffffffu, ok)) {  // the warp leaves together
                if (EO::IN) drain_in();
                break;
            }
            tc_fence_after();
            const uint32_t trow = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * CF::ACC_COLS + hh * BN);
            bool in_ok = true;
#pragma unroll 1
            for (int ch = 0; ch < NCH; ch++) {
                const int c0 = col0 + ch * EO::CW;
                const int gn0 = nb * BN + c0;
                const int ib = ch % NIN;
                float v[EO::CW];
                {  // both halves of the chunk in flight, one wait
                    uint32_t r[EO::CW];
                    tmem_ld32_raw(trow + c0, r);
                    if (EO::CW == 64) tmem_ld32_raw(trow + c0 + 32, r + 32);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < EO::CW; i++) v[i] = __uint_as_float(r[i]);
                }
                if (EO::IN) {
                    const bool ok_in = mbar_wait(&ibar[ib], (in_par >> ib) & 1, abort_flag, p.flags);
                    if (__all_sync(0xffffffffu, ok_in)) {
                        in_par ^= 1u << ib;
                        pend &= ~(1 << ib);
                    } else {
                        in_ok = false;  // the load stays pending: drained below
                    }
                }
                epilogue_math<EPI>(p, v, inb + ib * 4096, lane, gn0);
                if (EO::IN && in_ok && ch + NIN < NCH) {
                    __syncwarp();  // every lane has read buffer ib
                    issue_in(ib, gn0 + NIN * EO::CW, gm0);
                }
                // the stores that last read this staging set have finished reading it: every
                // group but the newest has; the newest too unless it reads the other set
                const int set = sbuf;
                uint8_t* stg = stg0 + set * (EO::NOUT * 4096);
                if (CF::STG_BUFS == 2) sbuf ^= 1;
                if (lane == 0) {
                    if (CF::STG_BUFS == 2 && newest_set != set)
                        bulk_wait_read1();
                    else
                        bulk_wait_read0();
                }
                __syncwarp();
                stage_row<EO::F32>(stg, lane, v);
                if (EPI == E_GELU) {
#pragma unroll
                    for (int i = 0; i < EO::CW; i += 2) {
                        const float2 gl = gelu2(make_float2(v[i], v[i + 1]));
                        v[i] = gl.x;
                        v[i + 1] = gl.y;
                    }
                    stage_row<false>(stg + 4096, lane, v);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0 && gm0 < p.M && gn0 < p.N && in_ok) {
                    if (EPI == E_PARTIAL)
                        tma_store_3d(&tmD, stg, gn0, gm0, sp);
                    else
                        tma_store_2d(&tmD, stg, gn0, gm0);
                    if (EPI == E_GELU) tma_store_2d(&tmD2, stg + 4096, gn0, gm0);
                    bulk_commit();
                    newest_set = set;
                }
                if constexpr (EPI == E_GELU_BWD) {
                    // the bias gradient of this pre-activation: lane l reads columns 2l and
                    // 2l + 1 of the warp's 32 staged rows (the stored bf16 values, 4-byte
                    // words one row apart, conflict-free) and adds them in row order; the
                    // TMA store reads the same buffer meanwhile.  Rows past M are zeros
                    // (zero-filled operand and pre-activation rows).
                    if (p.cs_part && gm0 < p.M && in_ok) {
                        const uint8_t* colp = stg + ((lane & 3) << 2);
                        float2 cs = make_float2(0.f, 0.f);
#pragma unroll
                        for (int r = 0; r < 32; r++) {
                            const uint32_t w =
                                *reinterpret_cast<const uint32_t*>(colp + r * 128 + ((((lane >> 2) ^ r) & 7) << 4));
                            cs = add2(cs, make_float2(bf16_lo(w), bf16_hi(w)));
                        }
                        const int j = gn0 + 2 * lane;
                        if (j < p.N) *reinterpret_cast<float2*>(p.cs_part + (size_t)(gm0 >> 5) * p.N + j) = cs;
                    }
                }
                if (!in_ok) {
                    // a wait gave up: let the loads already issued land before leaving
                    drain_in();
                    break;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {  // a pair's accumulator is free once both CTAs have read theirs
                if (PAIR && rank != 0)
                    mbar_arrive_remote(mapa_rank(smem_u32(&tempty_bar[acc]), 0));
                else
                    mbar_arrive(&tempty_bar[acc]);
            }
            if (++acc == NB) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        if (lane == 0) bulk_wait0();  // this warp's stores are complete before the CTA ends
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // neither CTA leaves while the other may still signal it
    tc_fence_after();
    if (warp == 1) {
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, CF::TMEM_COLS);
        else
            tmem_dealloc(tmem_base, CF::TMEM_COLS);
    }
}

// Fixed-order sum of the split-K partials: out[i] = sum_s ws[s][i].
__global__ void splitk_reduce_k(float* out, long long ldo, const float* ws, int M, int N, int splits) {
    G2_PDL_ENTRY();
    size_t n = (size_t)M * N;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        float a = 0.f;
        for (int s = 0; s < splits; s++) a += ws[(size_t)s * n + i];
        int m = (int)(i / N), c = (int)(i % N);
        out[(size_t)m * ldo + c] = a;
    }
}

// The same sum four columns at a time (N and ldo multiples of 4, 16-byte aligned buffers,
// M * N / 4 < 2^31): splits added in the same order from 0, so the result is bitwise that
// of splitk_reduce_k, with one 32-bit division per four elements instead of a 64-bit one
// per element.
__global__ void splitk_reduce4_k(float* out, long long ldo, const float* ws, int M, int N, int splits) {
    G2_PDL_ENTRY();
    const int n4 = N / 4;
    const unsigned nv = (unsigned)M * (unsigned)n4;
    const size_t n = (size_t)M * N;
    for (unsigned v = blockIdx.x * blockDim.x + threadIdx.x; v < nv; v += gridDim.x * blockDim.x) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 0; sp < splits; sp++) {
            const float4 b = reinterpret_cast<const float4*>(ws + (size_t)sp * n)[v];
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        const unsigned m = v / (unsigned)n4, c = (v - m * (unsigned)n4) * 4u;
        *reinterpret_cast<float4*>(out + (size_t)m * ldo + c) = a;
    }
}

// The same sum with the forward epilogue of a split product: v = sum_s ws[s][m][n]
// (+ bias[n]) (+ R[m,n]); D = v (bf16, or fp32 with d_f32); with D2, D2 = gelu(v) from the
// unrounded v (as the fused GELU epilogue does).
__global__ void splitk_epilogue_k(void* D, long long ldd, int d_f32, const float* ws, int M, int N, int splits,
                                  const float* bias, const bf16* R, long long ldr, bf16* D2, long long ldd2) {
    G2_PDL_ENTRY();
    size_t n = (size_t)M * N;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        float a = 0.f;
        for (int s = 0; s < splits; s++) a += ws[(size_t)s * n + i];
        const int m = (int)(i / N), c = (int)(i % N);
        if (bias) a += bias[c];
        if (R) a += __bfloat162float(R[(size_t)m * ldr + c]);
        if (d_f32)
            ((float*)D)[(size_t)m * ldd + c] = a;
        else
            ((bf16*)D)[(size_t)m * ldd + c] = __float2bfloat16_rn(a);
        if (D2) D2[(size_t)m * ldd2 + c] = __float2bfloat16_rn(gelu_tanh_fast(a));
    }
}

// ------------------------------------------------------------------ host side
static int num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

// Launch of the fixed-order split-K sum: the four-column form where it applies.
static void launch_splitk_reduce(float* out, long long ldo, const float* ws, int M, int N, int splits,
                                 cudaStream_t s) {
    const size_t n = (size_t)M * N;
    const bool vec = (N % 4) == 0 && (ldo % 4) == 0 && (((uintptr_t)out | (uintptr_t)ws) & 15) == 0 &&
                     n / 4 < (size_t)1 << 31;
    const size_t work = vec ? n / 4 : n;
    const unsigned blocks = (unsigned)std::min<size_t>((work + 255) / 256, (size_t)num_sms() * 8);
    if (vec)
        ::g2::launch_k(splitk_reduce4_k, blocks, 256, 0, s, out, ldo, ws, M, N, splits);
    else
        ::g2::launch_k(splitk_reduce_k, blocks, 256, 0, s, out, ldo, ws, M, N, splits);
}

// Tile mode of a bf16 product: 128- or 256-row tiles on one SM each, or TILE_PAIR: 256-row
// tiles computed by a cluster of two CTAs (128 rows each, cta_group::2).
constexpr int TILE_PAIR = 2;

// Clusters of two CTAs of the pair kernel that can be resident at once (0: pairs are not
// available), from the occupancy calculator on one representative instantiation: every
// pair instantiation takes the whole shared memory of its SM.
static int pair_max_clusters() {
    static int n = -1;
    static std::once_flag once;
    std::call_once(once, [] {
        using CF = Cfg<256, 128, E_STORE, true>;
        auto kern = gemm_tc_kernel<256, 128, false, false, E_STORE, false, true>;
        int v = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_BYTES) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * num_sms());
            cfg.blockDim = dim3(CF::THREADS);
            cfg.dynamicSmemBytes = CF::SMEM_BYTES;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&v, kern, &cfg) != cudaSuccess) {
                v = 0;
                cudaGetLastError();
            }
        } else {
            cudaGetLastError();
        }
        n = v;
    });
    return n;
}

template <int BN, int BMT, bool A_MN, bool B_MN, int EPI, bool TF = false, bool PAIR = false>
static cudaError_t launch_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td,
                            const CUtensorMap& td2, const CUtensorMap& tx, const Params& p, cudaStream_t s) {
    using CF = Cfg<BN, BMT, EPI, PAIR>;
    auto kern = gemm_tc_kernel<BN, BMT, A_MN, B_MN, EPI, TF, PAIR>;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    if constexpr (PAIR) {
        const int clusters = std::min(p.num_units, pair_max_clusters());
        if (clusters < 1) return cudaErrorNotSupported;
        ::g2::launch_k_cluster(kern, 2 * clusters, CF::THREADS, CF::SMEM_BYTES, s, 2u, ta, tb, td, td2, tx, p);
    } else {
        int grid = std::min(p.num_units, num_sms());
        ::g2::launch_k(kern, grid, CF::THREADS, CF::SMEM_BYTES, s, ta, tb, td, td2, tx, p);
    }
    return cudaGetLastError();
}

struct Maps {
    CUtensorMap a, b, d, d2, x;
};

template <int BN, int EPI>
static cudaError_t launch_layout(int bmt, bool a_mn, bool b_mn, const Maps& m, const Params& p, cudaStream_t s) {
    if (bmt == TILE_PAIR) {
        if constexpr (BN == 256) {
            if (!a_mn && !b_mn) return launch_t<BN, 128, false, false, EPI, false, true>(m.a, m.b, m.d, m.d2, m.x, p, s);
            if (!a_mn && b_mn) return launch_t<BN, 128, false, true, EPI, false, true>(m.a, m.b, m.d, m.d2, m.x, p, s);
            if (a_mn && b_mn) return launch_t<BN, 128, true, true, EPI, false, true>(m.a, m.b, m.d, m.d2, m.x, p, s);
            return launch_t<BN, 128, true, false, EPI, false, true>(m.a, m.b, m.d, m.d2, m.x, p, s);
        } else {
            return cudaErrorNotSupported;
        }
    }
    if (bmt == 256) {
        if (!a_mn && !b_mn) return launch_t<BN, 256, false, false, EPI>(m.a, m.b, m.d, m.d2, m.x, p, s);
        if (!a_mn && b_mn) return launch_t<BN, 256, false, true, EPI>(m.a, m.b, m.d, m.d2, m.x, p, s);
        if (a_mn && b_mn) return launch_t<BN, 256, true, true, EPI>(m.a, m.b, m.d, m.d2, m.x, p, s);
        return launch_t<BN, 256, true, false, EPI>(m.a, m.b, m.d, m.d2, m.x, p, s);
    }
    if (!a_mn && !b_mn) return launch_t<BN, 128, false, false, EPI>(m.a, m.b, m.d, m.d2, m.x, p, s);
    if (!a_mn && b_mn) return launch_t<BN, 128, false, true, EPI>(m.a, m.b, m.d, m.d2, m.x, p, s);
    if (a_mn && b_mn) return launch_t<BN, 128, true, true, EPI>(m.a, m.b, m.d, m.d2, m.x, p, s);
    return launch_t<BN, 128, true, false, EPI>(m.a, m.b, m.d, m.d2, m.x, p, s);
}

// TF32 products: K-major operands only, fp32 output (plain store or split-K partial).
template <int BN, int EPI>
static cudaError_t launch_tf32(int bmt, const Maps& m, const Params& p, cudaStream_t s) {
    if (bmt == 256) return launch_t<BN, 256, false, false, EPI, true>(m.a, m.b, m.d, m.d2, m.x, p, s);
    return launch_t<BN, 128, false, false, EPI, true>(m.a, m.b, m.d, m.d2, m.x, p, s);
}

}  // namespace tc

using namespace tc;

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

// Timeout flag used when the caller passes none.
__device__ int g_gemm_tc_timeout_flag;
static int* fallback_flag() {
    static int* ptr = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gemm_tc_timeout_flag) == cudaSuccess) ptr = (int*)p;
    });
    return ptr;
}

// Tile-height override (0: chosen per shape) and a description of the last launch, so
// that the variants large shapes pick can be run, and identified, on small ones.
static std::atomic<int> g_force_rows{0};
static std::mutex g_variant_mu;
static char g_variant[128] = "none";

// Tile height: 256-row tiles halve the operand bytes each SM receives per FLOP for B but
// leave no room in tensor memory for a second accumulator, so their epilogue does not
// overlap the next tile; they pay off for long K (many K blocks per tile) when there are
// plenty of tiles.  Otherwise 128-row tiles with double-buffered accumulators.  Products
// with a staged epilogue input always take 128-row tiles, whatever the override.
static int tile_rows(int M, int N, int K, int BN, bool staged_input = false) {
    if (staged_input) return 128;
    const int forced = g_force_rows.load(std::memory_order_relaxed);
    if (forced == 128 || forced == 256) return forced;
    const long long tiles128 = (long long)((M + 127) / 128) * ((N + BN - 1) / BN);
    const bool long_k = K >= 2048 && tiles128 >= 4LL * num_sms();
    const bool very_many_tiles = tiles128 >= 64LL * num_sms();  // e.g. the LM head forward
    return (long_k || very_many_tiles) ? 256 : 128;
}

int gemm_tc_force_tile_rows(int rows) {
    return g_force_rows.exchange(rows == 128 || rows == 256 || rows == TILE_PAIR ? rows : 0);
}

// Tile mode of a bf16 product.  CTA pairs (256-row tiles, 128 rows and half of B per SM:
// 32 KB of operands per SM per 512 clocks of tensor work, against 48 KB for a 128-row tile
// on one SM, with the accumulator still double-buffered) for the forward layout (A and B
// K-major) with 256-column tiles and more than one row tile: measured at B=32, T=1024 they
// beat the best one-SM tiles by 2-5% (QKV 91 -> 87 us, LM head 1.80 -> 1.70 ms, bias +
// GELU 153 -> 150 us, residual 46.1 -> 45.2 us); on the input- and weight-gradient
// layouts they tie or lose (LM-head gradients 1.57 / 1.45 ms on 256-row tiles against
// 1.71 / 1.55 ms).  The forced setting when given; one-SM tiles when pairs cannot launch.
static int tile_mode(int M, int N, int K, int BN, bool staged_input, bool skinny, bool fwd_layout) {
    const int forced = g_force_rows.load(std::memory_order_relaxed);
    const bool pair_ok = BN == 256 && !skinny && M > 128 && pair_max_clusters() > 0;
    if (forced == TILE_PAIR) return pair_ok ? TILE_PAIR : tile_rows(M, N, K, BN, staged_input);
    if (forced) return tile_rows(M, N, K, BN, staged_input);
    if (pair_ok && fwd_layout) return TILE_PAIR;
    return tile_rows(M, N, K, BN, staged_input);
}

void gemm_tc_note_variant(const char* v) {
    std::lock_guard<std::mutex> lk(g_variant_mu);
    snprintf(g_variant, sizeof g_variant, "%s", v);
}

void gemm_tc_last_variant(char* out, size_t n) {
    std::lock_guard<std::mutex> lk(g_variant_mu);
    snprintf(out, n, "%s", g_variant);
}

// Split-K plan for a product with few output tiles and a long K (bke: elements per K
// block, 64 for bf16 operands, 32 for fp32 ones).
static void plan(int M, int N, int K, int BN, int rows, int& splits, int& kb_per, int bke = BK) {
    int tiles = ((M + rows - 1) / rows) * ((N + BN - 1) / BN);
    int num_kb = (K + bke - 1) / bke;
    int sms = num_sms();
    splits = 1;
    if (tiles < sms && num_kb >= 8) {
        splits = std::min(std::max(1, (2 * sms) / tiles), num_kb / 4);
        splits = std::max(splits, 1);
    }
    kb_per = (num_kb + splits - 1) / splits;
    splits = (num_kb + kb_per - 1) / kb_per;
}

// Split-K plan for a product with a single row tile (a few rows: the one-token steps of
// generation), where the time goes into streaming B: enough (column tile, split) units
// to keep every SM loading, while the fp32 partials (splits*M*N*4 bytes) stay within
// half of B's own bytes (N*K*2).
static int skinny_bn(int M, int N) {
    const int tiles256 = (N + 255) / 256;
    return (N <= 128 || (M <= 128 && tiles256 < num_sms())) ? 128 : 256;
}
static void plan_skinny(int M, int N, int K, int BN, int& splits, int& kb_per) {
    const int tiles = (N + BN - 1) / BN;
    const int num_kb = (K + BK - 1) / BK;
    const int want = (2 * num_sms() + tiles - 1) / tiles;
    const int cap = std::max(1, K / (4 * std::max(M, 1)));
    splits = std::max(1, std::min(std::min(want, num_kb), cap));
    kb_per = (num_kb + splits - 1) / splits;
    splits = (num_kb + kb_per - 1) / kb_per;
}

size_t gemm_tc_skinny_workspace_bytes(int M, int N, int K) {
    if (M > 128) return 0;
    const int BN = skinny_bn(M, N);
    int splits, kb_per;
    plan_skinny(M, N, K, BN, splits, kb_per);
    return splits > 1 ? (size_t)splits * M * N * sizeof(float) : 0;
}

size_t gemm_tc_workspace_bytes(int M, int N, int K) {
    // the most splits any tile height or operand type can plan
    const int BN = N > 128 ? 256 : 128;
    size_t b = 0;
    for (int rows : {128, 256})
        for (int bke : {BK, 32}) {
            int splits, kb_per;
            plan(M, N, K, BN, rows, splits, kb_per, bke);
            if (splits > 1) b = std::max(b, (size_t)splits * M * N * sizeof(float));
        }
    return b;
}

// TF32 products (fp32 operands): both operands K-major, rows 16-byte aligned, fp32
// output with a plain or bias epilogue (the dispatcher transposes operands and applies
// the other epilogues around this kernel).
bool gemm_tc_tf32_supported(const GemmArgs& a) {
    if (a.in_type != ACT_F32 || !encode_fn()) return false;
    if (a.M < 1 || a.N < 1 || a.K < 32) return false;
    if (a.sAk != 1 || a.sBk != 1) return false;
    if ((a.sAm % 4) || (a.sBn % 4) || !aligned16(a.A) || !aligned16(a.B)) return false;
    if (!aligned16(a.D) || (a.ldd % 4)) return false;
    if (a.epi != EPI_STORE || a.R || a.D2 || a.P) return false;
    if (a.bias && !aligned16(a.bias)) return false;
    return true;
}

bool gemm_tc_supported(const GemmArgs& a) {
    if (a.in_type == ACT_F32) return a.tf32 && gemm_tc_tf32_supported(a);
    if (a.in_type != ACT_BF16 || !encode_fn()) return false;
    if (a.M < 1 || a.N < 1 || a.K < 16) return false;
    bool a_k = a.sAk == 1, b_k = a.sBk == 1;
    long long lda = a_k ? a.sAm : a.sAk, ldb = b_k ? a.sBn : a.sBk;
    if (!a_k && a.sAm != 1) return false;
    if (!b_k && a.sBn != 1) return false;
    if ((lda % 8) || (ldb % 8) || !aligned16(a.A) || !aligned16(a.B)) return false;
    // inner extents of the tensor maps must reach one 128-byte swizzle row
    if (a_k ? a.K < 64 : a.M < 64) return false;
    if (b_k ? a.K < 64 : a.N < 64) return false;
    if (!aligned16(a.D) || (a.ldd % 8)) return false;
    if (a.epi == EPI_GELU && (!a.D2 || (a.ldd2 % 8) || !aligned16(a.D2))) return false;
    if (a.epi == EPI_GELU_BWD && (!a.P || (a.ldp % 8) || !aligned16(a.P))) return false;
    if (a.R && ((a.ldr % 8) || !aligned16(a.R))) return false;
    if (a.R && a.d_f32) return false;  // the residual epilogue writes bf16 only
    if (a.bias && !aligned16(a.bias)) return false;
    return true;
}

bool gemm_tc_fuses_colsum(const GemmArgs& a) {
    return a.colsum_part && a.epi == EPI_GELU_BWD && a.in_type == ACT_BF16 && !a.d_f32 && (a.N % 2) == 0 &&
           ((uintptr_t)a.colsum_part & 7) == 0 && gemm_tc_supported(a);
}

// D (fp32) = A . B^T (+ bias) with fp32 operands read as TF32.
static cudaError_t gemm_tc_tf32(const GemmArgs& a, float* ws, size_t ws_bytes, int* flags, cudaStream_t s) {
    const int BN = a.N > 128 ? 256 : 128;
    const int bmt = tile_rows(a.M, a.N, a.K, BN);
    constexpr int BKE = OperandT<true>::BKE;
    Maps mp;
    {
        const uint64_t da[2] = {(uint64_t)a.K, (uint64_t)a.M}, sa[1] = {(uint64_t)a.sAm * 4};
        const uint32_t ba[2] = {(uint32_t)BKE, (uint32_t)bmt};
        const uint64_t db[2] = {(uint64_t)a.K, (uint64_t)a.N}, sb[1] = {(uint64_t)a.sBn * 4};
        const uint32_t bb[2] = {(uint32_t)BKE, (uint32_t)BN};
        if (!make_map_nd(&mp.a, a.A, true, 2, da, sa, ba) || !make_map_nd(&mp.b, a.B, true, 2, db, sb, bb))
            return cudaErrorInvalidValue;
    }
    Params p{};
    p.M = a.M; p.N = a.N; p.K = a.K;
    p.tiles_m = (a.M + bmt - 1) / bmt;
    p.tiles_n = (a.N + BN - 1) / BN;
    p.num_kb = (a.K + BKE - 1) / BKE;
    int splits = 1, kb_per = p.num_kb;
    if (!a.bias) plan(a.M, a.N, a.K, BN, bmt, splits, kb_per, BKE);
    if (splits > 1 && (!ws || ws_bytes < (size_t)splits * a.M * a.N * sizeof(float) || a.N % 4)) {
        splits = 1;
        kb_per = p.num_kb;
    }
    p.splits = splits;
    p.kb_per_split = kb_per;
    p.num_units = p.tiles_m * p.tiles_n * splits;
    p.D = a.D; p.ldd = a.ldd; p.d_f32 = 1;
    p.bias = a.bias;
    p.ws = ws;
    p.flags = flags ? flags : fallback_flag();
    bool ok;
    const uint32_t box_f32[2] = {32, 32};
    if (splits > 1) {
        const uint64_t dims[3] = {(uint64_t)a.N, (uint64_t)a.M, (uint64_t)splits};
        const uint64_t st[2] = {(uint64_t)a.N * 4, (uint64_t)a.M * a.N * 4};
        const uint32_t box3[3] = {32, 32, 1};
        ok = make_map_nd(&mp.d, ws, true, 3, dims, st, box3);
    } else {
        const uint64_t dims[2] = {(uint64_t)a.N, (uint64_t)a.M};
        const uint64_t st[1] = {(uint64_t)a.ldd * 4};
        ok = make_map_nd(&mp.d, a.D, true, 2, dims, st, box_f32);
    }
    if (!ok) return cudaErrorInvalidValue;
    mp.d2 = mp.d;
    mp.x = mp.d;
    {
        std::lock_guard<std::mutex> lk(g_variant_mu);
        snprintf(g_variant, sizeof g_variant, "rows=%d cols=%d splits=%d a=k b=k epi=store f32 tf32", bmt, BN,
                 splits);
    }
    if (splits > 1) {
        cudaError_t e = BN == 256 ? launch_tf32<256, E_PARTIAL>(bmt, mp, p, s) : launch_tf32<128, E_PARTIAL>(bmt, mp, p, s);
        if (e != cudaSuccess) return e;
        launch_splitk_reduce((float*)a.D, a.ldd, ws, a.M, a.N, splits, s);
        return cudaGetLastError();
    }
    return BN == 256 ? launch_tf32<256, E_STORE_F32>(bmt, mp, p, s) : launch_tf32<128, E_STORE_F32>(bmt, mp, p, s);
}

cudaError_t gemm_tc(const GemmArgs& a, float* ws, size_t ws_bytes, int* flags, cudaStream_t s) {
    if (a.in_type == ACT_F32) return gemm_tc_tf32(a, ws, ws_bytes, flags, s);
    const bool a_mn = a.sAk != 1, b_mn = a.sBk != 1;
    const bool skinny = a.skinny_split && a.M <= 128 && a.epi != EPI_GELU_BWD;
    const int BN = skinny ? skinny_bn(a.M, a.N) : (a.N > 128 ? 256 : 128);
    const bool staged_in = a.epi == EPI_GELU_BWD || (a.epi == EPI_STORE && a.R && !a.d_f32);
    const int bmt = tile_mode(a.M, a.N, a.K, BN, staged_in, skinny, !a_mn && !b_mn);
    const int unit_rows = bmt == 128 ? 128 : 256;  // rows of a work unit (a pair: 128 per SM)
    const int a_box = bmt == 256 ? 256 : 128, b_box = bmt == TILE_PAIR ? BN / 2 : BN;
    Maps mp;
    bool ok;
    if (!a_mn)
        ok = make_map(&mp.a, a.A, a.K, a.M, a.sAm, BK, a_box);
    else
        ok = make_map(&mp.a, a.A, a.M, a.K, a.sAk, 64, BK);
    if (!ok) return cudaErrorInvalidValue;
    if (!b_mn)
        ok = make_map(&mp.b, a.B, a.K, a.N, a.sBn, BK, b_box);
    else
        ok = make_map(&mp.b, a.B, a.N, a.K, a.sBk, 64, BK);
    if (!ok) return cudaErrorInvalidValue;

    Params p{};
    p.M = a.M; p.N = a.N; p.K = a.K;
    p.tiles_m = (a.M + unit_rows - 1) / unit_rows;
    p.tiles_n = (a.N + BN - 1) / BN;
    p.num_kb = (a.K + BK - 1) / BK;
    int splits = 1, kb_per = p.num_kb;
    if (skinny)
        plan_skinny(a.M, a.N, a.K, BN, splits, kb_per);
    else if (a.epi == EPI_STORE && a.d_f32 && !a.bias && !a.R)
        plan(a.M, a.N, a.K, BN, unit_rows, splits, kb_per);
    if (splits > 1 && (!ws || ws_bytes < (size_t)splits * a.M * a.N * sizeof(float))) {
        splits = 1;
        kb_per = p.num_kb;
    }
    p.splits = splits;
    p.kb_per_split = kb_per;
    p.num_units = p.tiles_m * p.tiles_n * splits;
    p.D = a.D; p.ldd = a.ldd; p.d_f32 = a.d_f32;
    p.bias = a.bias;
    p.R = (const bf16*)a.R; p.ldr = a.ldr;
    p.D2 = (bf16*)a.D2; p.ldd2 = a.ldd2;
    p.P = (const bf16*)a.P; p.ldp = a.ldp;
    p.ws = ws;
    p.cs_part = gemm_tc_fuses_colsum(a) ? a.colsum_part : nullptr;
    p.flags = flags ? flags : fallback_flag();

    // output maps for the TMA stores: 32-row boxes of 128 bytes (64 bf16 or 32 fp32)
    const uint32_t box_bf16[2] = {64, 32}, box_f32[2] = {32, 32};
    if (splits > 1) {
        const uint64_t dims[3] = {(uint64_t)a.N, (uint64_t)a.M, (uint64_t)splits};
        const uint64_t st[2] = {(uint64_t)a.N * 4, (uint64_t)a.M * a.N * 4};
        const uint32_t box3[3] = {32, 32, 1};
        ok = (a.N % 4 == 0) && make_map_nd(&mp.d, ws, true, 3, dims, st, box3);
    } else {
        const uint64_t dims[2] = {(uint64_t)a.N, (uint64_t)a.M};
        const uint64_t st[1] = {(uint64_t)a.ldd * (a.d_f32 ? 4 : 2)};
        ok = make_map_nd(&mp.d, a.D, a.d_f32 != 0, 2, dims, st, a.d_f32 ? box_f32 : box_bf16);
    }
    if (!ok) return cudaErrorInvalidValue;
    mp.d2 = mp.d;
    mp.x = mp.d;
    const bool has_in = staged_in;
    if (has_in) {
        const void* xb = a.epi == EPI_GELU_BWD ? a.P : a.R;
        const long long ldx = a.epi == EPI_GELU_BWD ? a.ldp : a.ldr;
        const uint64_t dims[2] = {(uint64_t)a.N, (uint64_t)a.M};
        const uint64_t st[1] = {(uint64_t)ldx * 2};
        if (!make_map_nd(&mp.x, xb, false, 2, dims, st, box_bf16)) return cudaErrorInvalidValue;
    }
    if (a.epi == EPI_GELU) {
        const uint64_t dims[2] = {(uint64_t)a.N, (uint64_t)a.M};
        const uint64_t st[1] = {(uint64_t)a.ldd2 * 2};
        if (!make_map_nd(&mp.d2, a.D2, false, 2, dims, st, box_bf16)) return cudaErrorInvalidValue;
    }

    {
        static const char* epi_names[] = {"store", "gelu", "gelu_bwd"};
        std::lock_guard<std::mutex> lk(g_variant_mu);
        char pairs[32] = "";
        if (bmt == TILE_PAIR) snprintf(pairs, sizeof pairs, " clusters=%d", pair_max_clusters());
        snprintf(g_variant, sizeof g_variant, "rows=%s cols=%d splits=%d a=%s b=%s epi=%s%s%s%s%s",
                 bmt == TILE_PAIR ? "pair256" : (bmt == 256 ? "256" : "128"), BN, splits,
                 a_mn ? "mn" : "k", b_mn ? "mn" : "k", epi_names[a.epi], a.d_f32 ? " f32" : "",
                 staged_in && a.epi == EPI_STORE ? " residual" : "", p.cs_part ? " colsum" : "", pairs);
    }
    cudaError_t e;
    if (splits > 1) {
        e = BN == 256 ? launch_layout<256, E_PARTIAL>(bmt, a_mn, b_mn, mp, p, s)
                      : launch_layout<128, E_PARTIAL>(bmt, a_mn, b_mn, mp, p, s);
        if (e != cudaSuccess) return e;
        size_t n = (size_t)a.M * a.N;
        unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, (size_t)num_sms() * 8);
        if (skinny)
            ::g2::launch_k(splitk_epilogue_k, blocks, 256, 0, s, 
                a.D, a.ldd, a.d_f32, ws, a.M, a.N, splits, a.bias, (const bf16*)a.R, a.ldr,
                a.epi == EPI_GELU ? (bf16*)a.D2 : nullptr, a.ldd2);
        else
            launch_splitk_reduce((float*)a.D, a.ldd, ws, a.M, a.N, splits, s);
        return cudaGetLastError();
    }
    switch (a.epi) {
        case EPI_GELU:
            return BN == 256 ? launch_layout<256, E_GELU>(bmt, a_mn, b_mn, mp, p, s)
                             : launch_layout<128, E_GELU>(bmt, a_mn, b_mn, mp, p, s);
        case EPI_GELU_BWD:
            return BN == 256 ? launch_layout<256, E_GELU_BWD>(bmt, a_mn, b_mn, mp, p, s)
                             : launch_layout<128, E_GELU_BWD>(bmt, a_mn, b_mn, mp, p, s);
        default:
            if (a.d_f32)
                return BN == 256 ? launch_layout<256, E_STORE_F32>(bmt, a_mn, b_mn, mp, p, s)
                                 : launch_layout<128, E_STORE_F32>(bmt, a_mn, b_mn, mp, p, s);
            if (has_in)
                return BN == 256 ? launch_layout<256, E_STORE_RES>(bmt, a_mn, b_mn, mp, p, s)
                                 : launch_layout<128, E_STORE_RES>(bmt, a_mn, b_mn, mp, p, s);
            return BN == 256 ? launch_layout<256, E_STORE>(bmt, a_mn, b_mn, mp, p, s)
                             : launch_layout<128, E_STORE>(bmt, a_mn, b_mn, mp, p, s);
    }
}

}  // namespace g2
