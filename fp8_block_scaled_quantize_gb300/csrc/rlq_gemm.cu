// Block-scaled FP8 GEMM on 5th-generation tensor cores (sm_103a).
//
// Jet-RL notes, section "细粒度 GEMM 量化方案": FProp, DGrad and WGrad all run
// as FP8 GEMMs on 1x128 / 128x128 (and, for WGrad, 128x1) scaled operands.
// One kernel serves the three passes:
//
//   out[r, c] = bf16( sum_b sa(b, r) * sb(b, c) * P_b[r, c] ),
//   P_b[r, c] = sum_{j in block b} A[r, j] * B[c, j]          (E4M3 x E4M3, exact in fp32)
//
// where b runs over 128-wide blocks of the contraction.  The hardware block
// scale formats (UE8M0 / E4M3 per 16 or 32 elements) do not express these fp32
// per-128 scales, so the scaling ("promotion") is done in software:
//
//   * a TMA warp streams 128x128 A tiles and 256x128 B tiles (128-byte swizzle)
//     into a 4-stage shared-memory ring guarded by mbarriers;
//   * two MMA warps issue, per contraction block (even blocks one warp, odd
//     blocks the other), four tcgen05.mma (kind::f8f6f4, M=128, N=256, K=32)
//     into one of two TMEM partial buffers (2 x 256 fp32 columns = the whole
//     512-column TMEM), then commit;
//   * eight epilogue warps read the finished partial with tcgen05.ld, multiply
//     by sa * sb and accumulate into fp32 registers (packed f32x2 FMA), release
//     the TMEM buffer, and after the tile's last block round to bf16 and store;
//   * a scale warp streams each block's scales (128 row scales, and the block
//     or per-column scales of the tile's columns) into an 8-slot shared-memory
//     ring with cp.async, up to 8 blocks ahead of the epilogue, so that their
//     global-memory latency never reaches the promotion.  These copies use the
//     generic proxy (cp.async + cp.async.mbarrier.arrive), not TMA: the
//     epilogue reads the ring with ordinary loads, and generic reads of a
//     buffer that the async proxy rewrites are not ordered by mbarriers alone
//     (a TMA-staged variant measured non-deterministic).
//
// Tiles are 128 x 256 per CTA.  Outputs of at least 256 rows run on CTA pairs
// (clusters of two, tcgen05.mma.cta_group::2, M = 256): each CTA stages its 128
// rows of A and half of B, the even CTA issues the pair's MMAs and commits to
// both CTAs' barriers, and the epilogue stages the bf16 tile in shared memory
// for TMA stores.  A single CTA (fewer rows, or a split contraction) stores its
// rows directly.  The kernel is persistent (one CTA per SM, one pair per two)
// and walks (tile, contraction split) units with the smaller operand resident in
// L2.  Every mbarrier wait is bounded: on timeout the waiting thread records an
// error word that rlq_check() reports, raises a CTA-wide abort flag, and the CTA
// drains its in-flight copies and MMAs, frees TMEM and exits.  Nothing traps.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "rlq_internal.h"
#include "rlq_tc.cuh"

namespace rlq {

namespace {

constexpr int BM = 128;                    // tile rows (TMEM lanes)
constexpr int BN = 256;                    // tile columns (MMA N)
constexpr int BK = 128;                    // contraction block = scale granularity = 128 bytes of E4M3
constexpr int UMMA_K = 32;                 // K of one kind::f8f6f4 MMA
constexpr int A_BYTES = BM * BK;           // 16 KB
// Warpgroup 0: warp 0 TMA, warps 1 and 3 MMA (even / odd contraction blocks; warp 1
// owns TMEM), warp 2 scales.
// Warpgroups 1-2: eight epilogue warps.  Registers are rebalanced with
// setmaxnreg: 128 x 40 + 256 x 232 = 384 x 168, the launch allocation.
constexpr int NUM_THREADS = 384;
constexpr int FIRST_EPI_WARP = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int REGS_PRODUCER = 40;
constexpr int REGS_EPILOGUE = 232;
constexpr int TMEM_COLS = 2 * BN;          // two partial buffers
constexpr int SCALE_SLOTS = 8;             // scale ring depth (contraction blocks)
constexpr int SLOT_FLOATS = BM + BN;       // 128 row scales + up to 256 column scales
constexpr int RING_BYTES = SCALE_SLOTS * SLOT_FLOATS * 4;

// Per-mode shared-memory plan.  Single CTA: the CTA holds the whole 256-row B tile
// (48 KB stages, 4 of them) and stores its output rows straight from registers
// (outputs under 256 rows and split-K partials, where the contraction per tile is
// long and the stores are a small share).  CTA pair (cta_group::2): an output tile
// is 256 x 256, each CTA holds its 128 rows of A and half of the B tile (32 KB
// stages); the pair's MMA reads both halves of B, so each byte of B is staged in
// one SM only.  A pair's bf16 tile leaves through TMA stores from a per-warp
// staging buffer of 32 rows x RLQ_STG_COLS columns (coalesced and asynchronous:
// the epilogue moves on while the copy drains); the rest of the shared memory
// goes to pipeline stages, whose depth keeps enough operand bytes in flight to
// cover the L2 / HBM latency.
#ifndef RLQ_PAIR_STAGES
#define RLQ_PAIR_STAGES 4
#endif
#ifndef RLQ_STG_COLS
#define RLQ_STG_COLS 64
#endif
constexpr int STG_COLS = RLQ_STG_COLS;            // bf16 columns per staged store round (64 or 128)
constexpr int STG_WARP_BYTES = 32 * STG_COLS * 2;  // one warp's staging buffer
static_assert(STG_COLS == 64 || STG_COLS == 128, "staged rounds of 64 or 128 columns");

template <bool kPair>
struct Cfg {
    static constexpr int STAGES = kPair ? RLQ_PAIR_STAGES : 4;
    static constexpr int STAGING = kPair ? NUM_EPI_WARPS * STG_WARP_BYTES : 0;
    static constexpr int B_ROWS = kPair ? BN / 2 : BN;  // B rows (output columns) staged per CTA
    static constexpr int B_BYTES = B_ROWS * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TILE_M = kPair ? 2 * BM : BM;  // output rows per tile
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 1 + 2 * SCALE_SLOTS;
    static constexpr int SMEM_BYTES =
        1024 /* alignment slack */ + STAGES * STAGE_BYTES + STAGING + RING_BYTES + NUM_BARS * 8 + 16;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    // Instruction descriptor of tcgen05.mma kind::f8f6f4: D fp32 (bits 4-5 = 1), A and
    // B E4M3 (format 0 in bits 7-9 / 10-12), A K-major (bit 15 = 0), B K-major (bit
    // 16 = 0) or MN-major (bit 16 = 1), N >> 3 in bits 17-22, M >> 4 in bits 24-28
    // (M = 256 for a CTA pair).
    static constexpr uint32_t IDESC_BK = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(TILE_M >> 4) << 24);
    static constexpr uint32_t IDESC_BMN = IDESC_BK | (1u << 16);
};


// First row, within a tile, of the rows this CTA owns.
template <bool kPair>
__device__ __forceinline__ int row_offset()
{
    if constexpr (kPair)
        return (int)cta_rank() * BM;
    return 0;
}

// Explicit shared-memory loads: the aligned dynamic-smem base is computed through
// an integer, so plain C++ loads through it compile to generic loads; those cost
// WGrad's promotion 14% (its 256 column scales per block).
__device__ __forceinline__ float lds_f32(uint32_t a)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ float4 lds_v4(uint32_t a)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a) : "memory");
    return v;
}

// The warp has read its part of a TMEM buffer (every tcgen05.ld waited for):
// signal the MMA warp that may overwrite it, on the issuing CTA's barrier.
template <bool kPair>
__device__ __forceinline__ void release_tmem(uint32_t tempty, int lane)
{
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
        if constexpr (kPair)
            mbar_arrive_cluster(cluster_addr(tempty, 0));
        else
            mbar_arrive(tempty);
    }
}

__device__ __forceinline__ float2 f2_of(uint32_t lo, uint32_t hi)
{
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}

// acc[0..15] += chunk * scale, two columns per packed fp32 FMA.
__device__ __forceinline__ void promote_chunk(float2 *acc, const uint32_t (&r)[32], float2 scl)
{
#pragma unroll
    for (int j = 0; j < 16; ++j)
        acc[j] = __ffma2_rn(f2_of(r[2 * j], r[2 * j + 1]), scl, acc[j]);
}

// acc[0..15] += fl(chunk * sa) * sb[column]; sb is 32 consecutive column scales in
// shared memory (shared-window address), read by every lane (broadcast).  The
// product with the row scale does not wait for the column scales' load, so only
// the FMA does (measured 4% faster on WGrad than scaling sa * sb first).
__device__ __forceinline__ void promote_chunk_cols(float2 *acc, const uint32_t (&r)[32], float2 sa2,
                                                   uint32_t sbs)
{
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float2 p01 = __fmul2_rn(f2_of(r[4 * j], r[4 * j + 1]), sa2);
        const float2 p23 = __fmul2_rn(f2_of(r[4 * j + 2], r[4 * j + 3]), sa2);
        const float4 sb4 = lds_v4(sbs + 16u * j);
        acc[2 * j] = __ffma2_rn(p01, make_float2(sb4.x, sb4.y), acc[2 * j]);
        acc[2 * j + 1] = __ffma2_rn(p23, make_float2(sb4.z, sb4.w), acc[2 * j + 1]);
    }
}

__device__ __forceinline__ uint32_t bf16x2_rn(float2 v)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(v.y), "f"(v.x));
    return d;
}

struct Params {
    const float *sa;
    int64_t ld_sa;
    const float *sb;
    int64_t sb_bstride;
    int64_t sb_cstride;
    int out_mode;     // OUT_BF16, OUT_F32_PARTIAL (split-K) or OUT_F32_ACC
    uint16_t *out;    // OUT_BF16
    int64_t ldo;
    float *acc_out;   // OUT_F32_ACC: acc_out[r * ld_acc + c] += the product
    int64_t ld_acc;
    int R, C;
    int kblocks;
    int m_tiles, n_tiles, num_tiles;
    int m_fastest;
    // split-K: unit u covers tile u / splits and contraction blocks
    // [(u % splits) * kbps, min(kblocks, ... + kbps)); with splits > 1 the
    // epilogue writes fp32 partials (OUT_F32_PARTIAL) to the workspace ws [splits][R][C]
    int splits, kbps, num_units;
    float *ws;
    uint64_t timeout_ns;
    // diagnostic (single CTA only): the producer withholds the loads of the CTA's
    // first stage, so the MMA warp's bounded wait on it runs out
    int withhold_first_load;
};

struct Unit {
    int mt, nt, split, kb0, kb1;
};


__device__ __forceinline__ void tile_coords(const Params &p, int tile, int &mt, int &nt)
{
    if (p.m_fastest) {
        mt = tile % p.m_tiles;
        nt = tile / p.m_tiles;
    } else {
        nt = tile % p.n_tiles;
        mt = tile / p.n_tiles;
    }
}

__device__ __forceinline__ Unit unit_of(const Params &p, int u)
{
    Unit w;
    const int tile = u / p.splits;
    w.split = u - tile * p.splits;
    tile_coords(p, tile, w.mt, w.nt);
    w.kb0 = w.split * p.kbps;
    w.kb1 = min(p.kblocks, w.kb0 + p.kbps);
    return w;
}

// Promotion modes.
//   MODE_BLOCK:  sb is one scale per (contraction block, 128 output columns):
//                FProp and DGrad, acc += P_b * (sa * sb).
//   MODE_COLS:   sb is one scale per (contraction block, output column): WGrad,
//                acc += P_b * (sa * sb[c]).
//   MODE_ONCE:   sa and sb are constant along the contraction (per-token x
//                per-channel FProp): the MMAs accumulate the whole contraction
//                range in TMEM and the epilogue scales once, out = P * (sa * sb[c]).
enum : int { MODE_BLOCK = 0, MODE_COLS = 1, MODE_ONCE = 2 };

// Epilogue outputs.
enum : int { OUT_BF16 = 0, OUT_F32_PARTIAL = 1, OUT_F32_ACC = 2 };

template <int kMode, bool kBMajorMN, bool kPair>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_block_scaled(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmOut, const Params p)
{
    pdl_begin();
    using Cf = Cfg<kPair>;
    constexpr int STAGES = Cf::STAGES;
    constexpr int STAGE_BYTES = Cf::STAGE_BYTES;
    constexpr int NUM_BARS = Cf::NUM_BARS;
    constexpr bool kOnce = kMode == MODE_ONCE;
    // A CTA pair (cluster of 2) shares one 256-row tile: CTA `rank` owns rows
    // rank * 128 .. rank * 128 + 127 of it; the even CTA issues the pair's MMAs.
    // (The rank is re-read where it is used rather than kept in a register.)
    const int unit0 = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int unit_step = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *staging = smem + STAGES * STAGE_BYTES;
    float *ring = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES + Cf::STAGING);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES + Cf::STAGING + RING_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NUM_BARS);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t smem0 = smem_u32(smem);
    auto a_stage = [&](int s) { return smem0 + (uint32_t)(s * STAGE_BYTES); };
    auto b_stage = [&](int s) { return smem0 + (uint32_t)(s * STAGE_BYTES + A_BYTES); };
    auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
    auto empty_bar = [&](int s) { return smem_u32(&bars[STAGES + s]); };
    auto tfull_bar = [&](int b) { return smem_u32(&bars[2 * STAGES + b]); };
    auto tempty_bar = [&](int b) { return smem_u32(&bars[2 * STAGES + 2 + b]); };
    const uint32_t teardown_bar = smem_u32(&bars[2 * STAGES + 4]);
    auto sfull_bar = [&](int k) { return smem_u32(&bars[2 * STAGES + 5 + k]); };
    auto sempty_bar = [&](int k) { return smem_u32(&bars[2 * STAGES + 5 + SCALE_SLOTS + k]); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);  // the stage is free once its MMAs completed
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            // a pair's buffer is free once the epilogue warps of both CTAs released it
            mbar_init(tempty_bar(b), kPair ? 2 * NUM_EPI_WARPS : NUM_EPI_WARPS);
        }
        mbar_init(teardown_bar, 2);  // one commit per MMA-issuing warp
        for (int k = 0; k < SCALE_SLOTS; ++k) {
            mbar_init(sfull_bar(k), 32);              // one cp.async arrival per scale-warp lane
            mbar_init(sempty_bar(k), NUM_EPI_WARPS);  // one arrival per epilogue warp
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        if constexpr (kPair) {
            // collective: one warp of each CTA of the pair; both receive the same address
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (kPair && p.out_mode != OUT_F32_PARTIAL)
            prefetch_tmap(&tmOut);
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (kPair)
        cluster_sync();  // both CTAs' barriers are initialised before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp < FIRST_EPI_WARP)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_PRODUCER));
    if (warp == 0) {
        // ------------------------------------------------ TMA producer ---
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            // the tile order walks the smaller operand fastest and re-reads it: keep it in L2
            const uint64_t pol_a = l2_policy(p.m_fastest != 0), pol_b = l2_policy(p.m_fastest == 0);
            for (int u = unit0; ok && u < p.num_units; u += unit_step) {
                const Unit w = unit_of(p, u);
                const int mt = w.mt, nt = w.nt;
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                    if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, p.timeout_ns, SITE_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    if constexpr (kPair) {
                        // both CTAs' copies complete on the even CTA's barrier, which
                        // expects the bytes of the two stages
                        const uint32_t fb = cluster_addr(full_bar(s), 0);
                        if (cta_rank() == 0)
                            mbar_arrive_expect_tx(full_bar(s), 2 * STAGE_BYTES);
                        tma_load_2d_pair_hint(a_stage(s), &tmA, fb, kb * BK, mt * Cf::TILE_M + row_offset<kPair>(),
                                              pol_a);
                        if (kBMajorMN)  // this CTA's 128 output columns: one 128 x 128 box
                            tma_load_2d_pair_hint(b_stage(s), &tmB, fb, nt * BN + row_offset<kPair>(), kb * BK, pol_b);
                        else
                            tma_load_2d_pair_hint(b_stage(s), &tmB, fb, kb * BK, nt * BN + row_offset<kPair>(), pol_b);
                    } else {
                        if (p.withhold_first_load && it == 0)
                            continue;  // nothing arrives on this stage's barrier
                        mbar_arrive_expect_tx(full_bar(s), STAGE_BYTES);
                        tma_load_2d(a_stage(s), &tmA, full_bar(s), kb * BK, mt * BM);
                        if (kBMajorMN) {
                            // B stored [contraction][output]: two 128-column boxes of 128 rows
                            tma_load_2d(b_stage(s), &tmB, full_bar(s), nt * BN, kb * BK);
                            tma_load_2d(b_stage(s) + Cf::B_BYTES / 2, &tmB, full_bar(s), nt * BN + 128, kb * BK);
                        } else {
                            tma_load_2d(b_stage(s), &tmB, full_bar(s), kb * BK, nt * BN);
                        }
                    }
                }
            }
            if constexpr (kPair) {
                if (!ok) {
                    // the copies complete on the even CTA's barriers: give them time to land
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < 200000ull)
                        __nanosleep(1000);
                }
            }
            if constexpr (!kPair) {
                // A CTA that aborted may still have copies in flight into stages no
                // MMA consumed: they complete on their own, and are waited for
                // (bounded) before the CTA's shared memory goes away.  Once both MMA
                // warps have made their final commit, every stage they did not
                // consume is known: if they finished normally they consumed all.
                volatile uint32_t never = 0;
                mbar_wait(teardown_bar, 0, &never, p.timeout_ns, SITE_TEARDOWN);
                if (!ok || *abort_flag || p.withhold_first_load) {
                    int first = it > STAGES ? it - STAGES : 0;
                    if (p.withhold_first_load && first == 0)
                        first = 1;  // the withheld stage has nothing in flight
                    for (int j = first; j < it; ++j)
                        mbar_wait(full_bar(j % STAGES), (uint32_t)(j / STAGES) & 1u, &never, 20000000ull,
                                  SITE_DRAIN);
                }
            }
        }
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------- MMA issuers ---
        // Per-block promotion: warp 1 issues the even contraction blocks (TMEM
        // buffer 0), warp 3 the odd ones (buffer 1), so that one thread's issue
        // latency overlaps the other's MMAs.  Scale-once: warp 1 issues every block
        // of a unit into the unit's buffer (units alternate between the buffers),
        // accumulating across the contraction.  (A pair's MMAs are issued by the
        // even CTA only.)
        const int parity = warp == 1 ? 0 : 1;
        if (lane == 0 && (!kPair || cta_rank() == 0) && (!kOnce || warp == 1)) {
            int it = 0, uc = 0;
            bool ok = true;
            for (int u = unit0; ok && u < p.num_units; u += unit_step, ++uc) {
                const Unit w = unit_of(p, u);
                if (kOnce) {
                    const uint32_t bph = (uint32_t)(uc >> 1) & 1u;
                    if (!mbar_wait(tempty_bar(uc & 1), bph ^ 1u, abort_flag, p.timeout_ns, SITE_MMA_TMEM_EMPTY)) {
                        ok = false;
                        break;
                    }
                }
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                    if (!kOnce && (it & 1) != parity)
                        continue;
                    const int s = it % STAGES;
                    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                    const int buf = kOnce ? (uc & 1) : (it & 1);
                    if (!kOnce) {
                        const uint32_t bph = (uint32_t)(it >> 1) & 1u;
                        if (!mbar_wait(tempty_bar(buf), bph ^ 1u, abort_flag, p.timeout_ns, SITE_MMA_TMEM_EMPTY)) {
                            ok = false;
                            break;
                        }
                    }
                    if (!mbar_wait(full_bar(s), ph, abort_flag, p.timeout_ns, SITE_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + (uint32_t)(buf * BN);
                    const uint64_t ad = sw128_desc(a_stage(s));
                    const uint64_t bd = kBMajorMN ? sw128_desc_mn(b_stage(s)) : sw128_desc(b_stage(s));
                    const bool first = !kOnce || kb == w.kb0;
#pragma unroll
                    for (int j = 0; j < BK / UMMA_K; ++j) {
                        // K-major: +32 bytes along K (+2 in the address field); MN-major:
                        // +32 contraction rows of 128 bytes (+256)
                        const uint64_t bj = kBMajorMN ? bd + (uint64_t)(256 * j) : bd + 2 * j;
                        tc_mma_f8<kPair>(d, ad + 2 * j, bj, kBMajorMN ? Cf::IDESC_BMN : Cf::IDESC_BK,
                                         (first && j == 0) ? 0u : 1u);
                    }
                    // (pair: arrives on the barrier at this offset in both CTAs)
                    tc_commit_t<kPair>(empty_bar(s));
                    if (!kOnce || kb + 1 == w.kb1)
                        tc_commit_t<kPair>(tfull_bar(buf));
                }
            }
        }
        if (lane == 0 && (!kPair || cta_rank() == 0)) {
            // every MMA this thread issued has completed once this commit arrives
            tc_commit_t<kPair>(teardown_bar);
            volatile uint32_t never = 0;
            mbar_wait(teardown_bar, 0, &never, 20000000ull, SITE_TEARDOWN);
        }
    } else if (warp == 2) {
        // ------------------------------------------------ scale loader ---
        // One ring slot per contraction block (scale-once: per unit, read at the
        // unit's first block, the scales being the same for every block).
        int it = 0;
        bool ok = true;
        for (int u = unit0; ok && u < p.num_units; u += unit_step) {
            const Unit w = unit_of(p, u);
            const int mt = w.mt, nt = w.nt;
            for (int kb = w.kb0; kb < (kOnce ? w.kb0 + 1 : w.kb1); ++kb, ++it) {
                const int k = it % SCALE_SLOTS;
                const uint32_t ph = (uint32_t)(it / SCALE_SLOTS) & 1u;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(sempty_bar(k), ph ^ 1u, abort_flag, p.timeout_ns,
                                                       SITE_SCALE_EMPTY))) {
                    ok = false;
                    break;
                }
                const uint32_t slot = smem_u32(ring + k * SLOT_FLOATS);
                const float *sa_row = p.sa + (int64_t)kb * p.ld_sa;
#pragma unroll
                for (int j = 0; j < BM / 32; ++j) {
                    const int r = mt * Cf::TILE_M + row_offset<kPair>() + lane + 32 * j;
                    cp_async4(slot + 4u * (lane + 32 * j), r < p.R ? sa_row + r : sa_row, r < p.R ? 4u : 0u);
                }
                if (kMode != MODE_BLOCK) {
                    const float *sb_row = p.sb + (int64_t)kb * p.sb_bstride;
                    // 256 column scales as 64 aligned 16-byte pieces (rows of sb are 16-byte
                    // aligned, C % 128 == 0: a piece is wholly inside or outside the tensor)
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j) {
                        const int c = nt * BN + 4 * (lane + 32 * j);
                        cp_async16(slot + 4u * (BM + 4 * (lane + 32 * j)), c < p.C ? sb_row + c : sb_row,
                                   c < p.C ? 16u : 0u);
                    }
                } else if (lane < BN / 128) {
                    const int c = nt * BN + lane * 128;
                    const float *src = p.sb + (int64_t)kb * p.sb_bstride + (int64_t)(c >> 7) * p.sb_cstride;
                    cp_async4(slot + 4u * (BM + lane), c < p.C ? src : p.sb, c < p.C ? 4u : 0u);
                }
                cp_async_arrive(sfull_bar(k));
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp >= FIRST_EPI_WARP) {
        // --------------------------------------------------- epilogue ---
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_EPILOGUE));
        const int q = warp & 3;                      // TMEM lane quarter this warp may access
        const int h = (warp - FIRST_EPI_WARP) >> 2;  // column half of the tile
        const int row = q * 32 + lane;               // tile row = TMEM lane

        int it = 0, uc = 0;
        bool ok = true;
        for (int u = unit0; ok && u < p.num_units; u += unit_step, ++uc) {
            const Unit wu = unit_of(p, u);
            const int mt = wu.mt, nt = wu.nt;
            const int col0 = nt * BN + h * 128;
            const bool half_ok = col0 < p.C;
            float2 acc[64];
#pragma unroll
            for (int j = 0; j < 64; ++j)
                acc[j] = make_float2(0.0f, 0.0f);
            for (int kb = wu.kb0; kb < (kOnce ? wu.kb0 + 1 : wu.kb1); ++kb, ++it) {
                const int buf = kOnce ? (uc & 1) : (it & 1);
                const uint32_t bph = kOnce ? ((uint32_t)(uc >> 1) & 1u) : ((uint32_t)(it >> 1) & 1u);
                const int k = it % SCALE_SLOTS;
                const uint32_t sph = (uint32_t)(it / SCALE_SLOTS) & 1u;
                // every lane acquires the scales and the partial itself; the
                // decision is warp-uniform because tcgen05.ld is .sync.aligned.  With
                // column scales both barriers are first probed back to back (two
                // independent shared-memory operations in flight; measured 2% on
                // WGrad); the block-scaled epilogue has no registers to spare for it.
                bool w;
                if (kMode != MODE_BLOCK && mbar_try_wait(sfull_bar(k), sph) & mbar_try_wait(tfull_bar(buf), bph))
                    w = true;
                else
                    w = mbar_wait(sfull_bar(k), sph, abort_flag, p.timeout_ns, SITE_EPI_SCALE_FULL) &&
                        mbar_wait(tfull_bar(buf), bph, abort_flag, p.timeout_ns, SITE_EPI_TMEM_FULL);
                if (!__all_sync(0xFFFFFFFFu, w)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t slot = smem_u32(ring) + (uint32_t)(k * SLOT_FLOATS * 4);
                const float sa = lds_f32(slot + 4u * row);
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + h * 128);
                uint32_t ra[32], rb[32];
                if (kMode == MODE_BLOCK) {
                    const float scl = sa * lds_f32(slot + 4u * (BM + h));
                    const float2 scl2 = make_float2(scl, scl);
                    tmem_ld32_async(taddr, ra);
                    tmem_wait32(ra);
                    tmem_ld32_async(taddr + 32, rb);
                    promote_chunk(&acc[0], ra, scl2);
                    tmem_wait32(rb);
                    tmem_ld32_async(taddr + 64, ra);
                    promote_chunk(&acc[16], rb, scl2);
                    tmem_wait32(ra);
                    tmem_ld32_async(taddr + 96, rb);
                    promote_chunk(&acc[32], ra, scl2);
                    tmem_wait32(rb);
                    promote_chunk(&acc[48], rb, scl2);
                    release_tmem<kPair>(tempty_bar(buf), lane);
                } else {
                    // MODE_COLS: acc += P * (sa * sb[c]); MODE_ONCE: the same product
                    // into a zero accumulator, once per unit
                    const uint32_t sbs = slot + 4u * (BM + h * 128);
                    const float2 sa2v = make_float2(sa, sa);
                    tmem_ld32_async(taddr, ra);
                    tmem_wait32(ra);
                    tmem_ld32_async(taddr + 32, rb);
                    promote_chunk_cols(&acc[0], ra, sa2v, sbs);
                    tmem_wait32(rb);
                    tmem_ld32_async(taddr + 64, ra);
                    promote_chunk_cols(&acc[16], rb, sa2v, sbs + 128);
                    tmem_wait32(ra);
                    tmem_ld32_async(taddr + 96, rb);
                    promote_chunk_cols(&acc[32], ra, sa2v, sbs + 256);
                    tmem_wait32(rb);
                    // column-scaled: released before the last chunk's FMAs (registers only);
                    // a same-box A/B measured this 1% faster for WGrad but 8% slower for the
                    // block-scaled mode above, which releases after them
                    release_tmem<kPair>(tempty_bar(buf), lane);
                    promote_chunk_cols(&acc[48], rb, sa2v, sbs + 384);
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(sempty_bar(k));  // the scales are read
            }
            if (kPair && p.out_mode == OUT_F32_ACC) {
                // this warp's 32 rows x 128 fp32 columns added into the caller's gradient
                // in rounds of 32 columns: each round is staged as 32 rows of 128 bytes
                // (16-byte chunks XOR-swizzled by row % 8, the map's 128-byte swizzle)
                // and added at L2 by a TMA reduce; rows beyond R and columns beyond C
                // are clipped by the tensor map
                const uint32_t stg = smem_u32(staging) + (uint32_t)((warp - FIRST_EPI_WARP) * STG_WARP_BYTES);
                const int y = mt * Cf::TILE_M + row_offset<kPair>() + q * 32;
#pragma unroll
                for (int rd = 0; rd < 4; ++rd) {
                    if (lane == 0)
                        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // buffer read out
                    __syncwarp();
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        const int j = 16 * rd + 2 * v;  // acc pairs of columns 32 rd + 4 v .. + 3
                        const uint32_t addr = stg + (uint32_t)(lane * 128 + ((v ^ (lane & 7)) << 4));
                        if (ok)
                            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(acc[j].x),
                                         "f"(acc[j].y), "f"(acc[j + 1].x), "f"(acc[j + 1].y)
                                         : "memory");
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> TMA reads
                    __syncwarp();
                    if (lane == 0 && ok && half_ok) {
                        tma_reduce_add_2d(&tmOut, stg, col0 + 32 * rd, y);
                        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                    }
                }
                continue;
            }
            if (kPair && p.out_mode == OUT_BF16) {
                // this warp's 32 rows x 128 columns in rounds of STG_COLS columns: each
                // round is staged as 32 rows of STG_COLS * 2 bytes (16-byte chunks
                // XOR-swizzled by row % 8, the tensor map's 128-byte swizzle; a 64-column
                // round is one 128-byte box row) and leaves by TMA stores; rows beyond R
                // are clipped by the tensor map
                const uint32_t stg = smem_u32(staging) + (uint32_t)((warp - FIRST_EPI_WARP) * STG_WARP_BYTES);
                const int y = mt * Cf::TILE_M + row_offset<kPair>() + q * 32;
#pragma unroll
                for (int rd = 0; rd < 128 / STG_COLS; ++rd) {
                    if (lane == 0)
                        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // buffer read out
                    __syncwarp();
#pragma unroll
                    for (int v = 0; v < STG_COLS / 8; ++v) {
                        const int j = rd * (STG_COLS / 2) + 4 * v;  // acc pairs of columns 8v .. 8v + 7
                        const uint32_t addr = stg + (uint32_t)((v >> 3) * 32 * 128 + lane * 128 +
                                                               (((v & 7) ^ (lane & 7)) << 4));
                        if (ok)
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                                         "r"(bf16x2_rn(acc[j])), "r"(bf16x2_rn(acc[j + 1])),
                                         "r"(bf16x2_rn(acc[j + 2])), "r"(bf16x2_rn(acc[j + 3]))
                                         : "memory");
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> TMA reads
                    __syncwarp();
                    if (lane == 0 && ok && half_ok) {
                        const uint64_t pol = l2_policy(false);  // the output is not read again here
                        tma_store_2d_hint(&tmOut, stg, col0 + rd * STG_COLS, y, pol);
                        if (STG_COLS == 128)
                            tma_store_2d_hint(&tmOut, stg + 32 * 128, col0 + rd * STG_COLS + 64, y, pol);
                        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                    }
                }
                continue;
            }
            // Single CTAs: this thread's row, 128 columns, stored directly (512 or 256
            // contiguous bytes per thread); rows beyond R are skipped.  (Pairs leave by
            // TMA above; the host pairs CTAs only for unsplit GEMMs.)
            const int grow = mt * Cf::TILE_M + row_offset<kPair>() + row;
            if (!kPair && ok && half_ok && grow < p.R) {
                if (p.out_mode == OUT_F32_PARTIAL) {
                    // fp32 partial of this contraction range, plane `split` of [splits][R][C]
                    float4 *dst = reinterpret_cast<float4 *>(p.ws + ((int64_t)wu.split * p.R + grow) * p.C + col0);
#pragma unroll
                    for (int v = 0; v < 32; ++v)
                        dst[v] = make_float4(acc[2 * v].x, acc[2 * v].y, acc[2 * v + 1].x, acc[2 * v + 1].y);
                } else if (p.out_mode == OUT_F32_ACC) {
                    // acc_out[r, c] += the product, in fp32 (each element owned by this thread)
                    float4 *dst = reinterpret_cast<float4 *>(p.acc_out + (int64_t)grow * p.ld_acc + col0);
#pragma unroll
                    for (int v = 0; v < 32; ++v) {
                        float4 o = dst[v];
                        o.x += acc[2 * v].x;
                        o.y += acc[2 * v].y;
                        o.z += acc[2 * v + 1].x;
                        o.w += acc[2 * v + 1].y;
                        dst[v] = o;
                    }
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + (int64_t)grow * p.ldo + col0);
#pragma unroll
                    for (int v = 0; v < 16; ++v)
                        dst[v] = make_uint4(bf16x2_rn(acc[4 * v]), bf16x2_rn(acc[4 * v + 1]),
                                            bf16x2_rn(acc[4 * v + 2]), bf16x2_rn(acc[4 * v + 3]));
                }
            }
        }
    }

    if (kPair && warp >= FIRST_EPI_WARP && lane == 0)
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // stores complete before exit
    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) {
        if (warp == 1) {
            if (cta_rank() == 1 && lane == 0) {
                // the even CTA's last commit: every MMA writing this CTA's TMEM or
                // reading its shared memory has completed
                volatile uint32_t never = 0;
                mbar_wait(teardown_bar, 0, &never, p.timeout_ns, SITE_TEARDOWN);
            }
            __syncwarp();
        }
        // neither CTA leaves while the other may still signal its barriers
        cluster_sync();
    }
    if (warp == 1) {
        tc_fence_after();
        if constexpr (kPair)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                         : "memory");
    }
}

// A barrier nothing arrives on: exercises the bounded wait and the error word.
__global__ void k_diag_wait(uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_wait(smem_u32(&bar), 0, &abort_flag, limit_ns, SITE_DIAG);
}

// Split-K reduction: out[r, c] = bf16_RN(sum over splits s, in order, of
// ws[(s * R + r) * C + c]); eight columns per thread (C % 128 == 0).
__global__ void __launch_bounds__(256) k_splitk_reduce(const float *__restrict__ ws, int splits, int R, int C,
                                                       uint16_t *__restrict__ out, int64_t ldo)
{
    pdl_begin();
    const int64_t per_row = C / 8;
    const int64_t total = (int64_t)R * per_row;
    const int64_t plane = (int64_t)R * C;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / per_row, c = (i - r * per_row) * 8;
        const float4 *src = reinterpret_cast<const float4 *>(ws + r * C + c);
        float4 a = src[0], b = src[1];
        for (int sp = 1; sp < splits; ++sp) {
            const float4 *t = reinterpret_cast<const float4 *>(ws + sp * plane + r * C + c);
            const float4 x = t[0], y = t[1];
            a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
            b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
        }
        *reinterpret_cast<uint4 *>(out + r * ldo + c) =
            make_uint4(bf16x2_rn(make_float2(a.x, a.y)), bf16x2_rn(make_float2(a.z, a.w)),
                       bf16x2_rn(make_float2(b.x, b.y)), bf16x2_rn(make_float2(b.z, b.w)));
    }
}

// acc[r][c] += the split sums added in split order (fp32), for an fp32
// gradient that accumulates several GEMMs (micro-batches).
__global__ void __launch_bounds__(256) k_splitk_reduce_acc(const float *__restrict__ ws, int splits, int R, int C,
                                                           float *__restrict__ acc, int64_t ld_acc)
{
    pdl_begin();
    const int64_t per_row = C / 4;
    const int64_t total = (int64_t)R * per_row;
    const int64_t plane = (int64_t)R * C;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / per_row, c = (i - r * per_row) * 4;
        float4 a = *reinterpret_cast<const float4 *>(ws + r * C + c);
        for (int sp = 1; sp < splits; ++sp) {
            const float4 x = *reinterpret_cast<const float4 *>(ws + sp * plane + r * C + c);
            a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
        }
        float4 *d = reinterpret_cast<float4 *>(acc + r * ld_acc + c);
        float4 v = *d;
        v.x += a.x; v.y += a.y; v.z += a.z; v.w += a.w;
        *d = v;
    }
}

// ---------------------------------------------------------------- host ---

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

uint64_t wait_limit_ns()
{
    static uint64_t ns = [] {
        const char *e = std::getenv("RLQ_WAIT_TIMEOUT_MS");
        long long ms = e ? std::atoll(e) : 1000;
        if (ms < 1)
            ms = 1;
        if (ms > 600000)
            ms = 600000;
        return (uint64_t)ms * 1000000ull;
    }();
    return ns;
}

// bf16 output [rows][cols], pitch ld elements; box 64 columns x 32 rows, 128-byte swizzle.
rlq_status encode_out_map(CUtensorMap *map, uint16_t *base, int64_t cols, int64_t rows, int64_t ld)
{
    auto enc = get_encode_fn();
    if (!enc)
        return fail(RLQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {64, 32};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(RLQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d) for the [%lld x %lld] output",
                    (int)r, (long long)rows, (long long)cols);
    return RLQ_OK;
}

// fp32 gradient [rows][cols], pitch ld elements, for TMA reduce-adds: box 32 columns
// (128 bytes) x 32 rows, 128-byte swizzle.
rlq_status encode_acc_map(CUtensorMap *map, float *base, int64_t cols, int64_t rows, int64_t ld)
{
    auto enc = get_encode_fn();
    if (!enc)
        return fail(RLQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(RLQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d) for the [%lld x %lld] fp32 gradient",
                    (int)r, (long long)rows, (long long)cols);
    return RLQ_OK;
}

// 2-D E4M3 tensor [rows][inner] with row pitch `ld` bytes; box 128 x box_rows.
rlq_status encode_map(CUtensorMap *map, const uint8_t *base, int64_t inner, int64_t rows, int64_t ld, int box_rows)
{
    auto enc = get_encode_fn();
    if (!enc)
        return fail(RLQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(RLQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d) for a [%lld x %lld] operand, pitch %lld",
                    (int)r, (long long)rows, (long long)inner, (long long)ld);
    return RLQ_OK;
}

struct DevInfo {
    int sms = 0;
    bool attr_set[16] = {};
    int max_clusters[16] = {};  // co-resident CTA pairs of each paired variant (0: not yet known, -1: none)
};

DevInfo &dev_info(int dev)
{
    static DevInfo info[64];
    static std::mutex mu;
    std::lock_guard<std::mutex> g(mu);
    DevInfo &d = info[dev & 63];
    if (d.sms == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        d.sms = n > 0 ? n : 1;
    }
    return d;
}

// ---- split-K planning ----
//
// Estimated time of an R x C x L GEMM cut into S contraction splits: the
// persistent grid runs ceil(tiles * S / SMs) waves of units, each unit streams
// ceil(kblocks / S) blocks of 128 x 256 x 128 plus a fixed fill/drain cost;
// splitting adds the fp32 partial planes (written once, read once) and the
// reduction launch.  Figures are per-SM steady-state rates of this kernel.
constexpr double SPLIT_T_BLOCK_US = 0.55;   // one 128x256x128 block on one SM
constexpr double SPLIT_T_UNIT_US = 1.5;     // pipeline fill + epilogue drain per unit
constexpr double SPLIT_T_REDUCE_US = 3.0;   // reduction launch and tail
constexpr double SPLIT_HBM_BYTES_US = 6.0e6;
constexpr int SPLIT_MAX = 16;
constexpr int SPLIT_MIN_BLOCKS = 4;         // contraction blocks per unit, at least

int plan_splits(int64_t R, int64_t C, int64_t L, int sms, int64_t ws_cap)
{
    const int64_t kblocks = (L + BK - 1) / BK;
    const int64_t tiles = ((R + BM - 1) / BM) * ((C + BN - 1) / BN);
    if (tiles == 0 || kblocks < 2 * SPLIT_MIN_BLOCKS)
        return 1;
    const double plane = (double)R * (double)C * 4.0;
    int best = 1;
    double best_t = 0.0;
    int prev_splits = 0;
    for (int s = 1; s <= SPLIT_MAX && s * SPLIT_MIN_BLOCKS <= kblocks; ++s) {
        const int64_t kbps = (kblocks + s - 1) / s;
        const int splits = (int)((kblocks + kbps - 1) / kbps);  // every split non-empty
        if (splits == prev_splits)
            continue;
        prev_splits = splits;
        if (splits > 1 && ws_cap >= 0 && (double)splits * plane > (double)ws_cap)
            break;
        const int64_t waves = (tiles * splits + sms - 1) / sms;
        double t = (double)waves * ((double)kbps * SPLIT_T_BLOCK_US + SPLIT_T_UNIT_US);
        if (splits > 1)
            t += (2.0 * splits * plane + (double)R * C * 2.0) / SPLIT_HBM_BYTES_US + SPLIT_T_REDUCE_US;
        if (splits == 1 || t < 0.97 * best_t) {  // a split must pay for itself clearly
            best = splits;
            best_t = t;
        }
    }
    return best;
}

// Pairs of CTAs (cta_group::2 MMAs) unless RLQ_GEMM_PAIR=0 is set in the environment.
bool pair_mode_enabled()
{
    static const bool on = [] {
        const char *e = std::getenv("RLQ_GEMM_PAIR");
        return !(e && e[0] == '0');
    }();
    return on;
}

template <int kMode, bool kBMN, bool kPair>
rlq_status launch_impl(const GemmArgs &a, int splits, cudaStream_t st, bool withhold_first_load = false)
{
    using Cf = Cfg<kPair>;
    CUtensorMap tmA, tmB, tmO;
    rlq_status rs = encode_map(&tmA, a.A, a.L, a.R, a.lda, BM);
    if (rs != RLQ_OK)
        return rs;
    // B is [C][L] (K-major; boxes of the B rows one CTA stages) or [L][C] (MN-major,
    // boxes of 128 columns x 128 rows)
    rs = kBMN ? encode_map(&tmB, a.B, a.C, a.L, a.ldb, BK) : encode_map(&tmB, a.B, a.L, a.C, a.ldb, Cf::B_ROWS);
    if (rs != RLQ_OK)
        return rs;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_status(e, "cudaGetDevice");
    DevInfo &di = dev_info(dev);
    const int variant = kMode * 4 + (kBMN ? 2 : 0) + (kPair ? 1 : 0);
    auto kernel = k_gemm_block_scaled<kMode, kBMN, kPair>;
    if (!di.attr_set[variant]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM_BYTES);
        if (e != cudaSuccess)
            return cuda_status(e, "cudaFuncSetAttribute(max dynamic shared memory)");
        di.attr_set[variant] = true;
    }
    // [0] programmatic dependent launch (every kernel of the library begins with
    // pdl_begin), [1] CTA pairs
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = 2;
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cf::SMEM_BYTES;
    cfg.stream = st;
    cfg.attrs = attrs;
    cfg.numAttrs = kPair ? 2 : 1;
    if constexpr (kPair) {
        if (di.max_clusters[variant] == 0) {
            cudaLaunchConfig_t q = cfg;  // the occupancy query sees the cluster shape only
            q.gridDim = dim3(2 * (di.sms / 2), 1, 1);
            q.attrs = attrs + 1;
            q.numAttrs = 1;
            int n = 0;
            e = cudaOccupancyMaxActiveClusters(&n, kernel, &q);
            if (e != cudaSuccess)
                return cuda_status(e, "cudaOccupancyMaxActiveClusters");
            di.max_clusters[variant] = n < 1 ? -1 : n;  // -1: no pair fits, use single CTAs
        }
        if (di.max_clusters[variant] < 0)
            return launch_impl<kMode, kBMN, false>(a, splits, st, withhold_first_load);
    }
    Params p;
    p.sa = a.sa;
    p.ld_sa = a.ld_sa;
    p.sb = a.sb;
    p.sb_bstride = a.sb_bstride;
    p.sb_cstride = a.sb_cstride;
    p.out = a.out;
    p.ldo = a.ldo;
    p.acc_out = a.acc;
    p.ld_acc = a.ld_acc;
    p.R = (int)a.R;
    p.C = (int)a.C;
    p.kblocks = (int)((a.L + BK - 1) / BK);
    p.m_tiles = (int)((a.R + Cf::TILE_M - 1) / Cf::TILE_M);
    p.n_tiles = (int)((a.C + BN - 1) / BN);
    p.num_tiles = p.m_tiles * p.n_tiles;
    // keep the smaller operand resident in L2: sweep the tiles along it
    p.m_fastest = (a.R * a.L <= a.C * a.L) ? 1 : 0;
    p.timeout_ns = wait_limit_ns();
    p.withhold_first_load = (!kPair && withhold_first_load) ? 1 : 0;
    p.kbps = (p.kblocks + splits - 1) / splits;
    p.splits = (p.kblocks + p.kbps - 1) / p.kbps;
    p.num_units = p.num_tiles * p.splits;
    p.ws = p.splits > 1 ? a.ws : nullptr;
    p.out_mode = p.splits > 1 ? OUT_F32_PARTIAL : (a.acc ? OUT_F32_ACC : OUT_BF16);
    if (kPair && p.out_mode == OUT_F32_ACC) {
        rs = encode_acc_map(&tmO, a.acc, a.C, a.R, a.ld_acc);
        if (rs != RLQ_OK)
            return rs;
    } else if (kPair && p.out_mode == OUT_BF16) {
        rs = encode_out_map(&tmO, a.out, a.C, a.R, a.ldo);
        if (rs != RLQ_OK)
            return rs;
    } else {
        tmO = tmA;  // not read
    }
    if (kPair) {
        const int pairs = p.num_units < di.max_clusters[variant] ? p.num_units : di.max_clusters[variant];
        cfg.gridDim = dim3(2 * pairs, 1, 1);
    } else {
        cfg.gridDim = dim3(p.num_units < di.sms ? p.num_units : di.sms, 1, 1);
    }
    e = cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmO, p);
    if (e == cudaSuccess)
        e = cudaGetLastError();
    if (e != cudaSuccess || p.splits == 1)
        return cuda_status(e, "block-scaled GEMM launch");
    const int64_t total = a.R * (a.C / 8);
    int64_t rgrid = (total + 255) / 256;
    if (rgrid > (int64_t)di.sms * 8)
        rgrid = (int64_t)di.sms * 8;
    if (a.acc)
        (void)launch_pdl(k_splitk_reduce_acc, dim3((int)rgrid), dim3(256), 0, st, a.ws, p.splits, p.R, p.C, a.acc, a.ld_acc);
    else
        (void)launch_pdl(k_splitk_reduce, dim3((int)rgrid), dim3(256), 0, st, a.ws, p.splits, p.R, p.C, a.out, a.ldo);
    return cuda_status(cudaGetLastError(), "split-K reduction launch");
}

template <int kMode, bool kBMN>
rlq_status launch_mode(const GemmArgs &a, int splits, cudaStream_t st, bool pair, bool stall)
{
    return pair ? launch_impl<kMode, kBMN, true>(a, splits, st) : launch_impl<kMode, kBMN, false>(a, splits, st, stall);
}

// One-shot diagnostic armed by arm_gemm_stall() for the calling thread.
thread_local bool t_stall_armed = false;

rlq_status current_sms(int *sms)
{
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_status(e, "cudaGetDevice");
    *sms = dev_info(dev).sms;
    return RLQ_OK;
}

}  // namespace

rlq_status launch_gemm(const GemmArgs &a, cudaStream_t st)
{
    if (a.R == 0 || a.C == 0)
        return RLQ_OK;
    if (a.L == 0) {
        // empty contraction: the sum is zero (nothing to add in accumulate mode)
        if (a.acc)
            return RLQ_OK;
        return cuda_status(cudaMemset2DAsync(a.out, (size_t)a.ldo * 2, 0, (size_t)a.C * 2, (size_t)a.R, st),
                           "cudaMemset2DAsync (empty contraction)");
    }
    int splits = 1;
    if (a.ws) {
        int64_t bytes = 0;
        const rlq_status rs = plan_splitk(a.R, a.C, a.L, a.ws_bytes, &splits, &bytes);
        if (rs != RLQ_OK)
            return rs;
    }
    // the armed stall diagnostic applies to this launch only, on single CTAs
    const bool stall = t_stall_armed;
    t_stall_armed = false;
    // CTA pairs for tiles of 256 output rows; one CTA per 128 rows when the output
    // has fewer rows or the contraction is split
    const bool pair = splits == 1 && a.R >= 2 * BM && pair_mode_enabled() && !stall;
    if (a.scale_once)
        return launch_mode<MODE_ONCE, false>(a, splits, st, pair, stall);
    if (a.per_col_sb)
        return launch_mode<MODE_COLS, false>(a, splits, st, pair, stall);
    if (a.b_mn_major)
        return launch_mode<MODE_BLOCK, true>(a, splits, st, pair, stall);
    return launch_mode<MODE_BLOCK, false>(a, splits, st, pair, stall);
}

void arm_gemm_stall() { t_stall_armed = true; }

rlq_status plan_splitk(int64_t R, int64_t C, int64_t L, int64_t ws_cap, int *splits, int64_t *ws_bytes)
{
    int sms = 0;
    const rlq_status rs = current_sms(&sms);
    if (rs != RLQ_OK)
        return rs;
    int s = (R > 0 && C > 0 && L > 0) ? plan_splits(R, C, L, sms, ws_cap) : 1;
    *splits = s;
    *ws_bytes = s > 1 ? (int64_t)s * R * C * 4 : 0;
    return RLQ_OK;
}

rlq_status launch_splitk_reduce(const float *ws, int splits, int64_t R, int64_t C, uint16_t *out, int64_t ldo, int sms,
                                cudaStream_t st)
{
    const int64_t total = R * (C / 8);
    int64_t rgrid = (total + 255) / 256;
    if (rgrid > (int64_t)sms * 8)
        rgrid = (int64_t)sms * 8;
    (void)launch_pdl(k_splitk_reduce, dim3((int)rgrid), dim3(256), 0, st, ws, splits, (int)R, (int)C, out, ldo);
    return cuda_status(cudaGetLastError(), "split-K reduction launch");
}

rlq_status check_device_errors(cudaStream_t st)
{
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return cuda_status(e, "cudaStreamSynchronize");
    // every translation unit with bounded-wait kernels keeps its own error word
    unsigned long long words[2] = {0, 0};
    e = take_error_word(st, &words[0]);
    if (e == cudaSuccess)
        e = take_nvfp4_error_word(st, &words[1]);
    if (e != cudaSuccess)
        return cuda_status(e, "reading and clearing the device error words");
    const unsigned long long word = words[0] ? words[0] : words[1];
    if (word == 0)
        return RLQ_OK;
    const uint32_t code = (uint32_t)word, site = (uint32_t)(word >> 32);
    static const char *names[] = {"?", "TMA producer (stage free)", "MMA issuer (TMEM buffer free)",
                                  "MMA issuer (stage loaded)", "epilogue (partial ready)", "teardown", "drain",
                                  "scale loader (slot free)", "epilogue (scales ready)", "FP4 converter (stage free)"};
    const char *where = site == SITE_DIAG ? "diagnostic wait" : (site < 10 ? names[site] : "?");
    return fail((rlq_status)code, "device-side wait ran out at site %u (%s)%s", site, where,
                words[1] && !words[0] ? " in the NVFP4 GEMM" : "");
}

rlq_status launch_diag_wait(int64_t timeout_us, cudaStream_t st)
{
    k_diag_wait<<<1, 32, 0, st>>>((uint64_t)timeout_us * 1000ull);
    return cuda_status(cudaGetLastError(), "diagnostic wait launch");
}

}  // namespace rlq
