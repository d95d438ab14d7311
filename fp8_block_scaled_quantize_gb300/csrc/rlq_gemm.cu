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
//   * an MMA warp issues, per contraction block, four tcgen05.mma
//     (kind::f8f6f4, M=128, N=256, K=32) into one of two TMEM partial buffers
//     (2 x 256 fp32 columns = the whole 512-column TMEM), then commits;
//   * eight epilogue warps read the finished partial with tcgen05.ld, multiply
//     by sa * sb and accumulate into fp32 registers (packed f32x2 FMA), release
//     the TMEM buffer, and after the last block round to bf16 and store.
//
// The scales are read by the epilogue straight from global memory, two blocks
// ahead of use (per-row / per-block scales into registers; WGrad's per-column
// scale rows through an L1 prefetch and broadcast loads).  They are not staged
// through the shared-memory ring: generic-proxy reads of a buffer that the
// async proxy (TMA) rewrites are not ordered by the stage barriers alone, and
// a ring-staged variant measured non-deterministic.
//
// Tiles are 128 x 256; the kernel is persistent (one CTA per SM) and walks
// the tile list with the smaller operand resident in L2.  Every mbarrier wait
// is bounded: on timeout the waiting thread records an error word that
// rlq_check() reports, raises a CTA-wide abort flag, and the CTA drains its
// in-flight copies and MMAs, frees TMEM and exits.  Nothing traps.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "rlq_internal.h"

namespace rlq {

// First error recorded on this device: bits 0..31 status code, 32..63 site.
__device__ unsigned long long g_rlq_error_word;

namespace {

constexpr int BM = 128;                    // tile rows (TMEM lanes)
constexpr int BN = 256;                    // tile columns (MMA N)
constexpr int BK = 128;                    // contraction block = scale granularity = 128 bytes of E4M3
constexpr int UMMA_K = 32;                 // K of one kind::f8f6f4 MMA
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;           // 16 KB
constexpr int B_BYTES = BN * BK;           // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
// Warpgroup 0: warp 0 TMA, warp 1 MMA (and TMEM owner), warps 2-3 idle.
// Warpgroups 1-2: eight epilogue warps.  Registers are rebalanced with
// setmaxnreg: 128 x 40 + 256 x 232 = 384 x 168, the launch allocation.
constexpr int NUM_THREADS = 384;
constexpr int FIRST_EPI_WARP = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int REGS_PRODUCER = 40;
constexpr int REGS_EPILOGUE = 232;
constexpr int TMEM_COLS = 2 * BN;          // two partial buffers
constexpr int NUM_BARS = 2 * STAGES + 4 + 1;
constexpr int SMEM_BYTES = 1024 /* alignment slack */ + STAGES * STAGE_BYTES + NUM_BARS * 8 + 16;

// Instruction descriptor of tcgen05.mma kind::f8f6f4: D fp32 (bits 4-5 = 1),
// A and B E4M3 (format 0 in bits 7-9 / 10-12), both K-major (bits 15/16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t IDESC = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

// Error sites (reported by rlq_check / rlq_last_error).
enum : uint32_t {
    SITE_PRODUCER_EMPTY = 1,
    SITE_MMA_TMEM_EMPTY = 2,
    SITE_MMA_FULL = 3,
    SITE_EPI_TMEM_FULL = 4,
    SITE_TEARDOWN = 5,
    SITE_DRAIN = 6,
    SITE_DIAG = 99,
};

// ------------------------------------------------------------ PTX helpers ---

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record_error(uint32_t code, uint32_t site)
{
    atomicCAS(&g_rlq_error_word, 0ull, ((unsigned long long)site << 32) | code);
}

// Waits for the phase of `bar` with the given parity.  Returns false, without
// waiting further, once the CTA's abort flag is up or after limit_ns; in the
// second case it records a timeout and raises the flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                       uint64_t limit_ns, uint32_t site)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 31) == 0) {
            if (*abort_flag)
                return false;
            if (global_timer_ns() - t0 > limit_ns) {
                record_error(RLQ_ERR_TIMEOUT, site);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        ::"r"(dst), "l"((uint64_t)map), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void prefetch_l1(const void *p)
{
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(IDESC), "r"(accumulate)
        : "memory");
}

// Issues a load of 32 consecutive fp32 columns of this warp's 32 TMEM lanes
// into r; the registers are valid only after tmem_wait32(r).
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Waits for the outstanding TMEM loads.  The registers of r are tied to the
// wait as in/out operands so that no use of them is scheduled before it.
__device__ __forceinline__ void tmem_wait32(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row core-matrix groups 1024 bytes apart (SBO), version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ uint64_t f2_bits(float lo, float hi)
{
    return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}

// acc += p * scale, two lanes at a time.
__device__ __forceinline__ void ffma2(uint64_t &acc, uint64_t p, uint64_t scale)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(p), "l"(scale));
}

__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Keeps the compiler from sinking the FMAs of one TMEM chunk below the next
// chunk's load (which would hold several chunks in registers at once).
__device__ __forceinline__ void reg_fence16(uint64_t *a)
{
    asm volatile(""
                 : "+l"(a[0]), "+l"(a[1]), "+l"(a[2]), "+l"(a[3]), "+l"(a[4]), "+l"(a[5]), "+l"(a[6]), "+l"(a[7]),
                   "+l"(a[8]), "+l"(a[9]), "+l"(a[10]), "+l"(a[11]), "+l"(a[12]), "+l"(a[13]), "+l"(a[14]), "+l"(a[15]));
}

// acc[0..15] += chunk * scale (one scale for the whole chunk).
__device__ __forceinline__ void promote_chunk(uint64_t *acc, const uint32_t (&r)[32], uint64_t scl2)
{
#pragma unroll
    for (int j = 0; j < 16; ++j)
        ffma2(acc[j], f2_bits(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), scl2);
    reg_fence16(acc);
}

// acc[0..15] += chunk * sa * sb[column]; sb is 32 consecutive column scales in
// global memory, read by every lane (broadcast).
__device__ __forceinline__ void promote_chunk_cols(uint64_t *acc, const uint32_t (&r)[32], uint64_t sa2,
                                                   const float4 *sbs)
{
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float4 sb4 = __ldg(sbs + j);
        const uint64_t s01 = fmul2(sa2, f2_bits(sb4.x, sb4.y));
        const uint64_t s23 = fmul2(sa2, f2_bits(sb4.z, sb4.w));
        ffma2(acc[2 * j], f2_bits(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1])), s01);
        ffma2(acc[2 * j + 1], f2_bits(__uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])), s23);
    }
    reg_fence16(acc);
}

__device__ __forceinline__ uint32_t bf16x2_rn(uint64_t v)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "r"((uint32_t)(v >> 32)), "r"((uint32_t)v));
    return d;
}

struct Params {
    const float *sa;
    int64_t ld_sa;
    const float *sb;
    int64_t sb_bstride;
    int64_t sb_cstride;
    uint16_t *out;
    int64_t ldo;
    int R, C;
    int kblocks;
    int m_tiles, n_tiles, num_tiles;
    int m_fastest;
    uint64_t timeout_ns;
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

template <bool kColScaleB>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_block_scaled(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
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

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);  // the stage is free once its MMAs completed
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), NUM_EPI_WARPS);
        }
        mbar_init(teardown_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp < FIRST_EPI_WARP)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_PRODUCER));
    if (warp == 0) {
        // ------------------------------------------------ TMA producer ---
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                int mt, nt;
                tile_coords(p, tile, mt, nt);
                for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                    if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, p.timeout_ns, SITE_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(s), STAGE_BYTES);
                    tma_load_2d(a_stage(s), &tmA, full_bar(s), kb * BK, mt * BM);
                    tma_load_2d(b_stage(s), &tmB, full_bar(s), kb * BK, nt * BN);
                }
            }
            if (!ok) {
                // drain: the copies issued into the last stages complete on their own
                const int first = it > STAGES ? it - STAGES : 0;
                for (int j = first; j < it; ++j) {
                    volatile uint32_t never = 0;
                    mbar_wait(full_bar(j % STAGES), (uint32_t)(j / STAGES) & 1u, &never, 20000000ull, SITE_DRAIN);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer ---
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                    const int buf = it & 1;
                    const uint32_t bph = (uint32_t)(it >> 1) & 1u;
                    if (!mbar_wait(tempty_bar(buf), bph ^ 1u, abort_flag, p.timeout_ns, SITE_MMA_TMEM_EMPTY) ||
                        !mbar_wait(full_bar(s), ph, abort_flag, p.timeout_ns, SITE_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + (uint32_t)(buf * BN);
                    const uint64_t ad = sw128_desc(a_stage(s));
                    const uint64_t bd = sw128_desc(b_stage(s));
#pragma unroll
                    for (int j = 0; j < BK / UMMA_K; ++j)  // +32 bytes along K = +2 in the address field
                        tc_mma_f8(d, ad + 2 * j, bd + 2 * j, j > 0 ? 1u : 0u);
                    tc_commit(empty_bar(s));
                    tc_commit(tfull_bar(buf));
                }
            }
            // every MMA issued above has completed once this commit arrives
            tc_commit(teardown_bar);
            volatile uint32_t never = 0;
            mbar_wait(teardown_bar, 0, &never, 20000000ull, SITE_TEARDOWN);
        }
    } else if (warp >= FIRST_EPI_WARP) {
        // --------------------------------------------------- epilogue ---
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_EPILOGUE));
        const int q = warp & 3;                      // TMEM lane quarter this warp may access
        const int h = (warp - FIRST_EPI_WARP) >> 2;  // column half of the tile
        const int row = q * 32 + lane;               // tile row = TMEM lane

        // The block scales are fetched two contraction blocks ahead (crossing
        // tile boundaries) so that their global-memory latency stays hidden.
        int pf_tile = blockIdx.x, pf_kb = 0;
        auto fetch = [&](float &sa_o, float &sb_o) {
            sa_o = 0.0f;
            sb_o = 0.0f;
            if (pf_tile < p.num_tiles) {
                int mt, nt;
                tile_coords(p, pf_tile, mt, nt);
                const int grow = mt * BM + row;
                if (grow < p.R)
                    sa_o = __ldg(p.sa + (int64_t)pf_kb * p.ld_sa + grow);
                const int col0 = nt * BN + h * 128;
                if (!kColScaleB) {
                    if (col0 < p.C)
                        sb_o = __ldg(p.sb + (int64_t)pf_kb * p.sb_bstride + (int64_t)(col0 >> 7) * p.sb_cstride);
                } else if (col0 < p.C && lane < 4) {
                    // the warp's 128 column scales: four 128-byte lines
                    prefetch_l1(p.sb + (int64_t)pf_kb * p.sb_bstride + col0 + lane * 32);
                }
                if (++pf_kb == p.kblocks) {
                    pf_kb = 0;
                    pf_tile += gridDim.x;
                }
            }
        };
        float sa0, sb0, sa1, sb1, sa2, sb2;
        fetch(sa0, sb0);
        fetch(sa1, sb1);

        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
            int mt, nt;
            tile_coords(p, tile, mt, nt);
            const int grow = mt * BM + row;
            const bool row_ok = grow < p.R;
            const int col0 = nt * BN + h * 128;
            const bool half_ok = col0 < p.C;
            uint64_t acc[64];
#pragma unroll
            for (int j = 0; j < 64; ++j)
                acc[j] = 0;
            for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                const int buf = it & 1;
                const uint32_t bph = (uint32_t)(it >> 1) & 1u;
                fetch(sa2, sb2);
                // every lane acquires the partial itself; the decision is made
                // warp-uniform because tcgen05.ld is a .sync.aligned instruction
                const bool w = mbar_wait(tfull_bar(buf), bph, abort_flag, p.timeout_ns, SITE_EPI_TMEM_FULL);
                if (!__all_sync(0xFFFFFFFFu, w)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + h * 128);
                uint32_t ra[32], rb[32];
                if (!kColScaleB) {
                    const float scl = sa0 * sb0;
                    const uint64_t scl2 = f2_bits(scl, scl);
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
                } else {
                    const float4 *sbs = reinterpret_cast<const float4 *>(
                        p.sb + (int64_t)kb * p.sb_bstride + (half_ok ? col0 : 0));
                    const uint64_t sa2v = f2_bits(sa0, sa0);
                    tmem_ld32_async(taddr, ra);
                    tmem_wait32(ra);
                    tmem_ld32_async(taddr + 32, rb);
                    promote_chunk_cols(&acc[0], ra, sa2v, sbs);
                    tmem_wait32(rb);
                    tmem_ld32_async(taddr + 64, ra);
                    promote_chunk_cols(&acc[16], rb, sa2v, sbs + 8);
                    tmem_wait32(ra);
                    tmem_ld32_async(taddr + 96, rb);
                    promote_chunk_cols(&acc[32], ra, sa2v, sbs + 16);
                    tmem_wait32(rb);
                    promote_chunk_cols(&acc[48], rb, sa2v, sbs + 24);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(tempty_bar(buf));
                sa0 = sa1;
                sb0 = sb1;
                sa1 = sa2;
                sb1 = sb2;
            }
            if (ok && row_ok && half_ok) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + (int64_t)grow * p.ldo + col0);
#pragma unroll
                for (int v = 0; v < 16; ++v)
                    dst[v] = make_uint4(bf16x2_rn(acc[4 * v]), bf16x2_rn(acc[4 * v + 1]), bf16x2_rn(acc[4 * v + 2]),
                                        bf16x2_rn(acc[4 * v + 3]));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
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
    bool attr_set[2] = {false, false};
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

template <bool kCol>
rlq_status launch_impl(const GemmArgs &a, cudaStream_t st)
{
    CUtensorMap tmA, tmB;
    rlq_status rs = encode_map(&tmA, a.A, a.L, a.R, a.lda, BM);
    if (rs != RLQ_OK)
        return rs;
    rs = encode_map(&tmB, a.B, a.L, a.C, a.ldb, BN);
    if (rs != RLQ_OK)
        return rs;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_status(e, "cudaGetDevice");
    DevInfo &di = dev_info(dev);
    if (!di.attr_set[kCol]) {
        e = cudaFuncSetAttribute(k_gemm_block_scaled<kCol>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess)
            return cuda_status(e, "cudaFuncSetAttribute(max dynamic shared memory)");
        di.attr_set[kCol] = true;
    }
    Params p;
    p.sa = a.sa;
    p.ld_sa = a.ld_sa;
    p.sb = a.sb;
    p.sb_bstride = a.sb_bstride;
    p.sb_cstride = a.sb_cstride;
    p.out = a.out;
    p.ldo = a.ldo;
    p.R = (int)a.R;
    p.C = (int)a.C;
    p.kblocks = (int)((a.L + BK - 1) / BK);
    p.m_tiles = (int)((a.R + BM - 1) / BM);
    p.n_tiles = (int)((a.C + BN - 1) / BN);
    p.num_tiles = p.m_tiles * p.n_tiles;
    // keep the smaller operand resident in L2: sweep the tiles along it
    p.m_fastest = (a.R * a.L <= a.C * a.L) ? 1 : 0;
    p.timeout_ns = wait_limit_ns();
    const int grid = p.num_tiles < di.sms ? p.num_tiles : di.sms;
    k_gemm_block_scaled<kCol><<<grid, NUM_THREADS, SMEM_BYTES, st>>>(tmA, tmB, p);
    return cuda_status(cudaGetLastError(), "block-scaled GEMM launch");
}

}  // namespace

rlq_status launch_gemm(const GemmArgs &a, cudaStream_t st)
{
    if (a.R == 0 || a.C == 0)
        return RLQ_OK;
    if (a.L == 0) {
        // empty contraction: the sum is zero
        return cuda_status(cudaMemset2DAsync(a.out, (size_t)a.ldo * 2, 0, (size_t)a.C * 2, (size_t)a.R, st),
                           "cudaMemset2DAsync (empty contraction)");
    }
    return a.per_col_sb ? launch_impl<true>(a, st) : launch_impl<false>(a, st);
}

rlq_status check_device_errors(cudaStream_t st)
{
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return cuda_status(e, "cudaStreamSynchronize");
    unsigned long long word = 0;
    e = cudaMemcpyFromSymbolAsync(&word, g_rlq_error_word, sizeof word, 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return cuda_status(e, "reading the device error word");
    if (word == 0)
        return RLQ_OK;
    const unsigned long long zero = 0;
    e = cudaMemcpyToSymbolAsync(g_rlq_error_word, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return cuda_status(e, "clearing the device error word");
    const uint32_t code = (uint32_t)word, site = (uint32_t)(word >> 32);
    static const char *names[] = {"?", "TMA producer (stage free)", "MMA issuer (TMEM buffer free)",
                                  "MMA issuer (stage loaded)", "epilogue (partial ready)", "teardown", "drain"};
    const char *where = site == SITE_DIAG ? "diagnostic wait" : (site < 7 ? names[site] : "?");
    return fail((rlq_status)code, "device-side wait ran out at site %u (%s)", site, where);
}

rlq_status launch_diag_wait(int64_t timeout_us, cudaStream_t st)
{
    k_diag_wait<<<1, 32, 0, st>>>((uint64_t)timeout_us * 1000ull);
    return cuda_status(cudaGetLastError(), "diagnostic wait launch");
}

}  // namespace rlq
