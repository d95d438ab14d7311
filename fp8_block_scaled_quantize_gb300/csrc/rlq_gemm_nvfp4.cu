// NVFP4 weight-only GEMM on 5th-generation tensor cores (sm_103a).
//
// QeRL news article: the rollout runs the policy with NVFP4 weights (4-bit E2M1
// values, an FP8 E4M3 scale per block of 16 elements and an FP32 tensor scale)
// in FP4 x BF16 kernels: the activations stay bf16.  This kernel computes
//
//   Y[m, n] = bf16_RN( st * sum_k X[m, k] * (e2m1(q[n, k]) * e4m3(sb[n, k / 16])) )
//
// with X bf16 [M, K], q the packed E2M1 codes [N, K/2], sb the block-scale codes
// [N, K/16] and st the fp32 tensor scale, as rlq_quant_nvfp4 writes them.  An
// E2M1 value times an E4M3 value has at most 6 significant bits and lies in
// [2^-10, 2688] (or is 0), so it is exact in bf16: the weight tile is expanded to
// bf16 in shared memory and the contraction runs on tcgen05.mma kind::f16 (bf16 x
// bf16 -> fp32), accumulated in TMEM over the whole K; st is applied once in the
// epilogue.
//
// Roles (one persistent CTA per SM, 768 threads):
//   * warp 0 (one thread): TMA producer.  Per 64-element contraction stage the
//     128 x 64 bf16 X tile (128-byte swizzle) into a 3-stage ring; per 256-element
//     chunk the 256 rows x 128 bytes of packed codes (128-byte swizzle) and 256 x 16
//     bytes of block scales into a 2-slot raw ring.
//   * warp 1 (one thread): MMA issuer (4 x M=128, N=256, K=16 per stage into one
//     of two TMEM accumulators, 256 fp32 columns each; tiles alternate); warp 1
//     owns the 512 TMEM columns.
//   * warps 4-19 (512 threads, two per weight row, 32 elements each per stage):
//     converters.  Eight codes become eight bf16 values: magnitudes through two
//     byte tables (prmt), signs replicated from each nibble's top bit (prmt sign
//     mode), then one bf16x2 multiply by the block's scale per pair (exact); the
//     values are stored as 16-byte chunks in the layout of the MMA's shared-memory
//     descriptor (128-byte swizzle).
//   * warps 20-23 (128 threads, one TMEM lane each): epilogue, tcgen05.ld in 32-
//     column chunks, times st, rounded to bf16 and stored row by row.
// Work units: (tile, split) pairs.  With splits > 1 each unit sums a contiguous
// range of contraction stages (a whole number of raw chunks) and the epilogue
// writes st times its fp32 sum to plane `split` of the caller's workspace; the
// split-K reduction then adds the planes in split order and rounds to bf16.
// Every mbarrier wait is bounded as in the FP8 GEMM: a wait that runs out records
// an error word (this translation unit's) and raises the CTA's abort flag; the
// CTA drains its TMA copies, frees TMEM and exits.
//
// Batches of up to 4 tokens take k_gemv_nvfp4 (below) instead: the same exact
// weight values on the CUDA cores, streaming the codes with no shared-memory ring.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "rlq_internal.h"
#include "rlq_tc.cuh"

namespace rlq {
namespace {

constexpr int NV_BM = 128;                  // X rows per tile (TMEM lanes)
constexpr int NV_BN = 256;                  // weight rows (output columns) per tile (MMA N)
constexpr int NV_BK = 64;                   // contraction elements per stage (128 bytes of bf16)
constexpr int NV_CHUNK = 4 * NV_BK;         // contraction elements per raw chunk (128 bytes of codes)
constexpr int NV_STAGES = 3;
constexpr int NV_RAW_SLOTS = 2;
constexpr int NV_A_BYTES = NV_BM * NV_BK * 2;          // 16 KB
constexpr int NV_B_BYTES = NV_BN * NV_BK * 2;          // 32 KB
constexpr int NV_CODE_BYTES = NV_BN * (NV_CHUNK / 2);  // 32 KB
constexpr int NV_SCALE_BYTES = NV_BN * (NV_CHUNK / 16);  // 4 KB
constexpr int NV_THREADS = 768;
constexpr int NV_CONV_WARP0 = 4;
constexpr int NV_CONV_WARPS = 16;            // two threads per weight row, 32 elements each per stage
constexpr int NV_EPI_WARP0 = 20;             // four warps, one per TMEM lane quarter (warp % 4)
constexpr int NV_EPI_WARPS = 4;
constexpr int NV_TMEM_COLS = 512;
constexpr int NV_PREFETCH_CHUNKS = 3;        // weight chunks prefetched into L2 ahead of the ring
constexpr int NV_UMMA_K = 16;
// barriers: a_full, b_full, stage_empty per stage; raw_full, raw_empty per raw
// slot; tfull, tempty per accumulator; teardown
constexpr int NV_NUM_BARS = 3 * NV_STAGES + 2 * NV_RAW_SLOTS + 4 + 1;
constexpr int NV_OFF_A = 0;
constexpr int NV_OFF_B = NV_OFF_A + NV_STAGES * NV_A_BYTES;
constexpr int NV_OFF_CODES = NV_OFF_B + NV_STAGES * NV_B_BYTES;
constexpr int NV_OFF_SCALES = NV_OFF_CODES + NV_RAW_SLOTS * NV_CODE_BYTES;
constexpr int NV_OFF_BARS = NV_OFF_SCALES + NV_RAW_SLOTS * NV_SCALE_BYTES;
constexpr int NV_SMEM = 1024 /* alignment slack */ + NV_OFF_BARS + NV_NUM_BARS * 8 + 16;
static_assert(NV_SMEM <= 232448, "shared memory budget");
// tcgen05.mma kind::f16 instruction descriptor: D fp32 (bits 4-5 = 1), A and B
// bf16 (format 1 in bits 7-9 and 10-12), both K-major, N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
constexpr uint32_t NV_IDESC =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NV_BN >> 3) << 17) | ((uint32_t)(NV_BM >> 4) << 24);

struct NvParams {
    const float *st;  // tensor scale (device)
    uint16_t *y;
    int64_t ldy;
    float *ws;        // split partials [splits][M][N] fp32 (splits > 1 only)
    int M, N, K;
    int kstages;      // K / 64
    int m_tiles, num_tiles;
    int splits;       // contraction splits per tile (1: no split)
    int kps;          // stages per split, a multiple of 4 (one raw chunk = 4 stages)
    int num_units;    // num_tiles * splits
    uint64_t timeout_ns;
};

// Unit u -> tile (mt, nt) and its stage range [ks0, ks1).
struct NvUnit {
    int mt, nt, split, ks0, ks1;
};

__device__ __forceinline__ NvUnit nv_unit(const NvParams &p, int u)
{
    NvUnit w;
    const int t = u / p.splits;
    w.split = u - t * p.splits;
    w.mt = t % p.m_tiles;
    w.nt = t / p.m_tiles;
    w.ks0 = w.split * p.kps;
    w.ks1 = w.ks0 + p.kps < p.kstages ? w.ks0 + p.kps : p.kstages;
    return w;
}

__device__ __forceinline__ void nv_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(NV_IDESC), "r"(accumulate)
        : "memory");
}

// Prefetch a tensor-map box into L2 (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2(const CUtensorMap *map, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"((uint64_t)map), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// bf16 bit pattern of a (non-negative, finite) E4M3 block-scale code: exact, since
// E4M3 has 3 mantissa bits and a range inside bf16's.
__device__ __forceinline__ uint32_t e4m3_to_bf16_bits(uint32_t e)
{
    const uint32_t ex = (e >> 3) & 15u, m = e & 7u;
    const float v = ex == 0 ? (float)m * 0x1p-9f : __uint_as_float(((ex + 120u) << 23) | (m << 20));
    return __float_as_uint(v) >> 16;
}

// Eight E2M1 codes (one 32-bit word, element 0 in the lowest nibble) times one
// bf16 scale (in both halves of s2): four bf16x2 words, element 0 lowest.
// Magnitude bytes of 0, 0.5, 1, 1.5, 2, 3, 4, 6 in bf16: high bytes 00 3F 3F 3F 40
// 40 40 40, low bytes 00 00 80 C0 00 40 80 C0.  Signs: element 2k's sign is bit 7
// of byte k of (w << 4), element 2k+1's bit 7 of byte k of w; a prmt selector with
// bit 3 set replicates the selected byte's bit 7, so one prmt gives the sign bytes
// of four elements, which are merged into their high bytes before the interleave.
__device__ __forceinline__ uint4 e2m1x8_to_bf16(uint32_t w, uint32_t s2)
{
    constexpr uint32_t HI0 = 0x3F3F3F00u, HI1 = 0x40404040u;
    constexpr uint32_t LO0 = 0xC0800000u, LO1 = 0xC0804000u;
    const uint32_t m = w & 0x77777777u;  // magnitudes: prmt selectors in plain (not sign) mode
    const uint32_t m2 = m >> 16;
    const uint32_t we = w << 4;
    const uint32_t s03 = prmt(we, w, 0xD9C8u);  // signs of elements 0, 1, 2, 3 as 00 / FF bytes
    const uint32_t s47 = prmt(we, w, 0xFBEAu);  // elements 4 .. 7
    const uint32_t h03 = prmt(HI0, HI1, m) | (s03 & 0x80808080u);
    const uint32_t h47 = prmt(HI0, HI1, m2) | (s47 & 0x80808080u);
    const uint32_t l03 = prmt(LO0, LO1, m), l47 = prmt(LO0, LO1, m2);
    uint4 out;
    out.x = mul_bf16x2(prmt(l03, h03, 0x5140u), s2);  // elements 0, 1
    out.y = mul_bf16x2(prmt(l03, h03, 0x7362u), s2);  // elements 2, 3
    out.z = mul_bf16x2(prmt(l47, h47, 0x5140u), s2);
    out.w = mul_bf16x2(prmt(l47, h47, 0x7362u), s2);
    return out;
}

__global__ void __launch_bounds__(NV_THREADS, 1)
    k_gemm_nvfp4w(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmS, const NvParams p)
{
    pdl_begin();
    extern __shared__ uint8_t nv_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(nv_smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NV_OFF_BARS);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NV_NUM_BARS);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t s0 = smem_u32(smem);
    auto a_stage = [&](int s) { return s0 + (uint32_t)(NV_OFF_A + s * NV_A_BYTES); };
    auto b_stage = [&](int s) { return s0 + (uint32_t)(NV_OFF_B + s * NV_B_BYTES); };
    auto codes_slot = [&](int r) { return s0 + (uint32_t)(NV_OFF_CODES + r * NV_CODE_BYTES); };
    auto scales_slot = [&](int r) { return s0 + (uint32_t)(NV_OFF_SCALES + r * NV_SCALE_BYTES); };
    auto a_full = [&](int s) { return smem_u32(&bars[s]); };
    auto b_full = [&](int s) { return smem_u32(&bars[NV_STAGES + s]); };
    auto st_empty = [&](int s) { return smem_u32(&bars[2 * NV_STAGES + s]); };
    auto raw_full = [&](int r) { return smem_u32(&bars[3 * NV_STAGES + r]); };
    auto raw_empty = [&](int r) { return smem_u32(&bars[3 * NV_STAGES + NV_RAW_SLOTS + r]); };
    auto tfull = [&](int b) { return smem_u32(&bars[3 * NV_STAGES + 2 * NV_RAW_SLOTS + b]); };
    auto tempty = [&](int b) { return smem_u32(&bars[3 * NV_STAGES + 2 * NV_RAW_SLOTS + 2 + b]); };
    const uint32_t teardown = smem_u32(&bars[3 * NV_STAGES + 2 * NV_RAW_SLOTS + 4]);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NV_STAGES; ++s) {
            mbar_init(a_full(s), 1);
            mbar_init(b_full(s), NV_CONV_WARPS);
            mbar_init(st_empty(s), 1);
        }
        for (int r = 0; r < NV_RAW_SLOTS; ++r) {
            mbar_init(raw_full(r), 1);
            mbar_init(raw_empty(r), NV_CONV_WARPS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), NV_EPI_WARPS);
        }
        mbar_init(teardown, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(NV_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ---
        if (lane == 0) {
            int it = 0, rc = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
                const NvUnit w = nv_unit(p, u);
                const int mt = w.mt, nt = w.nt;
                for (int ks = w.ks0; ks < w.ks1; ++ks, ++it) {
                    if ((ks & 3) == 0) {
                        const int r = rc % NV_RAW_SLOTS;
                        if (!mbar_wait(raw_empty(r), ((uint32_t)(rc / NV_RAW_SLOTS) & 1u) ^ 1u, abort_flag,
                                       p.timeout_ns, SITE_PRODUCER_EMPTY)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(raw_full(r), NV_CODE_BYTES + NV_SCALE_BYTES);
                        tma_load_2d(codes_slot(r), &tmQ, raw_full(r), (ks >> 2) * (NV_CHUNK / 2), nt * NV_BN);
                        tma_load_2d(scales_slot(r), &tmS, raw_full(r), (ks >> 2) * (NV_CHUNK / 16), nt * NV_BN);
                        // start the weight stream a few chunks ahead into L2 (this unit's
                        // chunks only; the two ring slots alone hold too few bytes in flight
                        // to cover HBM latency)
                        const int ahead = (ks >> 2) + NV_PREFETCH_CHUNKS;
                        if (4 * ahead < w.ks1) {
                            tma_prefetch_l2(&tmQ, ahead * (NV_CHUNK / 2), nt * NV_BN);
                            tma_prefetch_l2(&tmS, ahead * (NV_CHUNK / 16), nt * NV_BN);
                        }
                        ++rc;
                    }
                    const int s = it % NV_STAGES;
                    if (!mbar_wait(st_empty(s), ((uint32_t)(it / NV_STAGES) & 1u) ^ 1u, abort_flag, p.timeout_ns,
                                   SITE_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(a_full(s), NV_A_BYTES);
                    tma_load_2d(a_stage(s), &tmX, a_full(s), ks * NV_BK, mt * NV_BM);
                }
            }
            // Once the MMA warp made its final commit, a normal run has consumed every
            // copy; a CTA that aborted waits (bounded) for the copies still in flight.
            volatile uint32_t never = 0;
            mbar_wait(teardown, 0, &never, p.timeout_ns, SITE_TEARDOWN);
            if (!ok || *abort_flag) {
                for (int j = it > NV_STAGES ? it - NV_STAGES : 0; j < it; ++j)
                    mbar_wait(a_full(j % NV_STAGES), (uint32_t)(j / NV_STAGES) & 1u, &never, 20000000ull, SITE_DRAIN);
                for (int j = rc > NV_RAW_SLOTS ? rc - NV_RAW_SLOTS : 0; j < rc; ++j)
                    mbar_wait(raw_full(j % NV_RAW_SLOTS), (uint32_t)(j / NV_RAW_SLOTS) & 1u, &never, 20000000ull,
                              SITE_DRAIN);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer ---
        if (lane == 0) {
            int it = 0, tc = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x, ++tc) {
                const NvUnit w = nv_unit(p, u);
                const int buf = tc & 1;
                if (!mbar_wait(tempty(buf), ((uint32_t)(tc >> 1) & 1u) ^ 1u, abort_flag, p.timeout_ns,
                               SITE_MMA_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                const uint32_t d = tmem_base + (uint32_t)(buf * NV_BN);
                for (int ks = w.ks0; ks < w.ks1; ++ks, ++it) {
                    const int s = it % NV_STAGES;
                    const uint32_t ph = (uint32_t)(it / NV_STAGES) & 1u;
                    if (!mbar_wait(a_full(s), ph, abort_flag, p.timeout_ns, SITE_MMA_FULL) ||
                        !mbar_wait(b_full(s), ph, abort_flag, p.timeout_ns, SITE_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(a_stage(s)), bd = sw128_desc(b_stage(s));
#pragma unroll
                    for (int j = 0; j < NV_BK / NV_UMMA_K; ++j)  // +32 bytes along K per MMA
                        nv_mma(d, ad + 2 * j, bd + 2 * j, (ks > w.ks0 || j > 0) ? 1u : 0u);
                    tc_commit(st_empty(s));
                    if (ks + 1 == w.ks1)
                        tc_commit(tfull(buf));
                }
            }
            // every MMA issued above has completed once this commit arrives
            tc_commit(teardown);
            volatile uint32_t never = 0;
            mbar_wait(teardown, 0, &never, 20000000ull, SITE_TEARDOWN);
        }
    } else if (warp >= NV_CONV_WARP0 && warp < NV_CONV_WARP0 + NV_CONV_WARPS) {
        // ------------------------------------------------- converters ---
        const int ct = threadIdx.x - NV_CONV_WARP0 * 32;  // 0..511
        const int row = ct >> 1;                           // weight row within the tile, 0..255
        const int half = ct & 1;                           // elements 32*half .. 32*half+31 of a stage
        const uint32_t sw = (uint32_t)(row & 7);
        int it = 0, rc = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
            const NvUnit w = nv_unit(p, u);
            for (int ks = w.ks0; ks < w.ks1; ++ks, ++it) {
                const int r = rc % NV_RAW_SLOTS;
                if ((ks & 3) == 0 &&
                    !__all_sync(0xFFFFFFFFu, mbar_wait(raw_full(r), (uint32_t)(rc / NV_RAW_SLOTS) & 1u, abort_flag,
                                                       p.timeout_ns, SITE_CONVERTER_EMPTY))) {
                    ok = false;
                    break;
                }
                const int s = it % NV_STAGES;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(st_empty(s), ((uint32_t)(it / NV_STAGES) & 1u) ^ 1u,
                                                       abort_flag, p.timeout_ns, SITE_CONVERTER_EMPTY))) {
                    ok = false;
                    break;
                }
                // this thread's 32 codes of the stage: 16-byte chunk 2q + half of the row's
                // 128-byte (swizzled) line in the raw slot, q = ks % 4; scale bytes 2 half,
                // 2 half + 1 of the row's four for the stage
                const int qk = ks & 3;
                uint4 c;
                {
                    const uint32_t a = codes_slot(r) + (uint32_t)(row * 128) +
                                       ((((uint32_t)(2 * qk + half)) ^ sw) << 4);
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(c.x), "=r"(c.y), "=r"(c.z), "=r"(c.w)
                                 : "r"(a));
                }
                uint32_t sc;
                asm volatile("ld.shared.u32 %0, [%1];" : "=r"(sc) : "r"(scales_slot(r) + (uint32_t)(row * 16 + qk * 4)));
                sc >>= 16 * half;
                const uint32_t sb0 = e4m3_to_bf16_bits(sc & 0xFFu), sb1 = e4m3_to_bf16_bits((sc >> 8) & 0xFFu);
                const uint32_t s0 = sb0 | (sb0 << 16), s1 = sb1 | (sb1 << 16);
                const uint32_t brow = b_stage(s) + (uint32_t)((row >> 3) * 1024 + (row & 7) * 128);
                const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {  // elements 8j .. 8j+7 of this half, block scale j / 2
                    const uint4 v = e2m1x8_to_bf16(w4[j], j < 2 ? s0 : s1);
                    const uint32_t chunk = (uint32_t)(4 * half + j);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(brow + ((chunk ^ sw) << 4)),
                                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                                 : "memory");
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> MMA reads
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(b_full(s));
                if (qk == 3 || ks + 1 == w.ks1) {  // the raw chunk is read out
                    if (lane == 0)
                        mbar_arrive(raw_empty(r));
                    ++rc;
                }
            }
        }
    } else if (warp >= NV_EPI_WARP0) {
        // --------------------------------------------------- epilogue ---
        const int q = warp & 3;  // TMEM lane quarter of this warp
        const int row = q * 32 + lane;
        const float st = *p.st;
        const float2 st2 = make_float2(st, st);
        int tc = 0;
        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++tc) {
            const NvUnit w = nv_unit(p, u);
            const int mt = w.mt, nt = w.nt;
            const int buf = tc & 1;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(tfull(buf), (uint32_t)(tc >> 1) & 1u, abort_flag, p.timeout_ns,
                                                   SITE_EPI_TMEM_FULL)))
                break;
            tc_fence_after();
            const int grow = mt * NV_BM + row;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * NV_BN);
            uint32_t r[32];
#pragma unroll 1
            for (int cc = 0; cc < NV_BN / 32; ++cc) {
                tmem_ld32_async(taddr + (uint32_t)(cc * 32), r);
                tmem_wait32(r);
                if (cc == NV_BN / 32 - 1) {  // the accumulator is read out
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(tempty(buf));
                }
                const int col = nt * NV_BN + cc * 32;
                if (p.splits > 1) {
                    if (grow < p.M && col < p.N) {
                        float4 *dst = reinterpret_cast<float4 *>(p.ws + ((int64_t)w.split * p.M + grow) * p.N + col);
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            const float2 a = __fmul2_rn(
                                make_float2(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1])), st2);
                            const float2 b = __fmul2_rn(
                                make_float2(__uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])), st2);
                            dst[v] = make_float4(a.x, a.y, b.x, b.y);
                        }
                    }
                } else if (grow < p.M && col < p.N) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.y + (int64_t)grow * p.ldy + col);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint32_t o[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float2 a = __fmul2_rn(make_float2(__uint_as_float(r[8 * v + 2 * u]),
                                                                    __uint_as_float(r[8 * v + 2 * u + 1])),
                                                        st2);
                            uint32_t d;
                            asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(a.y), "f"(a.x));
                            o[u] = d;
                        }
                        dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(NV_TMEM_COLS)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// Decode-sized batches (up to NV_GEMV_MAX_M tokens) on the CUDA cores.  With a
// handful of tokens the tensor-core kernel's time per weight stage does not
// depend on M and is several times the time to stream the weights from HBM.
// Here a warp owns R weight rows at a time and its lanes split the contraction:
// per step a lane takes a pair of 16-element blocks (16 bytes of codes and two
// scale bytes per row), U steps' loads issued together, so a warp reads 512
// contiguous bytes of each row per step.  Where the layer has too few rows to
// give every SM enough warps (down projections: long contractions, few output
// rows) a row group is shared by ks warps of a CTA, each taking every ks-th
// chunk of the contraction.  An E2M1 pair becomes an f16 pair (hardware
// conversion), its product with the block scale is taken in f16 (exact: at most
// 6 significant bits within [2^-10, 2688], f16 normals), widened to fp32 and
// multiplied with the bf16 activations by fp32 FMAs.  A lane's partial sums are
// added across its warp by a halving butterfly, the ks warps' sums in warp order
// through shared memory, st applied once and the result rounded to bf16.  The
// fp32 additions run in a fixed order, so results repeat bit for bit.

constexpr int NV_GEMV_MAX_M = 4;        // tokens the CUDA-core kernel takes
constexpr int NV_GEMV_SPLIT_MAX_M = 2;  // ... also when a split-K workspace is offered
constexpr int NV_GEMV_THREADS = 256;
constexpr int NV_GEMV_TASKS_PER_SM = 32;  // warp tasks per SM below which a row group is split across warps

// Eight E2M1 codes (element 2j in the low nibble of byte j) times a block scale
// held as an f16 pair: h[j] holds elements 2j (low half) and 2j + 1 (high half).
__device__ __forceinline__ void nv_e2m1x8_scaled(uint32_t codes, uint32_t scale2, uint32_t *h)
{
    asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
        "mov.b32 {c0, c1, c2, c3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, c0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, c1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, c2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, c3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(codes));
#pragma unroll
    for (int j = 0; j < 4; ++j)
        asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h[j]) : "r"(scale2));
}

// An E4M3 code as an f16 pair (both halves), exact.
__device__ __forceinline__ uint32_t nv_e4m3_f16x2(uint32_t code)
{
    uint32_t h;
    const uint16_t two = (uint16_t)(code | (code << 8));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(two));
    return h;
}

__device__ __forceinline__ float2 nv_f16x2_f32(uint32_t h)
{
    float lo, hi;
    asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, u;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
    return make_float2(lo, hi);
}

__device__ __forceinline__ uint4 nv_ld_stream16(const uint8_t *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t nv_ld_stream_u16(const uint8_t *p)
{
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// Halving butterfly over a warp: afterwards lane l holds the warp's sum of
// v[l >> (5 - log2 NVAL)] (the other lanes of that value's group hold it too).
template <int NVAL>
__device__ __forceinline__ float nv_warp_sums(float (&v)[NVAL], int lane)
{
    static_assert(NVAL >= 1 && NVAL <= 32 && (NVAL & (NVAL - 1)) == 0, "a power of two up to 32");
#pragma unroll
    for (int n = NVAL, off = 16; n > 1; n >>= 1, off >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
        }
    }
    float s = v[0];
#pragma unroll
    for (int off = 16 / NVAL; off > 0; off >>= 1)
        s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
    return s;
}

// MT tokens (M <= MT), R weight rows per warp, U steps of a pair of blocks per
// lane and chunk, MINB CTAs per SM (the register budget).  The CTA's 8 warps work on 8 / ks row groups at a time, ks
// warps per group, each taking every ks-th chunk of the group's contraction; the
// ks partial sums of a group are added through shared memory in warp order.
template <int MT, int R, int U, int MINB>
__global__ void __launch_bounds__(NV_GEMV_THREADS, MINB)
    k_gemv_nvfp4(const uint16_t *__restrict__ x, int64_t ldx, const uint8_t *__restrict__ wq, int64_t ldwq,
                 const uint8_t *__restrict__ wsb, int64_t ldwsb, const float *__restrict__ st,
                 uint16_t *__restrict__ y, int64_t ldy, int M, int N, int K, int ks)
{
    pdl_begin();
    constexpr int WARPS = NV_GEMV_THREADS / 32;
    constexpr int NVAL = R * MT;
    constexpr int LOG_NVAL = NVAL >= 32 ? 5 : NVAL >= 16 ? 4 : NVAL >= 8 ? 3 : NVAL >= 4 ? 2 : NVAL >= 2 ? 1 : 0;
    __shared__ float red[WARPS][NVAL];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gpc = WARPS / ks;                             // row groups per CTA round
    const int npairs = K >> 5;                              // pairs of 16-element blocks per row (K % 64 == 0)
    const int nchunks = (npairs + 32 * U - 1) / (32 * U);  // chunks per row group
    const int groups = (N + R - 1) / R;
    const float stv = *st;
    for (int round = blockIdx.x; round * gpc < groups; round += gridDim.x) {
        const int g = round * gpc + warp / ks;
        const int slice = warp % ks;
        float2 acc[R][MT];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m)
                acc[r][m] = make_float2(0.0f, 0.0f);
        if (g < groups) {
            const uint8_t *qrow[R];
            const uint8_t *srow[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int n = min(g * R + r, N - 1);  // (rows past N repeat the last row; their sums are not stored)
                qrow[r] = wq + (int64_t)n * ldwq;
                srow[r] = wsb + (int64_t)n * ldwsb;
            }
            for (int ci = slice; ci < nchunks; ci += ks) {
                uint4 c[U][R];
                uint32_t sc2[U][R];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int p = ci * 32 * U + 32 * u + lane;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        if (p < npairs) {
                            c[u][r] = nv_ld_stream16(qrow[r] + 16 * (int64_t)p);
                            sc2[u][r] = nv_ld_stream_u16(srow[r] + 2 * (int64_t)p);
                        } else {
                            c[u][r] = make_uint4(0, 0, 0, 0);
                            sc2[u][r] = 0;
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int p = ci * 32 * U + 32 * u + lane;
                    if (p >= npairs)
                        break;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {  // the two blocks of the pair
                        // the block's 16 activations per token as fp32 pairs (L1-allocating: every warp reads them)
                        float2 xf[MT][8];
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0;
                            if (m < M) {
                                const uint4 *xp =
                                    reinterpret_cast<const uint4 *>(x + (int64_t)m * ldx + 32 * (int64_t)p + 16 * j);
                                x0 = __ldg(xp);
                                x1 = __ldg(xp + 1);
                            }
                            const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                xf[m][i] =
                                    make_float2(__uint_as_float(xw[i] << 16), __uint_as_float(xw[i] & 0xFFFF0000u));
                        }
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t sc = nv_e4m3_f16x2((sc2[u][r] >> (8 * j)) & 0xFFu);
                            uint32_t h[8];
                            nv_e2m1x8_scaled(j ? c[u][r].z : c[u][r].x, sc, h);
                            nv_e2m1x8_scaled(j ? c[u][r].w : c[u][r].y, sc, h + 4);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float2 w = nv_f16x2_f32(h[i]);
#pragma unroll
                                for (int m = 0; m < MT; ++m)
                                    acc[r][m] = __ffma2_rn(w, xf[m][i], acc[r][m]);
                            }
                        }
                    }
                }
            }
        }
        float v[NVAL];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m)
                v[r * MT + m] = acc[r][m].x + acc[r][m].y;
        const float sum = nv_warp_sums<NVAL>(v, lane);
        if ((lane & ((32 >> LOG_NVAL) - 1)) == 0)
            red[warp][lane >> (5 - LOG_NVAL)] = sum;
        __syncthreads();
        if (threadIdx.x < gpc * NVAL) {
            const int gi = threadIdx.x / NVAL, idx = threadIdx.x - gi * NVAL;
            const int gg = round * gpc + gi;
            const int r = idx / MT, m = idx - (idx / MT) * MT;
            float t = red[gi * ks][idx];
            for (int k = 1; k < ks; ++k)
                t += red[gi * ks + k][idx];
            if (gg < groups && m < M && gg * R + r < N) {
                const float o = __fmul_rn(t, stv);
                uint16_t bits;
                asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(bits) : "f"(o));
                y[(int64_t)m * ldy + gg * R + r] = bits;
            }
        }
        __syncthreads();  // red is reused by the next round
    }
}

// ---------------------------------------------------------------- host ---

PFN_cuTensorMapEncodeTiled_v12000 nv_encode_fn()
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

rlq_status nv_map(CUtensorMap *map, CUtensorMapDataType dt, const void *base, int64_t inner, int64_t rows,
                  int64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz, const char *what)
{
    auto enc = nv_encode_fn();
    if (!enc)
        return fail(RLQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)pitch_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(RLQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d) for the %s", (int)r, what);
    return RLQ_OK;
}

uint64_t nv_wait_limit_ns()
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

// Split plan for an [M, N] output with K / 64 contraction stages on `sms` SMs.
// A unit costs about NV_UNIT_US to start plus NV_STAGE_US per stage (the
// converter ring's pace on one SM); units run in waves of `sms`; more than one
// split adds the reduction (launch plus the partials' traffic).  The plan takes
// the cheapest split count up to 16 whose partials fit ws_cap bytes (-1: no
// limit), with every split a whole number of raw chunks and none empty.
constexpr double NV_UNIT_US = 2.0, NV_STAGE_US = 0.65, NV_REDUCE_US = 2.0, NV_REDUCE_BYTES_PER_US = 4.0e6;

void nv_plan(int64_t M, int64_t N, int64_t K, int sms, int64_t ws_cap, int *splits_out, int *kps_out)
{
    const int64_t kstages = K / NV_BK;
    const int64_t tiles = ((M + NV_BM - 1) / NV_BM) * ((N + NV_BN - 1) / NV_BN);
    int best_s = 1;
    int64_t best_kps = kstages;
    double best = 1e300;
    for (int s = 1; s <= 16; ++s) {
        int64_t kps = (kstages + s - 1) / s;
        kps = (kps + 3) / 4 * 4;
        if (s > 1 && (kstages + kps - 1) / kps != s)
            continue;  // this count leaves a split empty: a smaller count covers it
        if (s > 1 && ws_cap >= 0 && (int64_t)s * M * N * 4 > ws_cap)
            break;
        const int64_t units = tiles * s;
        const int64_t waves = (units + sms - 1) / sms;
        double cost = (double)waves * (NV_UNIT_US + (double)(s == 1 ? kstages : kps) * NV_STAGE_US);
        if (s > 1)
            cost += NV_REDUCE_US + (double)(s + 1) * (double)M * (double)N * 4.0 / NV_REDUCE_BYTES_PER_US;
        if (cost < best) {
            best = cost;
            best_s = s;
            best_kps = s == 1 ? kstages : kps;
        }
    }
    *splits_out = best_s;
    *kps_out = (int)best_kps;
}

rlq_status nv_sms(int *sms)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
    return e == cudaSuccess ? RLQ_OK : cuda_status(e, "device query");
}

}  // namespace

rlq_status plan_nvfp4_splitk(int64_t M, int64_t N, int64_t K, int64_t ws_cap, int *splits, int64_t *ws_bytes)
{
    int sms = 0, kps = 0;
    const rlq_status rs = nv_sms(&sms);
    if (rs != RLQ_OK)
        return rs;
    int s = 1;
    if (M > NV_GEMV_SPLIT_MAX_M && N > 0 && K > 0)  // (one or two tokens run one pass on the CUDA cores)
        nv_plan(M, N, K, sms, ws_cap, &s, &kps);
    *splits = s;
    *ws_bytes = s > 1 ? (int64_t)s * M * N * 4 : 0;
    return RLQ_OK;
}

namespace {

template <int MT, int R, int U, int MINB>
rlq_status launch_gemv(const uint16_t *x, int64_t ldx, const uint8_t *wq, int64_t ldwq, const uint8_t *wsb,
                       int64_t ldwsb, const float *st, uint16_t *y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                       cudaStream_t stream)
{
    int sms = 0;
    const rlq_status rs = nv_sms(&sms);
    if (rs != RLQ_OK)
        return rs;
    constexpr int WARPS = NV_GEMV_THREADS / 32;
    const int64_t groups = (N + R - 1) / R;
    const int64_t nchunks = (K / 32 + 32 * U - 1) / (32 * U);
    // warps per row group: enough warp tasks to fill the GPU when the layer has few
    // output rows (a long contraction and few rows: down projections)
    int ks = 1;
    while (ks < WARPS && ks < nchunks && groups * ks < (int64_t)sms * NV_GEMV_TASKS_PER_SM)
        ks *= 2;
    const int64_t rounds = (groups + WARPS / ks - 1) / (WARPS / ks);
    int64_t grid = rounds < (int64_t)sms * 16 ? rounds : (int64_t)sms * 16;
    (void)launch_pdl(k_gemv_nvfp4<MT, R, U, MINB>, dim3((unsigned)grid), dim3(NV_GEMV_THREADS), 0, stream, x, ldx, wq,
                     ldwq, wsb, ldwsb, st, y, ldy, (int)M, (int)N, (int)K, ks);
    return cuda_status(cudaGetLastError(), "NVFP4 decode GEMM launch");
}

}  // namespace

rlq_status launch_gemm_nvfp4w(const uint16_t *x, int64_t ldx, const uint8_t *wq, int64_t ldwq, const uint8_t *wsb,
                              int64_t ldwsb, const float *st, uint16_t *y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                              void *workspace, int64_t workspace_bytes, cudaStream_t stream)
{
    // A handful of tokens: the CUDA-core kernel, one pass.  Three or four tokens
    // with a split-K workspace take the split tensor-core path instead (faster for
    // long contractions over few output rows, about even elsewhere).
    if (M <= NV_GEMV_SPLIT_MAX_M || (M <= NV_GEMV_MAX_M && workspace == nullptr)) {
        if (M == 1)
            return launch_gemv<1, 2, 4, 3>(x, ldx, wq, ldwq, wsb, ldwsb, st, y, ldy, M, N, K, stream);
        if (M == 2)
            return launch_gemv<2, 4, 2, 2>(x, ldx, wq, ldwq, wsb, ldwsb, st, y, ldy, M, N, K, stream);
        return launch_gemv<4, 4, 2, 2>(x, ldx, wq, ldwq, wsb, ldwsb, st, y, ldy, M, N, K, stream);
    }
    CUtensorMap tmX, tmQ, tmS;
    rlq_status rs = nv_map(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, ldx * 2, NV_BK, NV_BM,
                           CU_TENSOR_MAP_SWIZZLE_128B, "bf16 activations");
    if (rs != RLQ_OK)
        return rs;
    rs = nv_map(&tmQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, K / 2, N, ldwq, NV_CHUNK / 2, NV_BN,
                CU_TENSOR_MAP_SWIZZLE_128B, "packed E2M1 weight codes");
    if (rs != RLQ_OK)
        return rs;
    rs = nv_map(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT8, wsb, K / 16, N, ldwsb, NV_CHUNK / 16, NV_BN,
                CU_TENSOR_MAP_SWIZZLE_NONE, "E4M3 block scales");
    if (rs != RLQ_OK)
        return rs;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return cuda_status(e, "device query");
    static bool attr[64] = {};
    if (!attr[dev & 63]) {
        e = cudaFuncSetAttribute(k_gemm_nvfp4w, cudaFuncAttributeMaxDynamicSharedMemorySize, NV_SMEM);
        if (e != cudaSuccess)
            return cuda_status(e, "cudaFuncSetAttribute(max dynamic shared memory)");
        attr[dev & 63] = true;
    }
    NvParams p;
    p.st = st;
    p.y = y;
    p.ldy = ldy;
    p.ws = static_cast<float *>(workspace);
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.kstages = (int)(K / NV_BK);
    p.m_tiles = (int)((M + NV_BM - 1) / NV_BM);
    p.num_tiles = p.m_tiles * (int)((N + NV_BN - 1) / NV_BN);
    p.splits = 1;
    p.kps = p.kstages;
    if (workspace)
        nv_plan(M, N, K, sms, workspace_bytes, &p.splits, &p.kps);
    p.num_units = p.num_tiles * p.splits;
    p.timeout_ns = nv_wait_limit_ns();
    const int grid = p.num_units < sms ? p.num_units : sms;
    (void)launch_pdl(k_gemm_nvfp4w, dim3(grid), dim3(NV_THREADS), NV_SMEM, stream, tmX, tmQ, tmS, p);
    e = cudaGetLastError();
    if (e != cudaSuccess || p.splits == 1)
        return cuda_status(e, "NVFP4 GEMM launch");
    return launch_splitk_reduce(p.ws, p.splits, M, N, y, ldy, sms, stream);
}

cudaError_t take_nvfp4_error_word(cudaStream_t st, unsigned long long *word) { return take_error_word(st, word); }

}  // namespace rlq
