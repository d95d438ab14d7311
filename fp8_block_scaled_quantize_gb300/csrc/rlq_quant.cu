// Fine-grained FP8 E4M3 quantizers and the UAQ fold (sm_103a).
//
// Jet-RL notes, section "细粒度 GEMM 量化方案" (Fig. 6): activations and
// gradients use 1x128 per-group scales, weights 128x128 per-block scales, and
// the WGrad operand grouped 128x1 is produced fused with the 1x128 one.
// QuRL notes, 关键设计 §1: the UAQ fold W/s (per column) and s*X (per row).
//
// Per group: amax = max |x|; s = fl32(amax / 448), or 1 when amax == 0;
// code = RN-even satfinite E4M3 of fl32(x / s).
//
// All kernels are HBM-bound streaming kernels: 16-byte loads of 8 bf16 per
// lane, a group of 128 spread over 16 lanes (warp-shuffle amax), packed code
// stores.  The per-element quotient x / s uses the group's reciprocal
// r = RN(1/s) plus one FMA residual correction (1.5 packed fp32x2 ops per
// element) instead of an IEEE division sequence.  For bf16 x with |x| <= amax and
// s = fl32(amax/448) this equals IEEE fp32 division wherever the E4M3 code can
// depend on it (every (x, amax) bf16 pair was enumerated); groups with a scale
// below 2^-100 are pre-scaled by 2^64, exactly, so that 1/s stays finite.
// Build without fast-math: subnormal inputs and scales are honoured.
#include <cuda_runtime.h>

#include "rlq_internal.h"

namespace rlq {
namespace {

constexpr int GRP = 128;

__device__ __forceinline__ uint4 ld_stream(const uint16_t *p)
{
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = bf_lo(w[i]);
        f[2 * i + 1] = bf_hi(w[i]);
    }
}

// Two E4M3 codes, RN-even with saturation to +-448: `lo` in bits 0..7.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// Division context of one group (or of a pair of groups, one per lane of a
// packed fp32x2 operation).
struct Quot {
    float f;   // exact pre-scale: 1, or 2^64 for scales below 2^-100
    float sd;  // s * f (exact)
    float r;   // RN(1 / sd)
};

__device__ __forceinline__ float group_scale(float amax)
{
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

__device__ __forceinline__ Quot make_quot(float s)
{
    Quot q;
    q.f = (s < 0x1p-100f) ? 0x1p64f : 1.0f;
    q.sd = __fmul_rn(s, q.f);
    q.r = __frcp_rn(q.sd);
    return q;
}


// fl32(x / s) for two elements at once, as described at the top of this file:
// q0 = x*r, e = x - q0*s (one FMA, rounded toward -inf), q1 = q0 + e*r.  The
// downward-rounded residual keeps the sign of a zero quotient (x = -0 gives -0);
// every (x, amax) bf16 pair was enumerated: q1 equals the IEEE quotient wherever
// the E4M3 code depends on it, sign included.  Each packed operation rounds
// each lane exactly as its scalar IEEE counterpart does.  kPrescale applies the
// exact 2^64 pre-scale of groups whose scale is below 2^-100.
template <bool kPrescale>
__device__ __forceinline__ float2 quot2(float2 x, float2 f, float2 r, float2 nsd)
{
    const float2 xs = kPrescale ? __fmul2_rn(x, f) : x;
    const float2 q0 = __fmul2_rn(xs, r);
    const float2 e = __ffma2_rd(q0, nsd, xs);  // xs - q0 * sd
    return __ffma2_rn(e, r, q0);
}

// Codes of 8 consecutive elements of one group, element 0 in the lowest byte.
template <bool kPrescale>
__device__ __forceinline__ uint2 encode8_t(const float (&v)[8], const Quot &c)
{
    const float2 f = make_float2(c.f, c.f), r = make_float2(c.r, c.r), nsd = make_float2(-c.sd, -c.sd);
    const float2 a = quot2<kPrescale>(make_float2(v[0], v[1]), f, r, nsd);
    const float2 b = quot2<kPrescale>(make_float2(v[2], v[3]), f, r, nsd);
    const float2 d = quot2<kPrescale>(make_float2(v[4], v[5]), f, r, nsd);
    const float2 g = quot2<kPrescale>(make_float2(v[6], v[7]), f, r, nsd);
    uint2 out;
    out.x = e4m3x2(a.x, a.y) | (e4m3x2(b.x, b.y) << 16);
    out.y = e4m3x2(d.x, d.y) | (e4m3x2(g.x, g.y) << 16);
    return out;
}

__device__ __forceinline__ uint2 encode8(const float (&v)[8], const Quot &c)
{
    return c.f == 1.0f ? encode8_t<false>(v, c) : encode8_t<true>(v, c);
}

// Codes of 32 rows of two adjacent columns (packed lanes: even, odd column),
// read from the staged tile; the words hold 4 rows each.
template <bool kPrescale>
__device__ __forceinline__ void encode_cols(const uint32_t *col, int rq, int tp2, float2 pf, float2 pr, float2 pn,
                                            uint32_t (&e)[8], uint32_t (&o)[8])
{
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float2 qq[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t wv = col[(rq * 32 + 4 * j + u) * tp2];
            qq[u] = quot2<kPrescale>(make_float2(bf_lo(wv), bf_hi(wv)), pf, pr, pn);
        }
        e[j] = e4m3x2(qq[0].x, qq[1].x) | (e4m3x2(qq[2].x, qq[3].x) << 16);
        o[j] = e4m3x2(qq[0].y, qq[1].y) | (e4m3x2(qq[2].y, qq[3].y) << 16);
    }
}

__device__ __forceinline__ float amax8(const float (&f)[8])
{
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        a = fmaxf(a, fabsf(f[i]));
    return a;
}

// amax over the 16 lanes of a half-warp (all 32 lanes must call).
__device__ __forceinline__ float halfwarp_max(float a)
{
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1)
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
    return a;
}

// One 1x128 group held by a half-warp (8 values per lane): quantize and store.
__device__ __forceinline__ void row_group(const uint4 &v, bool valid, int64_t m, int64_t kb, int l16,
                                          uint8_t *__restrict__ q, int64_t ldq, float *__restrict__ s,
                                          int64_t lds)
{
    float f[8];
    unpack8(v, f);
    const float amax = halfwarp_max(amax8(f));
    const float sc = group_scale(amax);
    const Quot c = make_quot(sc);
    const uint2 codes = encode8(f, c);
    if (valid) {
        *reinterpret_cast<uint2 *>(q + m * ldq + kb * GRP + l16 * 8) = codes;
        if (l16 == 0)
            s[kb * lds + m] = sc;
    }
}

// ---------------------------------------------------------------------------
// 1x128 row-wise: each half-warp takes a group; a warp owns two consecutive
// groups per slot and two slots per iteration (four 16-byte loads in flight
// per lane pair).  Group g = m * KB + kb, advanced incrementally.
__global__ void __launch_bounds__(256) k_quant_rows(const uint16_t *__restrict__ x, int64_t M, int KB,
                                                    int64_t ldx, uint8_t *__restrict__ q, int64_t ldq,
                                                    float *__restrict__ s, int64_t lds)
{
    const int lane = threadIdx.x & 31, half = lane >> 4, l16 = lane & 15;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t G = M * KB;
    const int64_t step = 2 * nwarps;  // groups between the two slots
    const int64_t dm = step / KB;
    const int dkb = (int)(step % KB);
    const int64_t g0 = 2 * warp + half;
    int64_t m = g0 / KB;
    int kb = (int)(g0 % KB);
    // the next iteration's two groups are loaded before this iteration's are quantized
    const uint4 zero = make_uint4(0, 0, 0, 0);
    auto second = [&](int64_t mm, int kk, int64_t &m1, int &kb1) {
        m1 = mm + dm;
        kb1 = kk + dkb;
        if (kb1 >= KB) {
            kb1 -= KB;
            ++m1;
        }
    };
    int64_t m1;
    int kb1;
    second(m, kb, m1, kb1);
    uint4 a = m < M ? ld_stream(x + m * ldx + (int64_t)kb * GRP + l16 * 8) : zero;
    uint4 b = m1 < M ? ld_stream(x + m1 * ldx + (int64_t)kb1 * GRP + l16 * 8) : zero;
    for (int64_t base = 2 * warp; base < G; base += 2 * step) {
        int64_t mn = m1 + dm;
        int kbn = kb1 + dkb;
        if (kbn >= KB) {
            kbn -= KB;
            ++mn;
        }
        int64_t mn1;
        int kbn1;
        second(mn, kbn, mn1, kbn1);
        const uint4 an = mn < M ? ld_stream(x + mn * ldx + (int64_t)kbn * GRP + l16 * 8) : zero;
        const uint4 bn = mn1 < M ? ld_stream(x + mn1 * ldx + (int64_t)kbn1 * GRP + l16 * 8) : zero;
        row_group(a, m < M, m, kb, l16, q, ldq, s, lds);
        row_group(b, m1 < M, m1, kb1, l16, q, ldq, s, lds);
        a = an;
        b = bn;
        m = mn;
        kb = kbn;
        m1 = mn1;
        kb1 = kbn1;
    }
}

// ---------------------------------------------------------------------------
// Fused 1x128 + 128x1 on a 128x128 tile: one read of x.  Row groups are
// quantized straight from registers; the tile is staged in shared memory
// (row pitch 272 B) for the column groups, whose codes are written transposed.
constexpr int TP = GRP + 8;  // staging row pitch in bf16 elements

__global__ void __launch_bounds__(256, 4) k_quant_dual(const uint16_t *__restrict__ x, int64_t M, int64_t ldx,
                                                    uint8_t *__restrict__ q, int64_t ldq,
                                                    float *__restrict__ s, int64_t lds,
                                                    uint8_t *__restrict__ qT, int64_t ldqT,
                                                    float *__restrict__ sc, int64_t ldsc, int64_t MB)
{
    __shared__ __align__(16) uint16_t tile[GRP * TP];
    __shared__ float cam[4][GRP];  // column maxima of the four row quarters
    const int t = threadIdx.x, lane = t & 31, half = lane >> 4, l16 = lane & 15, warp = t >> 5;
    const int hw16 = warp * 2 + half;  // 0..15
    const int64_t kb = blockIdx.x;
    const int c2 = t & 63, rq = t >> 6;

    for (int64_t mb = blockIdx.y; mb < MB; mb += gridDim.y) {
        const int64_t m0 = mb * GRP;
        const int rows = (int)((M - m0) < GRP ? (M - m0) : GRP);

        // ---- row pass: half-warp hw16 owns rows hw16 + 16 i; lane l16 owns
        // columns 8 l16 .. 8 l16 + 7.  Rows beyond M read as zero.
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = hw16 + 16 * i;
            v[i] = (r < rows) ? ld_stream(x + (m0 + r) * ldx + kb * GRP + l16 * 8) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = hw16 + 16 * i;
            float f[8];
            unpack8(v[i], f);
            const float amax = halfwarp_max(amax8(f));
            const float scl = group_scale(amax);
            const Quot c = make_quot(scl);
            const uint2 codes = encode8(f, c);
            if (r < rows) {
                *reinterpret_cast<uint2 *>(q + (m0 + r) * ldq + kb * GRP + l16 * 8) = codes;
                if (l16 == 0)
                    s[kb * lds + m0 + r] = scl;
            }
            *reinterpret_cast<uint4 *>(&tile[r * TP + l16 * 8]) = v[i];
        }
        __syncthreads();

        // ---- column pass: thread owns columns 2*c2, 2*c2+1 over rows rq*32 .. +31;
        // first the column maxima (four row quarters combined through smem)
        const uint32_t *col = reinterpret_cast<const uint32_t *>(tile) + c2;
        float a0 = 0.0f, a1 = 0.0f;
#pragma unroll 8
        for (int rr = 0; rr < 32; ++rr) {
            const uint32_t wv = col[(rq * 32 + rr) * (TP / 2)];
            a0 = fmaxf(a0, fabsf(bf_lo(wv)));
            a1 = fmaxf(a1, fabsf(bf_hi(wv)));
        }
        cam[rq][2 * c2] = a0;
        cam[rq][2 * c2 + 1] = a1;
        __syncthreads();
        a0 = fmaxf(fmaxf(cam[0][2 * c2], cam[1][2 * c2]), fmaxf(cam[2][2 * c2], cam[3][2 * c2]));
        a1 = fmaxf(fmaxf(cam[0][2 * c2 + 1], cam[1][2 * c2 + 1]), fmaxf(cam[2][2 * c2 + 1], cam[3][2 * c2 + 1]));
        const float s0 = group_scale(a0), s1 = group_scale(a1);
        const Quot c0 = make_quot(s0), c1 = make_quot(s1);
        // one packed lane per column: (even column, odd column) of the same row
        const float2 pf = make_float2(c0.f, c1.f), pr = make_float2(c0.r, c1.r), pn = make_float2(-c0.sd, -c1.sd);
        const bool fast = (c0.f == 1.0f) && (c1.f == 1.0f);
        uint32_t e[8], o[8];  // 32 codes of each column, 4 per word
        if (fast)
            encode_cols<false>(col, rq, TP / 2, pf, pr, pn, e, o);
        else
            encode_cols<true>(col, rq, TP / 2, pf, pr, pn, e, o);
        const int64_t k = kb * GRP + 2 * c2;
        const int r0 = rq * 32;
        uint8_t *d0 = qT + k * ldqT + m0 + r0;
        uint8_t *d1 = d0 + ldqT;
        if (r0 + 32 <= rows) {
            reinterpret_cast<uint4 *>(d0)[0] = make_uint4(e[0], e[1], e[2], e[3]);
            reinterpret_cast<uint4 *>(d0)[1] = make_uint4(e[4], e[5], e[6], e[7]);
            reinterpret_cast<uint4 *>(d1)[0] = make_uint4(o[0], o[1], o[2], o[3]);
            reinterpret_cast<uint4 *>(d1)[1] = make_uint4(o[4], o[5], o[6], o[7]);
        } else {
#pragma unroll
            for (int rr = 0; rr < 32; ++rr) {
                if (r0 + rr < rows) {
                    d0[rr] = (uint8_t)(e[rr >> 2] >> (8 * (rr & 3)));
                    d1[rr] = (uint8_t)(o[rr >> 2] >> (8 * (rr & 3)));
                }
            }
        }
        if (rq == 0) {
            sc[mb * ldsc + k] = s0;
            sc[mb * ldsc + k + 1] = s1;
        }
        __syncthreads();  // tile and cam are reused by the next mb
    }
}

// ---------------------------------------------------------------------------
// 128x128 weight blocks: one CTA per block.  The block is read once (16-byte
// loads), its amax reduced while the raw values are stashed in shared memory,
// then quantized from shared memory; the same buffer is reused to transpose the
// codes for the optional [K,N] copy.  32 KB of shared memory and few registers
// per thread keep several blocks in flight per SM.
constexpr int CTP = GRP + 16;  // code staging row pitch (bytes) for the transposed copy

__global__ void __launch_bounds__(256, 4) k_quant_weight(const uint16_t *__restrict__ w, int64_t ldw,
                                                         uint8_t *__restrict__ q, int64_t ldq,
                                                         float *__restrict__ s, int64_t lds,
                                                         uint8_t *__restrict__ qT, int64_t ldqT, int64_t NB)
{
    __shared__ __align__(16) uint16_t wt[GRP * GRP];  // raw block, row pitch 256 bytes
    __shared__ float red[8];
    uint8_t *ct = reinterpret_cast<uint8_t *>(wt);     // code staging, reuses the raw buffer
    const int t = threadIdx.x, lane = t & 31, half = lane >> 4, l16 = lane & 15, warp = t >> 5;
    const int hw16 = warp * 2 + half;
    const int64_t kb = blockIdx.x;

    for (int64_t nb = blockIdx.y; nb < NB; nb += gridDim.y) {
        const int64_t n0 = nb * GRP;
        // ---- read, amax, stash
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = ld_stream(w + (n0 + hw16 + 16 * i) * ldw + kb * GRP + l16 * 8);
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float f[8];
            unpack8(v[i], f);
            a = fmaxf(a, amax8(f));
            *reinterpret_cast<uint4 *>(&wt[(hw16 + 16 * i) * GRP + l16 * 8]) = v[i];
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
        if (lane == 0)
            red[warp] = a;
        __syncthreads();
        a = red[0];
#pragma unroll
        for (int i = 1; i < 8; ++i)
            a = fmaxf(a, red[i]);
        const float sc = group_scale(a);
        const Quot c = make_quot(sc);
        if (t == 0)
            s[nb * lds + kb] = sc;
        // ---- quantize from shared memory
        uint2 cd[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = hw16 + 16 * i;
            float f[8];
            unpack8(*reinterpret_cast<const uint4 *>(&wt[r * GRP + l16 * 8]), f);
            cd[i] = encode8(f, c);
            *reinterpret_cast<uint2 *>(q + (n0 + r) * ldq + kb * GRP + l16 * 8) = cd[i];
        }
        if (qT) {
            __syncthreads();  // the raw block is no longer read: reuse it for the codes
#pragma unroll
            for (int i = 0; i < 8; ++i)
                *reinterpret_cast<uint2 *>(&ct[(hw16 + 16 * i) * CTP + l16 * 8]) = cd[i];
            __syncthreads();
            // thread -> output row k0 + cc of qT, 64 consecutive n (rows nh*64 .. +63 of the block)
            const int cc = t >> 1, nh = t & 1;
            uint32_t wv[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int r = nh * 64 + 4 * j;
                wv[j] = (uint32_t)ct[(r + 0) * CTP + cc] | ((uint32_t)ct[(r + 1) * CTP + cc] << 8) |
                        ((uint32_t)ct[(r + 2) * CTP + cc] << 16) | ((uint32_t)ct[(r + 3) * CTP + cc] << 24);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(qT + (kb * GRP + cc) * ldqT + n0 + nh * 64);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                dst[j] = make_uint4(wv[4 * j], wv[4 * j + 1], wv[4 * j + 2], wv[4 * j + 3]);
        }
        __syncthreads();  // wt / red are reused by the next block
    }
}

// ---------------------------------------------------------------------------
// UAQ fold, in place: divide (w) or multiply (prev) column k by s[k] in fp32,
// round to bf16.  8 elements per thread and vector; each thread handles FOLD_ROWS
// rows per iteration with all their loads issued first (bytes in flight hide
// the memory latency); row groups over blockIdx.y (grid-stride).
constexpr int FOLD_ROWS = 4;

template <bool kDivide>
__global__ void __launch_bounds__(256) k_uaq_fold(uint16_t *__restrict__ a, int64_t rows, int64_t K8,
                                                  int64_t lda, const float *__restrict__ s)
{
    const int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= K8)
        return;
    const float4 s0 = __ldg(reinterpret_cast<const float4 *>(s) + 2 * v);
    const float4 s1 = __ldg(reinterpret_cast<const float4 *>(s) + 2 * v + 1);
    const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    for (int64_t r0 = (int64_t)blockIdx.y * FOLD_ROWS; r0 < rows; r0 += (int64_t)gridDim.y * FOLD_ROWS) {
        uint4 in[FOLD_ROWS];
#pragma unroll
        for (int i = 0; i < FOLD_ROWS; ++i)
            if (r0 + i < rows)
                in[i] = *(reinterpret_cast<const uint4 *>(a + (r0 + i) * lda) + v);
#pragma unroll
        for (int i = 0; i < FOLD_ROWS; ++i) {
            if (r0 + i >= rows)
                break;
            float f[8];
            unpack8(in[i], f);
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float x0 = kDivide ? __fdiv_rn(f[2 * j], sv[2 * j]) : __fmul_rn(f[2 * j], sv[2 * j]);
                const float x1 = kDivide ? __fdiv_rn(f[2 * j + 1], sv[2 * j + 1]) : __fmul_rn(f[2 * j + 1], sv[2 * j + 1]);
                uint32_t pk;
                asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(pk) : "f"(x1), "f"(x0));
                o[j] = pk;
            }
            *(reinterpret_cast<uint4 *>(a + (r0 + i) * lda) + v) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    return n;
}

}  // namespace

cudaError_t launch_quant_rows(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, int64_t ldq,
                              float *s, int64_t lds, cudaStream_t st)
{
    const int KB = (int)(K / GRP);
    const int64_t groups = M * KB;
    const int64_t warps_needed = (groups + 3) / 4;  // 4 groups per warp per iteration
    int64_t blocks = (warps_needed + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    k_quant_rows<<<(unsigned)blocks, 256, 0, st>>>(x, M, KB, ldx, q, ldq, s, lds);
    return cudaGetLastError();
}

cudaError_t launch_quant_dual(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, int64_t ldq,
                              float *s, int64_t lds, uint8_t *qT, int64_t ldqT, float *sc, int64_t ldsc,
                              cudaStream_t st)
{
    const int64_t MB = (M + GRP - 1) / GRP;
    const dim3 grid((unsigned)(K / GRP), (unsigned)(MB < 65535 ? MB : 65535));
    k_quant_dual<<<grid, 256, 0, st>>>(x, M, ldx, q, ldq, s, lds, qT, ldqT, sc, ldsc, MB);
    return cudaGetLastError();
}

cudaError_t launch_quant_weight(const uint16_t *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq,
                                float *s, int64_t lds, uint8_t *qT, int64_t ldqT, cudaStream_t st)
{
    const int64_t NB = N / GRP;
    const dim3 grid((unsigned)(K / GRP), (unsigned)(NB < 65535 ? NB : 65535));
    k_quant_weight<<<grid, 256, 0, st>>>(w, ldw, q, ldq, s, lds, qT, ldqT, NB);
    return cudaGetLastError();
}

cudaError_t launch_uaq_fold(uint16_t *w, int64_t N, int64_t K, int64_t ldw, const float *s, uint16_t *prev,
                            int64_t R, int64_t ldp, cudaStream_t st)
{
    const int64_t K8 = K / 8;
    const unsigned gx = (unsigned)((K8 + 255) / 256);
    auto gy = [](int64_t rows) {
        const int64_t g = (rows + FOLD_ROWS - 1) / FOLD_ROWS;
        return (unsigned)(g < 65535 ? g : 65535);
    };
    if (N > 0) {
        k_uaq_fold<true><<<dim3(gx, gy(N)), 256, 0, st>>>(w, N, K8, ldw, s);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    if (prev && R > 0) {
        k_uaq_fold<false><<<dim3(gx, gy(R)), 256, 0, st>>>(prev, R, K8, ldp, s);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace rlq
