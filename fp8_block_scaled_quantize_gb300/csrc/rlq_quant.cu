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
// All kernels are HBM-bound streaming kernels with vector loads and packed
// code stores; a group's scale is computed once (not by every lane that holds
// part of the group) and handed to the encoding lanes by shuffle or through
// shared memory.  The per-element quotient x / s uses the group's reciprocal
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

// Loads of a kernel's input, which no thread of the kernel writes: the read-only
// path without L1 allocation (measured 2% faster for the dual quantizer than an
// evict-first streaming load, the same elsewhere).
__device__ __forceinline__ uint4 ld_stream(const uint16_t *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
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

__device__ __forceinline__ uint32_t pack_bf16x2(float2 v)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(v.y), "f"(v.x));
    return d;
}

// RMSNorm of 8 consecutive bf16 elements of one row with that row's r and the
// matching 8 norm weights: x = bf16_RN(fl32(fl32(h * r) * gamma)), each product
// rounded on its own (packed fp32 multiplies round each lane as the scalar op).
__device__ __forceinline__ uint4 norm8(const uint4 &v, float r, const uint4 &g)
{
    const float2 r2 = make_float2(r, r);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w}, gw[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 hr = __fmul2_rn(make_float2(bf_lo(w[i]), bf_hi(w[i])), r2);
        o[i] = pack_bf16x2(__fmul2_rn(hr, make_float2(bf_lo(gw[i]), bf_hi(gw[i]))));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
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
// q0 = x*r, e = x - q0*s (one FMA, rounded toward -inf), q1 = q0 + e*r.  This is
// the quotient-correction step of Markstein's division (P. Markstein, IBM J. Res.
// Dev. 34(1), 1990; "IA-64 and Elementary Functions", 2000): with an FMA the
// residual x - q0*s is exact, and one multiply-add of it by the reciprocal moves
// q0 to the correctly rounded quotient under conditions that the enumeration
// below checks for this input domain.  The
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

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t babs2(uint32_t a) { return a & 0x7FFF7FFFu; }

// amax of a packed pair of candidates; an all-NaN group reads as 0, as a
// running fmaxf from 0 would give.
__device__ __forceinline__ float bmax_final(uint32_t p) { return fmaxf(fmaxf(bf_lo(p), bf_hi(p)), 0.0f); }

// max(|a|, |b|) per half, with the sign of the product (only the magnitude is used)
__device__ __forceinline__ uint32_t bmaxabs2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// ---------------------------------------------------------------------------
// 1x128 row-wise, one warp per row segment.  Rows are cut into `segs` segments
// of 256 nv elements (nv <= QR_NV) and a warp takes a whole segment, all of its
// 16-byte loads in flight before any group is quantized.  Load i of lane l holds
// elements 256 i + 8 l .. + 7 of the segment, so half-warp h holds group 2 i + h
// in load i.  The QR_NV group maxima of a half-warp are reduced in one transposed
// exchange (each step hands half of the remaining groups to the partner lane),
// after which lane pair (2 i, 2 i + 1) of the half holds the amax of its group in
// load i and computes that group's scale once: the maxima, the division and the
// reciprocal cost a few instructions per segment rather than per pair of groups.
// The encoding lanes fetch (r, s[, f]) by shuffle.  Elements at or past K read as
// zero and write nothing.  kNorm: x is a hidden state h, normalised on the fly
// (rmsnorm row factor rstd[m], weight gamma[k]) before it is quantized.
constexpr int QR_NV = 8;

template <bool kPrescale>
__device__ __forceinline__ void rows_seg_codes(const uint4 (&v)[QR_NV], const Quot &own, int lane, int nv,
                                               int64_t kleft, uint8_t *__restrict__ qp)
{
    const int src0 = lane & 16;
#pragma unroll
    for (int i = 0; i < QR_NV; ++i) {
        if (i >= nv)
            break;
        Quot c;
        c.r = __shfl_sync(0xFFFFFFFFu, own.r, src0 + 2 * i);
        c.sd = __shfl_sync(0xFFFFFFFFu, own.sd, src0 + 2 * i);
        c.f = kPrescale ? __shfl_sync(0xFFFFFFFFu, own.f, src0 + 2 * i) : 1.0f;
        float f[8];
        unpack8(v[i], f);
        const uint2 codes = encode8_t<kPrescale>(f, c);
        if (256 * i < kleft)
            *reinterpret_cast<uint2 *>(qp + 256 * i) = codes;
    }
}

template <bool kNorm>
__global__ void __launch_bounds__(256, 4) k_quant_rows_seg(const uint16_t *__restrict__ x, int64_t M, int64_t K,
                                                        int segs, int nv, int64_t ldx, uint8_t *__restrict__ q,
                                                        int64_t ldq, float *__restrict__ s, int64_t lds,
                                                        const float *__restrict__ rstd,
                                                        const uint16_t *__restrict__ gamma)
{
    pdl_begin();
    static_assert(QR_NV == 8, "the exchange below reduces eight groups per half-warp");
    const int lane = threadIdx.x & 31, half = lane >> 4, l16 = lane & 15;
    const bool b3 = l16 & 8, b2 = l16 & 4, b1 = l16 & 2;
    const int jo = l16 >> 1;  // the load whose group this lane's scale belongs to
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t items = M * segs;
    for (int64_t it = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < items; it += nwarps) {
        const int64_t m = it / segs;
        const int64_t k0 = (it - m * segs) * 256 * nv;  // first element of the segment
        const int64_t kleft = K - k0 - 8 * lane;        // load i is in range iff 256 i < kleft
        const uint16_t *xp = x + m * ldx + k0 + 8 * lane;
        uint4 v[QR_NV];
#pragma unroll
        for (int i = 0; i < QR_NV; ++i)
            v[i] = (i < nv && 256 * i < kleft) ? ld_stream(xp + 256 * i) : make_uint4(0, 0, 0, 0);
        if (kNorm) {
            const float r = rstd[m];
            const uint16_t *gp = gamma + k0 + 8 * lane;
#pragma unroll
            for (int i = 0; i < QR_NV; ++i)
                if (i < nv && 256 * i < kleft)
                    v[i] = norm8(v[i], r, *reinterpret_cast<const uint4 *>(gp + 256 * i));
        }
        uint32_t pm[QR_NV], p1[4], p2[2];
#pragma unroll
        for (int i = 0; i < QR_NV; ++i)
            pm[i] = bmaxabs2(bmaxabs2(v[i].x, v[i].y), bmaxabs2(v[i].z, v[i].w));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t keep = b3 ? pm[k + 4] : pm[k], send = b3 ? pm[k] : pm[k + 4];
            p1[k] = bmaxabs2(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 8));
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint32_t keep = b2 ? p1[k + 2] : p1[k], send = b2 ? p1[k] : p1[k + 2];
            p2[k] = bmaxabs2(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 4));
        }
        uint32_t p3;
        {
            const uint32_t keep = b1 ? p2[1] : p2[0], send = b1 ? p2[0] : p2[1];
            p3 = bmaxabs2(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 2));
        }
        p3 = bmaxabs2(p3, __shfl_xor_sync(0xFFFFFFFFu, p3, 1));
        const float own_s = group_scale(bmax_final(babs2(p3)));
        const Quot own = make_quot(own_s);
        const int64_t kbo = (k0 >> 7) + 2 * jo + half;  // this lane's group
        if ((l16 & 1) == 0 && jo < nv && kbo * GRP < K)
            s[kbo * lds + m] = own_s;
        uint8_t *qp = q + m * ldq + k0 + 8 * lane;
        if (__any_sync(0xFFFFFFFFu, own.f != 1.0f))
            rows_seg_codes<true>(v, own, lane, nv, kleft, qp);
        else
            rows_seg_codes<false>(v, own, lane, nv, kleft, qp);
    }
}

// ---------------------------------------------------------------------------
// Fused 1x128 + 128x1 on a 128x128 tile: one read of x.
//
// Row pass (registers): half-warp hw16 holds rows hw16 + 16 i (i = 0..7), lane
// l16 columns 8 l16 .. 8 l16 + 7.  Both maxima come from the packed bf16 words
// (|x| by clearing the sign bits, then max.bf16x2; the maximum of bf16 values is
// one of them, so it is exact): one word per row (two candidates) and one per
// column pair over the lane's eight rows.  The eight row maxima of a half-warp
// are reduced in one transposed exchange (each step hands half of the remaining
// groups to the partner lane), after which lane pair (2g, 2g+1) holds group g's
// amax and computes its scale once; the encoding lanes fetch (r, s) by shuffle.
// The raw tile is staged in shared memory (row pitch 272 B): the row encode reads
// its rows back from there (the registers are not held across the reductions),
// and so does the column pass.
//
// Column pass: 128 threads reduce the eight per-warp column maxima and compute
// the 128 column scales once; then every thread encodes two adjacent columns
// over 32 rows from the staged tile, and the transposed codes go back through
// the same buffer so that they leave as whole 128-byte lines of qT.
//
// Tiles are ordered with the row block fastest: CTAs that run together write
// whole rows of the transposed codes (contiguous 128-byte pieces of one row)
// rather than one piece of many rows.
constexpr int TP = GRP + 8;  // staging row pitch in bf16 elements
// pitch in bytes of the transposed codes staged in the same buffer (128 rows of 128
// codes); it fits in the tile's 128 x TP bf16
constexpr int TQ_PITCH = GRP + 16;
static_assert(GRP * TQ_PITCH <= GRP * TP * 2, "the staged codes must fit in the tile buffer");

// Row codes of the eight rows a lane holds, read back from the staged tile (each
// lane reads the words it wrote itself); (r, s[, f]) of row group i come from
// lane (half * 16 + 2 i), which computed it.
template <bool kPrescale>
__device__ __forceinline__ void dual_row_codes(const uint16_t *tile, const Quot &own, int lane, int hw16, int l16,
                                               int rows, uint8_t *__restrict__ qrow, int64_t ldq)
{
    const int src0 = lane & 16;
#pragma unroll 4  // full unrolling hoists every load and shuffle and spills at 64 registers
    for (int i = 0; i < 8; ++i) {
        Quot c;
        c.r = __shfl_sync(0xFFFFFFFFu, own.r, src0 + 2 * i);
        c.sd = __shfl_sync(0xFFFFFFFFu, own.sd, src0 + 2 * i);
        c.f = kPrescale ? __shfl_sync(0xFFFFFFFFu, own.f, src0 + 2 * i) : 1.0f;
        const int r = hw16 + 16 * i;
        float f[8];
        unpack8(*reinterpret_cast<const uint4 *>(&tile[r * TP + l16 * 8]), f);
        const uint2 codes = encode8_t<kPrescale>(f, c);
        if (r < rows)
            *reinterpret_cast<uint2 *>(qrow + (int64_t)r * ldq + l16 * 8) = codes;
    }
}

template <bool kNorm>
__global__ void __launch_bounds__(256, 4) k_quant_dual(const uint16_t *__restrict__ x, int64_t M, int64_t ldx,
                                                    uint8_t *__restrict__ q, int64_t ldq,
                                                    float *__restrict__ s, int64_t lds,
                                                    uint8_t *__restrict__ qT, int64_t ldqT,
                                                    float *__restrict__ sc, int64_t ldsc, int64_t MB, int64_t KB,
                                                    const float *__restrict__ rstd,
                                                    const uint16_t *__restrict__ gamma)
{
    pdl_begin();
    __shared__ __align__(16) uint16_t tile[GRP * TP];
    __shared__ __align__(16) uint32_t ccm[8][GRP / 2];  // per-warp column-pair maxima
    __shared__ __align__(8) float col_r[GRP], col_nsd[GRP], col_f[GRP];
    const int t = threadIdx.x, lane = t & 31, half = lane >> 4, l16 = lane & 15, warp = t >> 5;
    const int hw16 = warp * 2 + half;  // 0..15
    const int c2 = t & 63, rq = t >> 6;

    for (int64_t kb = blockIdx.y; kb < KB; kb += gridDim.y)
    for (int64_t mb = blockIdx.x; mb < MB; mb += gridDim.x) {
        const int64_t m0 = mb * GRP;
        const int rows = (int)((M - m0) < GRP ? (M - m0) : GRP);

        // ---- row pass.  Rows beyond M read as zero (they raise no maximum).
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = hw16 + 16 * i;
            v[i] = (r < rows) ? ld_stream(x + (m0 + r) * ldx + kb * GRP + l16 * 8) : make_uint4(0, 0, 0, 0);
        }
        uint4 g = make_uint4(0, 0, 0, 0);
        if (kNorm)
            g = *reinterpret_cast<const uint4 *>(gamma + kb * GRP + l16 * 8);
        uint32_t pm[8], cm[4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (kNorm) {
                const int r = hw16 + 16 * i;
                v[i] = norm8(v[i], r < rows ? __ldg(rstd + m0 + r) : 0.0f, g);
            }
            const uint32_t a0 = babs2(v[i].x), a1 = babs2(v[i].y), a2 = babs2(v[i].z), a3 = babs2(v[i].w);
            pm[i] = bmax2(bmax2(a0, a1), bmax2(a2, a3));
            if (i == 0) {
                cm[0] = a0, cm[1] = a1, cm[2] = a2, cm[3] = a3;
            } else {
                cm[0] = bmax2(cm[0], a0), cm[1] = bmax2(cm[1], a1);
                cm[2] = bmax2(cm[2], a2), cm[3] = bmax2(cm[3], a3);
            }
            *reinterpret_cast<uint4 *>(&tile[(hw16 + 16 * i) * TP + l16 * 8]) = v[i];
        }
        // column maxima: the two half-warps hold the same columns
#pragma unroll
        for (int j = 0; j < 4; ++j)
            cm[j] = bmax2(cm[j], __shfl_xor_sync(0xFFFFFFFFu, cm[j], 16));
        if (half == 0)
            *reinterpret_cast<uint4 *>(&ccm[warp][4 * l16]) = make_uint4(cm[0], cm[1], cm[2], cm[3]);
        // row maxima: transposed exchange over the half-warp (lane bits 3, 2, 1
        // pick the group kept at each step; bit 0 pairs lanes with equal results)
        const bool b3 = l16 & 8, b2 = l16 & 4, b1 = l16 & 2;
        uint32_t p1[4], p2[2];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t keep = b3 ? pm[k + 4] : pm[k], send = b3 ? pm[k] : pm[k + 4];
            p1[k] = bmax2(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 8));
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint32_t keep = b2 ? p1[k + 2] : p1[k], send = b2 ? p1[k] : p1[k + 2];
            p2[k] = bmax2(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 4));
        }
        uint32_t p3;
        {
            const uint32_t keep = b1 ? p2[1] : p2[0], send = b1 ? p2[0] : p2[1];
            p3 = bmax2(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 2));
        }
        p3 = bmax2(p3, __shfl_xor_sync(0xFFFFFFFFu, p3, 1));
        const int gr = hw16 + 16 * (l16 >> 1);  // the row whose scale this lane computes
        const float own_s = group_scale(bmax_final(p3));
        const Quot own = make_quot(own_s);
        if ((l16 & 1) == 0 && gr < rows)
            s[kb * lds + m0 + gr] = own_s;
        uint8_t *qrow = q + m0 * ldq + kb * GRP;
        if (__any_sync(0xFFFFFFFFu, own.f != 1.0f))
            dual_row_codes<true>(tile, own, lane, hw16, l16, rows, qrow, ldq);
        else
            dual_row_codes<false>(tile, own, lane, hw16, l16, rows, qrow, ldq);
        __syncthreads();

        // ---- column scales, once per column
        if (t < GRP) {
            uint32_t m = ccm[0][t >> 1];
#pragma unroll
            for (int w = 1; w < 8; ++w)
                m = bmax2(m, ccm[w][t >> 1]);
            const float am = fmaxf((t & 1) ? bf_hi(m) : bf_lo(m), 0.0f);
            const float cs = group_scale(am);
            const Quot c = make_quot(cs);
            col_r[t] = c.r;
            col_nsd[t] = -c.sd;
            col_f[t] = c.f;
            sc[mb * ldsc + kb * GRP + t] = cs;
        }
        __syncthreads();

        // ---- column pass: thread owns columns 2*c2, 2*c2+1 over rows rq*32 .. +31
        const uint32_t *col = reinterpret_cast<const uint32_t *>(tile) + c2;
        // one packed lane per column: (even column, odd column) of the same row
        const float2 pf = *reinterpret_cast<const float2 *>(&col_f[2 * c2]);
        const float2 pr = *reinterpret_cast<const float2 *>(&col_r[2 * c2]);
        const float2 pn = *reinterpret_cast<const float2 *>(&col_nsd[2 * c2]);
        uint32_t e[8], o[8];  // 32 codes of each column, 4 per word
        if (pf.x == 1.0f && pf.y == 1.0f)
            encode_cols<false>(col, rq, TP / 2, pf, pr, pn, e, o);
        else
            encode_cols<true>(col, rq, TP / 2, pf, pr, pn, e, o);
        const int64_t k = kb * GRP + 2 * c2;
        const int r0 = rq * 32;
        uint8_t *d0 = qT + k * ldqT + m0 + r0;
        uint8_t *d1 = d0 + ldqT;
        if (rows == GRP) {
            // full tile: the transposed codes are staged in the tile buffer (every thread
            // has read its columns of it) and leave by whole 128-byte lines, each warp
            // writing four rows of qT, rather than as 32-byte runs of 64 rows per warp
            // (measured 11% faster on [8192, 14336])
            __syncthreads();
            uint8_t *tq = reinterpret_cast<uint8_t *>(tile);
            *reinterpret_cast<uint4 *>(tq + (2 * c2) * TQ_PITCH + r0) = make_uint4(e[0], e[1], e[2], e[3]);
            *reinterpret_cast<uint4 *>(tq + (2 * c2) * TQ_PITCH + r0 + 16) = make_uint4(e[4], e[5], e[6], e[7]);
            *reinterpret_cast<uint4 *>(tq + (2 * c2 + 1) * TQ_PITCH + r0) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4 *>(tq + (2 * c2 + 1) * TQ_PITCH + r0 + 16) = make_uint4(o[4], o[5], o[6], o[7]);
            __syncthreads();
#pragma unroll
            for (int rd = 0; rd < 4; ++rd) {
                const int cl = rd * 32 + (t >> 3), ch = t & 7;
                const uint4 v = *reinterpret_cast<const uint4 *>(tq + cl * TQ_PITCH + ch * 16);
                *reinterpret_cast<uint4 *>(qT + (kb * GRP + cl) * ldqT + m0 + ch * 16) = v;
            }
        } else if (r0 + 32 <= rows) {
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
        __syncthreads();  // tile, ccm and the column scales are reused by the next mb
    }
}

// ---------------------------------------------------------------------------
// RMSNorm row factor (QuRL notes, 关键设计 §1: the UAQ scale is folded into the
// norm's weight, so the normalised activation is what the quantizers take):
//   acc = sum of h[m,k]^2 over k in index order, by fused multiply-adds in fp32
//   rstd[m] = fl32(1 / fl32(sqrt(fl32(fl32(acc / K) + eps))))
// The index order makes the sum, and so every code downstream, independent of
// the launch shape.  One thread owns one row and runs its chain of K FMAs, so
// the kernel's floor is K dependent FMA latencies, and everything else is kept
// off that chain: a CTA of two warps takes 32 rows, warp 1 copies 32 rows x 128
// columns per step into a ring of RMS_STAGES shared-memory slots (16-byte
// cp.async copies) and warp 0 runs the chains.  Hardware named barriers pass
// each slot between them (full: the producer's copies of the slot have landed;
// empty: the consumer has read it), so no thread spins.  The FMAs take the bf16
// halves of each word directly (mixed-precision FMA: the bf16 operands enter
// exactly, one rounding to fp32, as fmaf on the widened values), so no
// unpacking sits between them.  Row pitch 272 bytes: the 16-byte reads of each
// quarter-warp fall in distinct bank groups.
constexpr int RMS_ROWS = 32;
constexpr int RMS_PITCH = GRP * 2 + 16;
constexpr int RMS_STAGES = 6;
constexpr int RMS_LOOKAHEAD = RMS_STAGES - 2;  // chunks in flight behind the one signalled full
constexpr int RMS_SMEM = RMS_STAGES * RMS_ROWS * RMS_PITCH;

__device__ __forceinline__ void cp_async16_q(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// named barriers 1 .. RMS_STAGES (slot full) and RMS_STAGES + 1 .. 2 RMS_STAGES
// (slot empty), each between the CTA's two warps
__device__ __forceinline__ void nbar_sync(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }
__device__ __forceinline__ void nbar_arrive(int id) { asm volatile("bar.arrive %0, 64;" ::"r"(id) : "memory"); }

// acc + lo * lo, then + hi * hi, for the two bf16 halves of w (lo = bits 0..15)
__device__ __forceinline__ float fma_sq_bf16x2(uint32_t w, float acc)
{
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "fma.rn.f32.bf16 %0, lo, lo, %0;\n\tfma.rn.f32.bf16 %0, hi, hi, %0;\n\t}"
        : "+f"(acc)
        : "r"(w));
    return acc;
}

__global__ void __launch_bounds__(2 * RMS_ROWS) k_rms_rstd(const uint16_t *__restrict__ h, int64_t M, int64_t K,
                                                           int64_t ldh, float eps, float *__restrict__ rstd)
{
    pdl_begin();
    extern __shared__ __align__(16) uint8_t rms_buf[];
    const int t = threadIdx.x & 31;
    const int64_t m0 = (int64_t)blockIdx.x * RMS_ROWS;
    const int rows = (int)((M - m0) < RMS_ROWS ? (M - m0) : RMS_ROWS);
    const int chunks = (int)(K / GRP);
    if (threadIdx.x >= 32) {
        // producer: copy i of lane t moves piece t & 15 of row (t >> 4) + 2 i, so
        // that each warp-wide copy reads 256 contiguous bytes of two rows; rows at
        // or past M are not copied (their sums are not used)
        const int r0 = t >> 4;
        const uint32_t dst0 = (uint32_t)__cvta_generic_to_shared(rms_buf) + (uint32_t)(r0 * RMS_PITCH + (t & 15) * 16);
        const char *src0 = reinterpret_cast<const char *>(h + m0 * ldh + (t & 15) * 8);
        const int64_t rstride = ldh * (int64_t)sizeof(uint16_t);
#pragma unroll 1
        for (int c = 0; c < chunks + RMS_LOOKAHEAD; ++c) {
            if (c < chunks) {
                const int slot = c % RMS_STAGES;
                if (c >= RMS_STAGES)
                    nbar_sync(1 + RMS_STAGES + slot);  // chunk c - RMS_STAGES has been read
                const uint32_t d = dst0 + (uint32_t)(slot * RMS_ROWS * RMS_PITCH);
                const char *p = src0 + (int64_t)c * GRP * (int64_t)sizeof(uint16_t);
#pragma unroll
                for (int i = 0; i < RMS_ROWS / 2; ++i)
                    if (r0 + 2 * i < rows)
                        cp_async16_q(d + (uint32_t)(2 * i * RMS_PITCH), p + (r0 + 2 * i) * rstride);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");  // one group per step, empty past the end
            const int cf = c - RMS_LOOKAHEAD;                   // the chunk that is now complete
            if (cf >= 0) {
                asm volatile("cp.async.wait_group %0;" ::"n"(RMS_LOOKAHEAD) : "memory");
                nbar_arrive(1 + cf % RMS_STAGES);
            }
        }
        return;
    }
    float acc = 0.0f;
#pragma unroll 1
    for (int c = 0; c < chunks; ++c) {
        const int slot = c % RMS_STAGES;
        nbar_sync(1 + slot);  // chunk c has landed
        const uint8_t *row = rms_buf + slot * RMS_ROWS * RMS_PITCH + t * RMS_PITCH;
        uint4 v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            v[j] = *reinterpret_cast<const uint4 *>(row + 16 * j);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            acc = fma_sq_bf16x2(v[j].x, acc);
            acc = fma_sq_bf16x2(v[j].y, acc);
            acc = fma_sq_bf16x2(v[j].z, acc);
            acc = fma_sq_bf16x2(v[j].w, acc);
        }
        if (c + RMS_STAGES < chunks)
            nbar_arrive(1 + RMS_STAGES + slot);  // every read of the slot is done: it may be refilled
    }
    if (t < rows) {
        const float ms = __fdiv_rn(acc, (float)K);
        rstd[m0 + t] = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
    }
}

// ---------------------------------------------------------------------------
// 128x128 weight blocks: one CTA per block, everything in registers.  Thread
// (warp a, lane j) loads rows 16 a .. 16 a + 15, columns 4 j .. 4 j + 3 (one
// 8-byte load per row; a warp covers whole 256-byte rows), so the block's amax
// is a packed bf16 maximum, a warp shuffle reduction and one exchange through
// shared memory.  Each thread then encodes its 64 elements: one 32-bit word of
// codes per row, and for the [K,N] copy four 4x4 byte transposes (byte
// permutes) turn the sixteen row words into four 16-byte runs, one per column,
// which go out through shared memory as whole 128-byte lines of the copy.
// Blocks are ordered with the row block fastest, as in the fused quantizer.
__device__ __forceinline__ uint2 ld_stream8(const uint16_t *p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Four rows of four bytes (r[i] = row i, column c in byte c) to four columns
// (c[k] = column k, row i in byte i).
__device__ __forceinline__ void transpose4x4(const uint32_t (&r)[4], uint32_t (&c)[4])
{
    const uint32_t t0 = prmt(r[0], r[1], 0x5140), t1 = prmt(r[0], r[1], 0x7362);
    const uint32_t t2 = prmt(r[2], r[3], 0x5140), t3 = prmt(r[2], r[3], 0x7362);
    c[0] = prmt(t0, t2, 0x5410);
    c[1] = prmt(t0, t2, 0x7632);
    c[2] = prmt(t1, t3, 0x5410);
    c[3] = prmt(t1, t3, 0x7632);
}

template <bool kPrescale>
__device__ __forceinline__ void encode_strip(const uint2 (&v)[16], const Quot &c, uint32_t (&cw)[16])
{
    const float2 f = make_float2(c.f, c.f), r = make_float2(c.r, c.r), nsd = make_float2(-c.sd, -c.sd);
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
        const float2 a = quot2<kPrescale>(make_float2(bf_lo(v[rr].x), bf_hi(v[rr].x)), f, r, nsd);
        const float2 b = quot2<kPrescale>(make_float2(bf_lo(v[rr].y), bf_hi(v[rr].y)), f, r, nsd);
        cw[rr] = e4m3x2(a.x, a.y) | (e4m3x2(b.x, b.y) << 16);
    }
}

__global__ void __launch_bounds__(256, 4) k_quant_weight(const uint16_t *__restrict__ w, int64_t ldw,
                                                         uint8_t *__restrict__ q, int64_t ldq,
                                                         float *__restrict__ s, int64_t lds,
                                                         uint8_t *__restrict__ qT, int64_t ldqT, int64_t NB, int64_t KB)
{
    pdl_begin();
    __shared__ float red[8];
    __shared__ __align__(16) uint8_t tqs[GRP * GRP];  // transposed codes: 128 rows of 128 bytes, swizzled
    const int t = threadIdx.x, j = t & 31, a = t >> 5;

    for (int64_t kb = blockIdx.y; kb < KB; kb += gridDim.y)
    for (int64_t nb = blockIdx.x; nb < NB; nb += gridDim.x) {
        const int64_t n0 = nb * GRP;
        const uint16_t *src = w + (n0 + 16 * a) * ldw + kb * GRP + 4 * j;
        uint2 v[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr)
            v[rr] = ld_stream8(src + rr * ldw);
        uint32_t m = 0;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr)
            m = bmax2(m, bmax2(babs2(v[rr].x), babs2(v[rr].y)));
        float am = bmax_final(m);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
        if (j == 0)
            red[a] = am;
        __syncthreads();
        am = red[0];
#pragma unroll
        for (int i = 1; i < 8; ++i)
            am = fmaxf(am, red[i]);
        const float sc = group_scale(am);
        const Quot c = make_quot(sc);
        if (t == 0)
            s[nb * lds + kb] = sc;
        uint32_t cw[16];  // codes of row 16 a + rr, columns 4 j .. 4 j + 3
        if (c.f == 1.0f)
            encode_strip<false>(v, c, cw);
        else
            encode_strip<true>(v, c, cw);
        uint8_t *dst = q + (n0 + 16 * a) * ldq + kb * GRP + 4 * j;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr)
            *reinterpret_cast<uint32_t *>(dst + rr * ldq) = cw[rr];
        if (qT) {
            uint32_t col[4][4];  // col[k][b]: column 4 j + k, rows 16 a + 4 b .. + 3
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const uint32_t rw[4] = {cw[4 * b], cw[4 * b + 1], cw[4 * b + 2], cw[4 * b + 3]};
                uint32_t cc[4];
                transpose4x4(rw, cc);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    col[k][b] = cc[k];
            }
            // staged as row 4 j + k of the block, 16-byte chunk a (XOR-swizzled by
            // (row / 4) % 8: conflict-free both ways), then written out as whole
            // 128-byte lines, each warp four rows of qT (measured 13-15% faster than
            // each warp writing 16 bytes into each of 128 rows)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint4 *>(tqs + (4 * j + k) * GRP + ((a ^ (j & 7)) << 4)) =
                    make_uint4(col[k][0], col[k][1], col[k][2], col[k][3]);
            __syncthreads();
#pragma unroll
            for (int rd = 0; rd < 4; ++rd) {
                const int cl = rd * 32 + (t >> 3), ch = t & 7;
                const uint4 v = *reinterpret_cast<const uint4 *>(tqs + cl * GRP + ((ch ^ ((cl >> 2) & 7)) << 4));
                *reinterpret_cast<uint4 *>(qT + (kb * GRP + cl) * ldqT + n0 + ch * 16) = v;
            }
        }
        __syncthreads();  // red and the staged codes are reused by the next block
    }
}

// ---------------------------------------------------------------------------
// Per-row quantization (QuRL notes, "损失函数 / 训练策略": per-token activations,
// per-channel weights): one group per row over all K columns.  A row is taken
// by one warp (kThreads = 32: enough rows to fill the GPU, or rows of at most
// 4096 elements) or by a whole CTA (kThreads = 256: few, long rows).  Pass 1 reads the row (16-byte loads, four
// in flight per lane) and takes the packed bf16 maximum, reduced by shuffles
// (and across the CTA's warps through shared memory); one thread computes the
// scale once and hands (r, s, f) to the others; pass 2 reads the row again,
// from L2 (it was read moments before), encodes it and stores the codes.  With
// s_rep set, the scale is also written to s_rep[kb * ld_rep + m] for every
// K-block, the layout the column-scaled GEMM reads.
template <bool kPrescale>
__device__ __forceinline__ void per_row_codes(const uint16_t *__restrict__ row, int64_t K, int t, int stride,
                                              const Quot &c, uint8_t *__restrict__ qrow)
{
#pragma unroll 4
    for (int64_t k = (int64_t)t * 8; k < K; k += stride) {
        float f[8];
        unpack8(ld_stream(row + k), f);
        *reinterpret_cast<uint2 *>(qrow + k) = encode8_t<kPrescale>(f, c);
    }
}

template <int kThreads>
__global__ void __launch_bounds__(256) k_quant_per_row(const uint16_t *__restrict__ x, int64_t M, int64_t K,
                                                       int64_t ldx, uint8_t *__restrict__ q, int64_t ldq,
                                                       float *__restrict__ s, float *__restrict__ s_rep,
                                                       int64_t ld_rep)
{
    pdl_begin();
    __shared__ uint32_t red[8];
    __shared__ float sh[4];  // s, r, s*f, f of the CTA's row
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = threadIdx.x % kThreads;  // thread within the row's team
    const int64_t team = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / kThreads;
    const int64_t nteams = ((int64_t)gridDim.x * blockDim.x) / kThreads;
    for (int64_t m = team; m < M; m += nteams) {
        const uint16_t *row = x + m * ldx;
        uint32_t pm = 0;
#pragma unroll 4
        for (int64_t k = (int64_t)t * 8; k < K; k += 8 * kThreads) {
            const uint4 v = *reinterpret_cast<const uint4 *>(row + k);  // kept in L2 for pass 2
            pm = bmaxabs2(pm, bmaxabs2(bmaxabs2(v.x, v.y), bmaxabs2(v.z, v.w)));
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            pm = bmaxabs2(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, o));
        float sc = 0.0f;
        Quot c{1.0f, 1.0f, 1.0f};
        if (kThreads == 32) {
            if (lane == 0) {
                sc = group_scale(bmax_final(babs2(pm)));
                c = make_quot(sc);
                s[m] = sc;
            }
            sc = __shfl_sync(0xFFFFFFFFu, sc, 0);
            c.r = __shfl_sync(0xFFFFFFFFu, c.r, 0);
            c.sd = __shfl_sync(0xFFFFFFFFu, c.sd, 0);
            c.f = __shfl_sync(0xFFFFFFFFu, c.f, 0);
        } else {
            if (lane == 0)
                red[warp] = babs2(pm);
            __syncthreads();
            if (t == 0) {
                uint32_t a = red[0];
#pragma unroll
                for (int w = 1; w < kThreads / 32; ++w)
                    a = bmax2(a, red[w]);
                const float v = group_scale(bmax_final(a));
                const Quot cq = make_quot(v);
                sh[0] = v, sh[1] = cq.r, sh[2] = cq.sd, sh[3] = cq.f;
                s[m] = v;
            }
            __syncthreads();
            sc = sh[0], c.r = sh[1], c.sd = sh[2], c.f = sh[3];
        }
        if (s_rep)
            for (int64_t kb = t; kb < K / GRP; kb += kThreads)
                s_rep[kb * ld_rep + m] = sc;
        if (c.f == 1.0f)
            per_row_codes<false>(row, K, t, 8 * kThreads, c, q + m * ldq);
        else
            per_row_codes<true>(row, K, t, 8 * kThreads, c, q + m * ldq);
        if (kThreads > 32)
            __syncthreads();  // red and sh are reused by the next row
    }
}

// Rows of at most 256 * NV elements: a warp per row holds the whole row in
// registers (NV 16-byte loads per lane, all in flight), so the row is read from
// memory once; same scale rule and encoding as k_quant_per_row.
template <int NV>
__global__ void __launch_bounds__(256) k_quant_per_row_reg(const uint16_t *__restrict__ x, int64_t M, int64_t K,
                                                           int64_t ldx, uint8_t *__restrict__ q, int64_t ldq,
                                                           float *__restrict__ s, float *__restrict__ s_rep,
                                                           int64_t ld_rep)
{
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int64_t team = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nteams = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t m = team; m < M; m += nteams) {
        const uint16_t *row = x + m * ldx;
        uint4 v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int k = (32 * i + lane) * 8;
            v[i] = k < K ? ld_stream(row + k) : make_uint4(0, 0, 0, 0);
        }
        uint32_t pm = 0;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            pm = bmaxabs2(pm, bmaxabs2(bmaxabs2(v[i].x, v[i].y), bmaxabs2(v[i].z, v[i].w)));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            pm = bmaxabs2(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, o));
        float sc = 0.0f;
        Quot c{1.0f, 1.0f, 1.0f};
        if (lane == 0) {
            sc = group_scale(bmax_final(babs2(pm)));
            c = make_quot(sc);
            s[m] = sc;
        }
        sc = __shfl_sync(0xFFFFFFFFu, sc, 0);
        c.r = __shfl_sync(0xFFFFFFFFu, c.r, 0);
        c.sd = __shfl_sync(0xFFFFFFFFu, c.sd, 0);
        c.f = __shfl_sync(0xFFFFFFFFu, c.f, 0);
        if (s_rep)
            for (int64_t kb = lane; kb < K / GRP; kb += 32)
                s_rep[kb * ld_rep + m] = sc;
        uint8_t *qrow = q + m * ldq;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int k = (32 * i + lane) * 8;
            if (k < K) {
                float f[8];
                unpack8(v[i], f);
                *reinterpret_cast<uint2 *>(qrow + k) = encode8(f, c);
            }
        }
    }
}

// Longer rows of at most 2048 * NV elements: a CTA per row holds it in registers
// (NV 16-byte loads per thread), one read of x.
template <int NV>
__global__ void __launch_bounds__(256) k_quant_per_row_reg_cta(const uint16_t *__restrict__ x, int64_t M, int64_t K,
                                                               int64_t ldx, uint8_t *__restrict__ q, int64_t ldq,
                                                               float *__restrict__ s, float *__restrict__ s_rep,
                                                               int64_t ld_rep)
{
    pdl_begin();
    __shared__ uint32_t red[8];
    __shared__ float sh[4];  // s, r, s*f, f of the CTA's row
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const uint16_t *row = x + m * ldx;
        uint4 v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int64_t k = ((int64_t)256 * i + t) * 8;
            v[i] = k < K ? ld_stream(row + k) : make_uint4(0, 0, 0, 0);
        }
        uint32_t pm = 0;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            pm = bmaxabs2(pm, bmaxabs2(bmaxabs2(v[i].x, v[i].y), bmaxabs2(v[i].z, v[i].w)));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            pm = bmaxabs2(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, o));
        if (lane == 0)
            red[warp] = babs2(pm);
        __syncthreads();
        if (t == 0) {
            uint32_t a = red[0];
#pragma unroll
            for (int w = 1; w < 8; ++w)
                a = bmax2(a, red[w]);
            const float sv = group_scale(bmax_final(a));
            const Quot cq = make_quot(sv);
            sh[0] = sv, sh[1] = cq.r, sh[2] = cq.sd, sh[3] = cq.f;
            s[m] = sv;
        }
        __syncthreads();
        const float sc = sh[0];
        Quot c;
        c.r = sh[1], c.sd = sh[2], c.f = sh[3];
        if (s_rep)
            for (int64_t kb = t; kb < K / GRP; kb += 256)
                s_rep[kb * ld_rep + m] = sc;
        uint8_t *qrow = q + m * ldq;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int64_t k = ((int64_t)256 * i + t) * 8;
            if (k < K) {
                float f[8];
                unpack8(v[i], f);
                *reinterpret_cast<uint2 *>(qrow + k) = encode8(f, c);
            }
        }
        __syncthreads();  // red and sh are reused by the next row
    }
}

// ---------------------------------------------------------------------------
// NVFP4 weight quantization (QeRL news article: 4-bit floats with two-level
// scaling, FP8 E4M3 block scales and an FP32 tensor scale).  E2M1 elements, blocks
// of 16 consecutive elements along K, tensor scale st = amax / (6 * 448):
//   block code  sb = E4M3_RNsat(fl32(fl32(amax_b / 6) / st)),
//   element     q  = E2M1_RNsat(fl32(x / fl32(decode(sb) * st))), +-0 when that is 0.
// Three launches: the tensor amax (packed maxima, one atomic max per warp, the
// bits of a non-negative float ordering as unsigned integers), the block pass
// (one thread per block; the codes of the IEEE quotients through a bracketing test
// that divides only next to a rounding point, E2M1 codes by the hardware
// conversion two at a time), and one thread that turns the amax into st.

// E2M1 codes of two values (RN-even onto 0, 0.5, 1, 1.5, 2, 3, 4, 6, saturating at
// +-6, sign of zero kept), `lo` in bits 0..3 and `hi` in bits 4..7: the hardware
// conversion, one instruction per pair.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi)
{
    uint32_t d;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(d)
        : "f"(hi), "f"(lo));
    return d;
}

// E2M1 codes of the pair fl32(x0 / S), fl32(x1 / S), for S a normal fp32 value above
// 2^-100 and r = RN(1 / S).  q = RN(x * r) is within about 1.5 ulps of the IEEE
// quotient, so q * (1 - 2^-20) and q * (1 + 2^-20) (each rounded) bracket it, and
// since rounding to E2M1 is monotone, where the two ends give the same codes those
// are the codes of the IEEE quotients; only pairs with a quotient within 2^-20 of a
// rounding point (a few in 10^5) take the divisions.  Sign of zero kept (q has the
// sign of x).
__device__ __forceinline__ uint32_t nv_codes2(float x0, float x1, float S, float r)
{
    const float2 q = __fmul2_rn(make_float2(x0, x1), make_float2(r, r));
    const float2 lo = __fmul2_rn(q, make_float2(1.0f - 0x1p-20f, 1.0f - 0x1p-20f));
    const float2 hi = __fmul2_rn(q, make_float2(1.0f + 0x1p-20f, 1.0f + 0x1p-20f));
    const uint32_t cl = e2m1x2(lo.x, lo.y), ch = e2m1x2(hi.x, hi.y);
    if (cl == ch)
        return cl;
    return e2m1x2(__fdiv_rn(x0, S), __fdiv_rn(x1, S));
}

// Exact fp32 value of a finite E4M3 code.
__device__ __forceinline__ float e4m3_value(uint32_t e)
{
    const uint32_t ex = (e >> 3) & 15u, m = e & 7u;
    const float v = ex == 0 ? (float)m * 0x1p-9f : __uint_as_float(((ex + 120u) << 23) | (m << 20));
    return (e & 0x80u) ? -v : v;
}

// 16-byte load that allocates in L2 (the amax pass leaves W there for the block
// pass) but not in L1, through the read-only path (measured 3-5% faster than a
// plain cached load for the amax pass).
__device__ __forceinline__ uint4 ld_keep(const uint16_t *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Tensor amax.  CTAs walk whole rows (no index division), threads 8 elements
// apart, four loads in flight per thread.
__global__ void __launch_bounds__(256) k_nvfp4_amax(const uint16_t *__restrict__ w, int64_t N, int64_t K, int64_t ldw,
                                                    unsigned int *__restrict__ amax_bits)
{
    pdl_begin();
    const int K8 = (int)(K / 8);
    uint32_t pm = 0;
    for (int64_t n = blockIdx.x; n < N; n += gridDim.x) {
        const uint16_t *row = w + n * ldw;
        for (int k8 = threadIdx.x; k8 < K8; k8 += 4 * 256) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                v[u] = k8 + 256 * u < K8 ? ld_keep(row + 8 * (k8 + 256 * u)) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                pm = bmaxabs2(pm, bmaxabs2(bmaxabs2(v[u].x, v[u].y), bmaxabs2(v[u].z, v[u].w)));
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        pm = bmaxabs2(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, o));
    if ((threadIdx.x & 31) == 0)
        atomicMax(amax_bits, __float_as_uint(bmax_final(babs2(pm))));
}

__global__ void __launch_bounds__(256) k_nvfp4_quant(const uint16_t *__restrict__ w, int64_t N, int64_t K,
                                                     int64_t ldw, uint8_t *__restrict__ q, int64_t ldq,
                                                     uint8_t *__restrict__ sb, int64_t ldsb,
                                                     const unsigned int *__restrict__ amax_bits)
{
    pdl_begin();
    const float amax = __uint_as_float(*amax_bits);
    const float st = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);  // 6 * 448
    // block codes by the bracketing test of nv_codes2: (amax_b * RN(1/6)) * RN(1/st) is
    // within a few ulps of fl32(fl32(amax_b / 6) / st), and where the E4M3 codes of
    // its two ends (x (1 -+ 2^-20)) agree they are the code; else both IEEE divisions.
    // A tensor scale below 2^-100 (1 / st may overflow) always divides.
    const bool st_fast = st >= 0x1p-100f;
    const float rst = __frcp_rn(st);
    constexpr float kR6 = 1.0f / 6.0f;  // RN(1/6)
    const int KB = (int)(K / 16);
    // CTAs walk whole rows, a thread per 16-element block; the next block's 32 bytes
    // are loaded before this one is encoded (two loads in flight per thread)
    int64_t n = blockIdx.x;
    int kb = threadIdx.x;
    auto next = [&](int64_t &nn, int &kk) {
        kk += 256;
        if (kk >= KB) {
            kk = threadIdx.x;
            nn += gridDim.x;
        }
    };
    uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0;
    if (kb < KB && n < N) {
        c0 = ld_stream(w + n * ldw + (int64_t)kb * 16);
        c1 = ld_stream(w + n * ldw + (int64_t)kb * 16 + 8);
    }
    for (; kb < KB && n < N;) {
        int64_t nn = n;
        int kk = kb;
        next(nn, kk);
        uint4 p0 = make_uint4(0, 0, 0, 0), p1 = p0;
        if (nn < N) {
            p0 = ld_stream(w + nn * ldw + (int64_t)kk * 16);
            p1 = ld_stream(w + nn * ldw + (int64_t)kk * 16 + 8);
        }
        float f[16];
        unpack8(c0, *reinterpret_cast<float(*)[8]>(&f[0]));
        unpack8(c1, *reinterpret_cast<float(*)[8]>(&f[8]));
        const uint32_t pm = bmaxabs2(bmaxabs2(bmaxabs2(c0.x, c0.y), bmaxabs2(c0.z, c0.w)),
                                     bmaxabs2(bmaxabs2(c1.x, c1.y), bmaxabs2(c1.z, c1.w)));
        const float ab = bmax_final(babs2(pm));
        uint32_t e;
        {
            const float qs = __fmul_rn(__fmul_rn(ab, kR6), rst);
            const uint32_t ew = e4m3x2(__fmul_rn(qs, 1.0f - 0x1p-20f), __fmul_rn(qs, 1.0f + 0x1p-20f));
            e = (st_fast && (ew & 0xFFu) == (ew >> 8)) ? (ew & 0xFFu)
                                                     : (e4m3x2(__fdiv_rn(__fdiv_rn(ab, 6.0f), st), 0.0f) & 0xFFu);
        }
        sb[n * ldsb + kb] = (uint8_t)e;
        const float S = __fmul_rn(e4m3_value(e), st);
        uint32_t word[2] = {0u, 0u};
        if (S == 0.0f) {  // a block below the format's range: +-0 codes, sign kept
#pragma unroll
            for (int j = 0; j < 16; ++j)
                word[j >> 3] |= (signbit(f[j]) ? 8u : 0u) << (4 * (j & 7));
        } else if (S < 0x1p-100f) {  // 1 / S may overflow: IEEE quotients throughout
#pragma unroll
            for (int j = 0; j < 16; j += 2)
                word[j >> 3] |= e2m1x2(__fdiv_rn(f[j], S), __fdiv_rn(f[j + 1], S)) << (4 * (j & 7));
        } else {
            const float r = __frcp_rn(S);
#pragma unroll
            for (int j = 0; j < 16; j += 2)
                word[j >> 3] |= nv_codes2(f[j], f[j + 1], S, r) << (4 * (j & 7));
        }
        *reinterpret_cast<uint2 *>(q + n * ldq + kb * 8) = make_uint2(word[0], word[1]);
        c0 = p0, c1 = p1, n = nn, kb = kk;
    }
}

__global__ void k_nvfp4_tensor_scale(float *st)
{
    pdl_begin();
    const float amax = *st;  // the amax pass left its bits here
    *st = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
}

// ---------------------------------------------------------------------------
// AQN (QeRL news article: channel-wise Gaussian noise in the LayerNorm scale):
// gamma[k] = bf16_RN(fl32(gamma[k] + fl32(sigma * z[k]))), in place.  The product
// and the sum are rounded separately (no contraction into an FMA).
__global__ void __launch_bounds__(256) k_aqn_perturb(uint16_t *__restrict__ gamma, int64_t K,
                                                     const float *__restrict__ z, float sigma)
{
    pdl_begin();
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < K; k += (int64_t)gridDim.x * blockDim.x) {
        const float v = __fadd_rn(bf_lo(gamma[k]), __fmul_rn(sigma, z[k]));
        uint16_t h;
        asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(v));
        gamma[k] = h;
    }
}

// ---------------------------------------------------------------------------
// UAQ fold, in place: divide (w) or multiply (prev) column k by s[k] in fp32,
// round to bf16.  8 elements per thread and vector; each thread handles FOLD_ROWS
// rows per iteration with all their loads issued first (bytes in flight hide
// the memory latency).  One launch for both tensors: CTA rows blockIdx.y < gw
// fold w (row groups grid-strided over gw), the rest fold prev.
constexpr int FOLD_ROWS = 4;

template <bool kDivide>
__device__ __forceinline__ void fold_rows(uint16_t *__restrict__ a, int64_t rows, int64_t lda, int64_t v,
                                          const float (&sv)[8], int64_t y, int64_t gy)
{
    for (int64_t r0 = y * FOLD_ROWS; r0 < rows; r0 += gy * FOLD_ROWS) {
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

__global__ void __launch_bounds__(256) k_uaq_fold(uint16_t *__restrict__ w, int64_t N, int64_t ldw,
                                                  uint16_t *__restrict__ prev, int64_t R, int64_t ldp, int64_t K8,
                                                  const float *__restrict__ s, int gw)
{
    pdl_begin();
    const int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= K8)
        return;
    const float4 s0 = __ldg(reinterpret_cast<const float4 *>(s) + 2 * v);
    const float4 s1 = __ldg(reinterpret_cast<const float4 *>(s) + 2 * v + 1);
    const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    if ((int)blockIdx.y < gw)
        fold_rows<true>(w, N, ldw, v, sv, blockIdx.y, gw);
    else
        fold_rows<false>(prev, R, ldp, v, sv, blockIdx.y - gw, (int64_t)gridDim.y - gw);
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
                              float *s, int64_t lds, cudaStream_t st, const float *rstd, const uint16_t *gamma)
{
    // segments of at most 256 * QR_NV elements, as few as cover the row, each the
    // same number of loads per lane
    const int64_t segs = (K + 256 * QR_NV - 1) / (256 * QR_NV);
    const int64_t nv = (K + 256 * segs - 1) / (256 * segs);
    int64_t blocks = (M * segs + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 64;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    if (rstd)
        (void)launch_pdl(k_quant_rows_seg<true>, dim3((unsigned)blocks), dim3(256), 0, st, x, M, K, (int)segs, (int)nv,
                         ldx, q, ldq, s, lds, rstd, gamma);
    else
        (void)launch_pdl(k_quant_rows_seg<false>, dim3((unsigned)blocks), dim3(256), 0, st, x, M, K, (int)segs, (int)nv,
                         ldx, q, ldq, s, lds, nullptr, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_quant_dual(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, int64_t ldq,
                              float *s, int64_t lds, uint8_t *qT, int64_t ldqT, float *sc, int64_t ldsc,
                              cudaStream_t st, const float *rstd, const uint16_t *gamma)
{
    const int64_t MB = (M + GRP - 1) / GRP, KB = K / GRP;
    const dim3 grid((unsigned)(MB < 0x7FFFFFFF ? MB : 0x7FFFFFFF), (unsigned)(KB < 65535 ? KB : 65535));
    if (rstd)
        (void)launch_pdl(k_quant_dual<true>, dim3(grid), dim3(256), 0, st, x, M, ldx, q, ldq, s, lds, qT, ldqT, sc,
                         ldsc, MB, KB, rstd, gamma);
    else
        (void)launch_pdl(k_quant_dual<false>, dim3(grid), dim3(256), 0, st, x, M, ldx, q, ldq, s, lds, qT, ldqT, sc,
                         ldsc, MB, KB, nullptr, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_rms_rstd(const uint16_t *h, int64_t M, int64_t K, int64_t ldh, float eps, float *rstd,
                            cudaStream_t st)
{
    static bool attr = false;  // benign race: every thread sets the same value
    if (!attr) {
        const cudaError_t e = cudaFuncSetAttribute(k_rms_rstd, cudaFuncAttributeMaxDynamicSharedMemorySize, RMS_SMEM);
        if (e != cudaSuccess)
            return e;
        attr = true;
    }
    const int64_t blocks = (M + RMS_ROWS - 1) / RMS_ROWS;
    (void)launch_pdl(k_rms_rstd, dim3((unsigned)blocks), dim3(2 * RMS_ROWS), RMS_SMEM, st, h, M, K, ldh, eps, rstd);
    return cudaGetLastError();
}

cudaError_t launch_quant_weight(const uint16_t *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq,
                                float *s, int64_t lds, uint8_t *qT, int64_t ldqT, cudaStream_t st)
{
    const int64_t NB = N / GRP, KB = K / GRP;
    const dim3 grid((unsigned)(NB < 0x7FFFFFFF ? NB : 0x7FFFFFFF), (unsigned)(KB < 65535 ? KB : 65535));
    (void)launch_pdl(k_quant_weight, dim3(grid), dim3(256), 0, st, w, ldw, q, ldq, s, lds, qT, ldqT, NB, KB);
    return cudaGetLastError();
}

cudaError_t launch_quant_per_row(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, int64_t ldq,
                                 float *s, float *s_rep, int64_t ld_rep, cudaStream_t st)
{
    const int64_t sms = sm_count();
    if (K <= 256 * 16) {  // rows of up to 4096: a warp per row, held in its registers (one read of x)
        int64_t blocks = (M + 7) / 8;
        if (blocks > sms * 2 * 16)
            blocks = sms * 2 * 16;
        if (K <= 256 * 4)
            (void)launch_pdl(k_quant_per_row_reg<4>, dim3((unsigned)blocks), dim3(256), 0, st, x, M, K, ldx, q, ldq, s,
                             s_rep, ld_rep);
        else if (K <= 256 * 8)
            (void)launch_pdl(k_quant_per_row_reg<8>, dim3((unsigned)blocks), dim3(256), 0, st, x, M, K, ldx, q, ldq, s,
                             s_rep, ld_rep);
        else if (K <= 256 * 12)
            (void)launch_pdl(k_quant_per_row_reg<12>, dim3((unsigned)blocks), dim3(256), 0, st, x, M, K, ldx, q, ldq, s,
                             s_rep, ld_rep);
        else
            (void)launch_pdl(k_quant_per_row_reg<16>, dim3((unsigned)blocks), dim3(256), 0, st, x, M, K, ldx, q, ldq, s,
                             s_rep, ld_rep);
    } else if (K <= 2048 * 16) {  // longer rows: a CTA per row, held in registers
        // as few loads per thread as cover the row (fewer registers, more resident CTAs;
        // measured: K = 18944 at 10 loads 0.81 of HBM, at 16 loads 0.66)
        const int64_t blocks = M < sms * 16 ? M : sms * 16;
        const int64_t nv = (K + 2047) / 2048;
        if (nv <= 4)
            (void)launch_pdl(k_quant_per_row_reg_cta<4>, dim3((unsigned)blocks), dim3(256), 0, st, x, M, K, ldx, q, ldq,
                             s, s_rep, ld_rep);
        else if (nv <= 6)
            (void)launch_pdl(k_quant_per_row_reg_cta<6>, dim3((unsigned)blocks), dim3(256), 0, st, x, M, K, ldx, q, ldq,
                             s, s_rep, ld_rep);
        else if (nv <= 8)
            (void)launch_pdl(k_quant_per_row_reg_cta<8>, dim3((unsigned)blocks), dim3(256), 0, st, x, M, K, ldx, q, ldq,
                             s, s_rep, ld_rep);
        else if (nv <= 10)
            (void)launch_pdl(k_quant_per_row_reg_cta<10>, dim3((unsigned)blocks), dim3(256), 0, st, x, M, K, ldx, q,
                             ldq, s, s_rep, ld_rep);
        else if (nv <= 12)
            (void)launch_pdl(k_quant_per_row_reg_cta<12>, dim3((unsigned)blocks), dim3(256), 0, st, x, M, K, ldx, q,
                             ldq, s, s_rep, ld_rep);
        else if (nv <= 14)
            (void)launch_pdl(k_quant_per_row_reg_cta<14>, dim3((unsigned)blocks), dim3(256), 0, st, x, M, K, ldx, q,
                             ldq, s, s_rep, ld_rep);
        else
            (void)launch_pdl(k_quant_per_row_reg_cta<16>, dim3((unsigned)blocks), dim3(256), 0, st, x, M, K, ldx, q,
                             ldq, s, s_rep, ld_rep);
    } else if (M >= sms * 64) {  // enough rows for every resident warp: a warp per row
        int64_t blocks = (M + 7) / 8;
        if (blocks > sms * 8 * 16)
            blocks = sms * 8 * 16;
        (void)launch_pdl(k_quant_per_row<32>, dim3((unsigned)blocks), dim3(256), 0, st, x, M, K, ldx, q, ldq, s, s_rep, ld_rep);
    } else {  // few, long rows: a CTA per row
        (void)launch_pdl(k_quant_per_row<256>, dim3((unsigned)M), dim3(256), 0, st, x, M, K, ldx, q, ldq, s, s_rep, ld_rep);
    }
    return cudaGetLastError();
}

cudaError_t launch_quant_nvfp4(const uint16_t *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq,
                               uint8_t *sb, int64_t ldsb, float *st, cudaStream_t st_stream)
{
    cudaError_t e = cudaMemsetAsync(st, 0, sizeof(float), st_stream);
    if (e != cudaSuccess)
        return e;
    unsigned int *amax_bits = reinterpret_cast<unsigned int *>(st);
    // one CTA per row while rows are few, else a grid-stride over rows
    const int64_t cap = (int64_t)sm_count() * 8;
    const int64_t g1 = N > cap ? cap : (N < 1 ? 1 : N);
    (void)launch_pdl(k_nvfp4_amax, dim3((unsigned)g1), dim3(256), 0, st_stream, w, N, K, ldw, amax_bits);
    const int64_t g2 = N > cap * 4 ? cap * 4 : (N < 1 ? 1 : N);
    (void)launch_pdl(k_nvfp4_quant, dim3((unsigned)g2), dim3(256), 0, st_stream, w, N, K, ldw, q, ldq, sb, ldsb, amax_bits);
    (void)launch_pdl(k_nvfp4_tensor_scale, dim3(1), dim3(1), 0, st_stream, st);
    return cudaGetLastError();
}

cudaError_t launch_aqn_perturb(uint16_t *gamma, int64_t K, const float *z, float sigma, cudaStream_t st)
{
    int64_t blocks = (K + 255) / 256;
    if (blocks > (int64_t)sm_count() * 8)
        blocks = (int64_t)sm_count() * 8;
    (void)launch_pdl(k_aqn_perturb, dim3((unsigned)blocks), dim3(256), 0, st, gamma, K, z, sigma);
    return cudaGetLastError();
}

cudaError_t launch_uaq_fold(uint16_t *w, int64_t N, int64_t K, int64_t ldw, const float *s, uint16_t *prev,
                            int64_t R, int64_t ldp, cudaStream_t st)
{
    const int64_t K8 = K / 8;
    const unsigned gx = (unsigned)((K8 + 255) / 256);
    auto gy = [](int64_t rows) {
        const int64_t g = (rows + FOLD_ROWS - 1) / FOLD_ROWS;
        return (int)(g < 32767 ? g : 32767);
    };
    const int gw = N > 0 ? gy(N) : 0;
    const int gp = (prev && R > 0) ? gy(R) : 0;
    if (gw + gp == 0)
        return cudaSuccess;
    (void)launch_pdl(k_uaq_fold, dim3(dim3(gx, (unsigned)(gw + gp))), dim3(256), 0, st, w, N, ldw, prev, R, ldp, K8, s, gw);
    return cudaGetLastError();
}

}  // namespace rlq
