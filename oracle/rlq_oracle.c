/*
 * Oracle for the quantized actor linear layer — TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load
 * this file's library.  The product path (the CUDA library) never does, and
 * this file includes nothing from it.
 *
 * What it computes (plain, slow, obviously correct; OpenMP over independent
 * groups only, no blocking or reordering inside a group):
 *
 *  - FP8 E4M3 ("fn" variant: max 448, no infinities, 0x7F/0xFF are NaN) decode
 *    and round-to-nearest-even, saturating encode.  The pages name FP8 for the
 *    GEMMs (Jet-RL notes, "细粒度 GEMM 量化方案") and E4M3 only as the NVFP4
 *    block-scale format (QeRL news article, key takeaways); the sub-format,
 *    the rounding and the saturation are the plainest readings of what the
 *    pages leave open.
 *  - Fine-grained quantization (Jet-RL notes, "细粒度 GEMM 量化方案", Fig. 6):
 *      * 1x128 groups along K for activations / gradients,
 *      * 128x1 groups along the token dimension for the second WGrad operand,
 *      * 128x128 blocks for weights.
 *    Per group: amax = max |x|, s = fl32(amax / 448) (1.0 when amax == 0),
 *    q = encode(fl32(x / s)) with IEEE fp32 division.  Scales are dequant
 *    multipliers: x ~= decode(q) * s.
 *  - Per-token activation and per-channel weight quantization (QuRL notes,
 *    "损失函数 / 训练策略": channel-wise weight and token-wise activation
 *    quantization, FP8 here): one group per row over all K columns, the same
 *    scale rule and encoding.
 *  - NVFP4 weight quantization (QeRL news article: FP4 with two-level scaling,
 *    E4M3 block scales and an FP32 tensor scale): E2M1 codes, blocks of 16
 *    along K, tensor scale amax / (6 * 448).
 *  - AQN (QeRL news article): channel-wise Gaussian noise added to a norm
 *    scale, gamma'[k] = bf16_RN(gamma[k] + sigma_t z[k]), sigma_t decaying
 *    geometrically from sigma_start to sigma_end; z is drawn by the caller.
 *  - The UAQ invariant-scaling fold WX = (W/s)(sX) (QuRL notes, 关键设计 §1):
 *    W'[n,k] = bf16_RN(fl32(W[n,k] / s_k)),  P'[r,k] = bf16_RN(fl32(P[r,k] * s_k)).
 *  - RMSNorm with the UAQ scale folded into its weight (same section: s can be
 *    folded into the norm's scale), the activation that the 1x128 quantizer then
 *    takes; its fp32 steps are spelled out at orc_rmsnorm.
 *
 * The fp64 GEMMs over dequantized operands live in oracle.py (NumPy).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no -ffast-math:
 * subnormals and IEEE division must be honoured).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs fp32 expressions evaluated in fp32 (FLT_EVAL_METHOD == 0)"
#endif

#define GRP 128

/* ---------------------------------------------------------------- bf16 --- */

static float bf16_bits_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even.  bf16 keeps the upper 16 bits
 * of the fp32 pattern, so rounding looks only at the 16 discarded bits. */
uint16_t orc_f32_to_bf16_rn(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN, outside the contract */
    uint32_t upper = u >> 16, lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1; /* may carry into the exponent, up to infinity: that is RN */
    return (uint16_t)upper;
}

/* ---------------------------------------------------------------- E4M3 --- */

/* Value of an E4M3 code: sign bit 7, exponent bits 6..3 (bias 7), mantissa
 * bits 2..0.  Exponent 0 is subnormal (m * 2^-9).  Exponent 15 with mantissa 7
 * is NaN; every other pattern is finite. */
double orc_e4m3_decode(uint8_t c)
{
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Round a non-negative exact double to an integer, ties to even. */
static double round_half_even(double t)
{
    double f = floor(t), r = t - f;
    if (r > 0.5)
        return f + 1.0;
    if (r < 0.5)
        return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* fp32 -> E4M3: nearest representable value, ties to the even mantissa, and
 * magnitudes at or above 448 clamp to 448 (satfinite).  The sign of zero is
 * kept.  NaN maps to 0x7F (outside the contract). */
uint8_t orc_e4m3_encode(float v)
{
    if (isnan(v))
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0)
        return sign | 0x7E;
    if (a < 0x1p-6) {
        /* subnormal grid: multiples of 2^-9; m == 8 is the first normal 2^-6,
         * whose code 0x08 is exactly the integer 8. */
        double m = round_half_even(a * 512.0);
        return sign | (uint8_t)m;
    }
    int e;
    (void)frexp(a, &e);
    e -= 1; /* a = 2^e * [1, 2) */
    double t = (ldexp(a, -e) - 1.0) * 8.0; /* exact: a has <= 24 significant bits */
    double m = round_half_even(t);
    if (m == 8.0) {
        m = 0.0;
        e += 1;
    }
    /* a < 448 keeps (e, m) at or below (8, 6): no NaN pattern can result. */
    return sign | (uint8_t)(((e + 7) << 3) | (int)m);
}

/* --------------------------------------------------------- group quant --- */

/* Scale of a group from its amax: fl32(amax / 448), or 1.0 for an all-zero
 * group. */
static float group_scale(float amax)
{
    return (amax == 0.0f) ? 1.0f : amax / 448.0f;
}

float orc_group_scale(float amax) { return group_scale(amax); }

/* One element of a group: encode(fl32(x / s)). */
uint8_t orc_quant_element(float x, float s) { return orc_e4m3_encode(x / s); }

/* 1x128 groups along K (row-wise).  x bf16 [M,K] (row pitch ldx elements);
 * q u8 [M,K] (pitch ldq); s f32, s[kb*lds + m]. */
void orc_quant_rows_1x128(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                          uint8_t *q, int64_t ldq, float *s, int64_t lds)
{
    int64_t KB = K / GRP;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            const uint16_t *g = x + m * ldx + kb * GRP;
            float amax = 0.0f;
            for (int i = 0; i < GRP; ++i) {
                float a = fabsf(bf16_bits_to_f32(g[i]));
                if (a > amax)
                    amax = a;
            }
            float sc = group_scale(amax);
            s[kb * lds + m] = sc;
            for (int i = 0; i < GRP; ++i)
                q[m * ldq + kb * GRP + i] = orc_e4m3_encode(bf16_bits_to_f32(g[i]) / sc);
        }
    }
}

/* One group per row over all K columns (per-token activations, per-channel
 * weights).  x bf16 [M,K] (pitch ldx); q u8 [M,K] (pitch ldq); s f32 [M]. */
void orc_quant_per_row(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                       uint8_t *q, int64_t ldq, float *s)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *row = x + m * ldx;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(bf16_bits_to_f32(row[k]));
            if (a > amax)
                amax = a;
        }
        float sc = group_scale(amax);
        s[m] = sc;
        for (int64_t k = 0; k < K; ++k)
            q[m * ldq + k] = orc_e4m3_encode(bf16_bits_to_f32(row[k]) / sc);
    }
}

/* 128x1 groups along M (column-wise), codes written transposed.
 * x bf16 [M,K]; qT u8, qT[k*ldqT + m] for m < M; sc f32, sc[mb*ldsc + k].
 * The last group of a column covers rows mb*128 .. M-1 only. */
void orc_quant_cols_128x1(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                          uint8_t *qT, int64_t ldqT, float *sc, int64_t ldsc)
{
    int64_t MB = (M + GRP - 1) / GRP;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < K; ++k) {
        for (int64_t mb = 0; mb < MB; ++mb) {
            int64_t m0 = mb * GRP, m1 = (m0 + GRP < M) ? m0 + GRP : M;
            float amax = 0.0f;
            for (int64_t m = m0; m < m1; ++m) {
                float a = fabsf(bf16_bits_to_f32(x[m * ldx + k]));
                if (a > amax)
                    amax = a;
            }
            float s = group_scale(amax);
            sc[mb * ldsc + k] = s;
            for (int64_t m = m0; m < m1; ++m)
                qT[k * ldqT + m] = orc_e4m3_encode(bf16_bits_to_f32(x[m * ldx + k]) / s);
        }
    }
}

/* 128x128 blocks (weights).  w bf16 [N,K]; q u8 [N,K]; s[nb*lds + kb];
 * optional qT u8 [K,N] (qT[k*ldqT + n]) holding the same codes transposed. */
void orc_quant_weight_128x128(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                              uint8_t *q, int64_t ldq, float *s, int64_t lds,
                              uint8_t *qT, int64_t ldqT)
{
    int64_t NB = N / GRP, KB = K / GRP;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t nb = 0; nb < NB; ++nb) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int64_t n = nb * GRP; n < (nb + 1) * GRP; ++n)
                for (int64_t k = kb * GRP; k < (kb + 1) * GRP; ++k) {
                    float a = fabsf(bf16_bits_to_f32(w[n * ldw + k]));
                    if (a > amax)
                        amax = a;
                }
            float sc = group_scale(amax);
            s[nb * lds + kb] = sc;
            for (int64_t n = nb * GRP; n < (nb + 1) * GRP; ++n)
                for (int64_t k = kb * GRP; k < (kb + 1) * GRP; ++k) {
                    uint8_t c = orc_e4m3_encode(bf16_bits_to_f32(w[n * ldw + k]) / sc);
                    q[n * ldq + k] = c;
                    if (qT)
                        qT[k * ldqT + n] = c;
                }
        }
    }
}

/* --------------------------------------------------------------- NVFP4 --- */

/* FP4 E2M1 (the element format of NVFP4; QeRL news article: NVFP4 is a 4-bit
 * float with two-level scaling, FP8 E4M3 block scales and an FP32 tensor scale).
 * Code: sign = bit 3, e = bits 2..1, m = bit 0; e = 0 gives +-m/2, otherwise
 * +-(1 + m/2) 2^(e-1): the magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double orc_e2m1_decode(uint8_t c)
{
    int sign = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = (e == 0) ? 0.5 * m : (1.0 + 0.5 * m) * ldexp(1.0, e - 1);
    return sign ? -v : v;
}

/* Round-to-nearest-even onto the E2M1 grid with saturation to +-6; the sign of
 * zero is kept.  Ties go to the code with an even mantissa bit. */
uint8_t orc_e2m1_encode(float v)
{
    uint8_t sign = signbit(v) ? 8 : 0;
    double a = fabs((double)v);
    if (isnan(v))
        return sign | 7;  /* out of contract: saturate */
    if (a >= 6.0)
        return sign | 7;
    uint8_t best = 0;
    for (uint8_t c = 1; c < 8; ++c) {
        double d = fabs(orc_e2m1_decode(c) - a), db = fabs(orc_e2m1_decode(best) - a);
        if (d < db || (d == db && (c & 1) == 0))
            best = c;
    }
    return sign | best;
}

/* NVFP4 quantization of a weight matrix w bf16 [N,K] (K % 16 == 0), two-level:
 *   tensor scale  st = fl32(amax(w) / (6 * 448)), or 1 when w is all zero;
 *   block of 16 consecutive elements along K: sb = E4M3_RNsat(fl32(fl32(amax_b / 6) / st)),
 *   effective block scale S = fl32(decode(sb) * st);
 *   element code q = E2M1_RNsat(fl32(x / S)), or +-0 when S == 0.
 * Outputs: q one code per byte (low nibble) [N,K] (pitch ldq), sb E4M3 codes
 * [N, K/16] (pitch ldsb), *st. */
void orc_quant_nvfp4(const uint16_t *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq,
                     uint8_t *sb, int64_t ldsb, float *st)
{
    float amax = 0.0f;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(bf16_bits_to_f32(w[n * ldw + k]));
            if (a > amax)
                amax = a;
        }
    float t = (amax == 0.0f) ? 1.0f : amax / (6.0f * 448.0f);
    *st = t;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t kb = 0; kb < K / 16; ++kb) {
            const uint16_t *g = w + n * ldw + kb * 16;
            float ab = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float a = fabsf(bf16_bits_to_f32(g[i]));
                if (a > ab)
                    ab = a;
            }
            uint8_t e = orc_e4m3_encode((ab / 6.0f) / t);
            sb[n * ldsb + kb] = e;
            float S = (float)orc_e4m3_decode(e) * t;
            for (int i = 0; i < 16; ++i) {
                float x = bf16_bits_to_f32(g[i]);
                q[n * ldq + kb * 16 + i] = (S == 0.0f) ? (signbit(x) ? 8 : 0) : orc_e2m1_encode(x / S);
            }
        }
    }
}

/* ----------------------------------------------------------------- AQN --- */

/* Noise level of step t of T (QeRL news article: channel-wise Gaussian noise in
 * the LayerNorm scale, decaying on an exponential schedule): geometric from
 * sigma_start at t = 0 to sigma_end at t = T - 1, computed in double and
 * rounded once to fp32; T == 1 gives sigma_start. */
float orc_aqn_sigma(float sigma_start, float sigma_end, int64_t t, int64_t T)
{
    if (T <= 1 || sigma_start == sigma_end)
        return sigma_start;
    double r = (double)t / (double)(T - 1);
    return (float)((double)sigma_start * pow((double)sigma_end / (double)sigma_start, r));
}

/* gamma'[k] = bf16_RN(fl32(gamma[k] + fl32(sigma * z[k]))), in place, for a norm
 * scale gamma (bf16 [K]) and one standard-normal draw z[k] per channel. */
void orc_aqn_perturb(uint16_t *gamma, int64_t K, const float *z, float sigma)
{
    for (int64_t k = 0; k < K; ++k) {
        float noise = sigma * z[k];
        gamma[k] = orc_f32_to_bf16_rn(bf16_bits_to_f32(gamma[k]) + noise);
    }
}

/* ----------------------------------------------------------- RMSNorm --- */

/* RMSNorm of the hidden state ahead of the linear layer, with the UAQ scale
 * already folded into its weight (QuRL notes, 关键设计 §1: the per-channel s
 * that multiplies the previous activation can be folded straight into the
 * LayerNorm / RMSNorm scale, gamma' = gamma * s).  The pages give no formula
 * for the norm itself; the reading used here is the standard one,
 * x = h / sqrt(mean(h^2) + eps) * gamma, with every step in fp32 and one final
 * rounding to bf16 (the activation the layer quantizes):
 *
 *   acc  = sum over k = 0 .. K-1, in index order, of h[m,k]^2, accumulated as
 *          acc = fmaf(h, h, acc) in fp32 from acc = 0
 *   ms   = fl32(acc / K)
 *   d    = fl32(sqrt(fl32(ms + eps)))
 *   r    = fl32(1 / d)                       (written to rstd[m])
 *   x    = bf16_RN(fl32(fl32(h[m,k] * r) * gamma[k]))
 *
 * h [M,K] bf16 (pitch ldh), gamma [K] bf16, x [M,K] bf16 (pitch ldx), rstd [M]. */
void orc_rmsnorm(const uint16_t *h, int64_t M, int64_t K, int64_t ldh, const uint16_t *gamma, float eps,
                 uint16_t *x, int64_t ldx, float *rstd)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        float acc = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float v = bf16_bits_to_f32(h[m * ldh + k]);
            acc = fmaf(v, v, acc);
        }
        float ms = acc / (float)K;
        float d = sqrtf(ms + eps);
        float r = 1.0f / d;
        rstd[m] = r;
        for (int64_t k = 0; k < K; ++k) {
            float hr = bf16_bits_to_f32(h[m * ldh + k]) * r;
            x[m * ldx + k] = orc_f32_to_bf16_rn(hr * bf16_bits_to_f32(gamma[k]));
        }
    }
}

/* ------------------------------------------------------------ UAQ fold --- */

/* W [N,K] bf16 in place: column k divided by s[k]; prev [R,K] bf16 in place
 * (nullable): column k multiplied by s[k].  Each result is rounded to bf16. */
void orc_uaq_fold(uint16_t *w, int64_t N, int64_t K, int64_t ldw, const float *s,
                  uint16_t *prev, int64_t R, int64_t ldp)
{
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * ldw + k] = orc_f32_to_bf16_rn(bf16_bits_to_f32(w[n * ldw + k]) / s[k]);
    if (prev) {
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < R; ++r)
            for (int64_t k = 0; k < K; ++k)
                prev[r * ldp + k] =
                    orc_f32_to_bf16_rn(bf16_bits_to_f32(prev[r * ldp + k]) * s[k]);
    }
}

/* --------------------------------------------------------- bulk helpers --- */

/* Element-wise encode / decode of arrays, for the pins. */
void orc_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(v[i]);
}

void orc_e4m3_decode_array(const uint8_t *c, int64_t n, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_decode(c[i]);
}

void orc_f32_to_bf16_array(const float *v, int64_t n, uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_f32_to_bf16_rn(v[i]);
}

/* Element map of the group quantizer for given (x, s) pairs. */
void orc_quant_element_array(const float *x, const float *s, int64_t n, uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_quant_element(x[i], s[i]);
}

int orc_num_threads(void);
void orc_set_num_threads(int n);
#ifdef _OPENMP
#include <omp.h>
int orc_num_threads(void) { return omp_get_max_threads(); }
void orc_set_num_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
#else
int orc_num_threads(void) { return 1; }
void orc_set_num_threads(int n) { (void)n; }
#endif
