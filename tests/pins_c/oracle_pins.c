/*
 * Exhaustive pins for the oracle's E4M3 encoder and group quantizer element map.
 *
 * These checks restate the rules in a different form from the oracle (nearest
 * search over the decoded code table, double-precision division correctly
 * rounded to fp32) and enumerate every input the rules can see:
 *
 *   pin_encode_exhaustive   all 2^32 fp32 bit patterns
 *   pin_quant_pairs         all (x, amax) bf16 pairs with |x| <= amax, amax > 0
 *
 * Compiled together with oracle/rlq_oracle.c by tests/test_oracle_e4m3.py.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

double orc_e4m3_decode(uint8_t c);
uint8_t orc_e4m3_encode(float v);
float orc_group_scale(float amax);
uint8_t orc_quant_element(float x, float s);

static float bits_f32(uint32_t u)
{
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Sorted non-negative finite magnitudes: code i (0..0x7E) has value T[i].
 * Monotonicity in i is itself asserted by the Python table test. */
static double T[127];

static void fill_table(void)
{
    for (int i = 0; i < 127; ++i)
        T[i] = orc_e4m3_decode((uint8_t)i);
}

/* The code index of the nearest magnitude, ties to the even index (even
 * mantissa), magnitudes >= 448 saturating to 0x7E.  a must be finite or +inf. */
static int nearest_index(double a)
{
    if (a >= T[126])
        return 126;
    int lo = 0, hi = 126; /* T[lo] <= a < T[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (T[mid] <= a)
            lo = mid;
        else
            hi = mid;
    }
    /* compare 2a with T[lo] + T[hi]: both sides are exact in double */
    double two_a = 2.0 * a, sum = T[lo] + T[hi];
    if (two_a < sum)
        return lo;
    if (two_a > sum)
        return hi;
    return (lo % 2 == 0) ? lo : hi;
}

/* Returns the number of mismatching patterns; *first gets the first one. */
uint64_t pin_encode_exhaustive(uint32_t *first)
{
    fill_table();
    uint64_t bad = 0;
    uint32_t first_bad = 0xFFFFFFFFu;
#pragma omp parallel for schedule(static, 1 << 20) reduction(+ : bad)
    for (int64_t i = 0; i < (int64_t)1 << 32; ++i) {
        uint32_t u = (uint32_t)i;
        float v = bits_f32(u);
        uint8_t c = orc_e4m3_encode(v);
        uint8_t want;
        if (isnan(v))
            want = 0x7F;
        else
            want = (uint8_t)((u >> 31 ? 0x80 : 0x00) | nearest_index(fabs((double)v)));
        if (c != want) {
            bad++;
#pragma omp critical
            if (u < first_bad)
                first_bad = u;
        }
    }
    *first = first_bad;
    return bad;
}

/* All (x, amax) with amax a positive finite bf16 and x any bf16 with |x| <= amax.
 * Checks, per pair:
 *   (1) s == fl32(amax / 448) computed as a correctly rounded double quotient
 *       (division rounded twice is exact for fp32 operands in double);
 *   (2) code == encode(fl32(x / s)), the quotient again via double;
 *   (3) x == amax gives code magnitude 0x7E;
 *   (4) |x - decode(code) * s| <= (ulp_E4M3(|x/s|)/2 + |x/s| * 2^-24) * s.
 * counts[0..3] receive the failure counts of (1)..(4); returns the pair count. */
uint64_t pin_quant_pairs(uint64_t counts[4])
{
    fill_table();
    uint64_t n = 0, c1 = 0, c2 = 0, c3 = 0, c4 = 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : n, c1, c2, c3, c4)
    for (int32_t ab = 1; ab <= 0x7F7F; ++ab) {
        float amax = bits_f32((uint32_t)ab << 16);
        float s = orc_group_scale(amax);
        if (s != (float)((double)amax / 448.0))
            c1++;
        for (int32_t xb = 0; xb <= ab; ++xb) {
            for (int sg = 0; sg < 2; ++sg) {
                float x = bits_f32(((uint32_t)xb << 16) | (sg ? 0x80000000u : 0u));
                uint8_t code = orc_quant_element(x, s);
                double qd = (double)x / (double)s;
                uint8_t want = orc_e4m3_encode((float)qd);
                if (code != want)
                    c2++;
                if (xb == ab && (code & 0x7F) != 0x7E)
                    c3++;
                double aq = fabs(qd);
                double half_ulp;
                if (aq < 0x1p-6) {
                    half_ulp = 0x1p-10;
                } else {
                    int e;
                    (void)frexp(aq, &e); /* aq in [2^(e-1), 2^e) */
                    half_ulp = ldexp(1.0, e - 1 - 4);
                }
                double err = fabs((double)x - orc_e4m3_decode(code) * (double)s);
                double bound = (half_ulp + aq * 0x1p-24) * (double)s;
                if (aq > 448.0)
                    bound = (aq - 448.0 + aq * 0x1p-24) * (double)s;
                if (err > bound)
                    c4++;
                n++;
            }
        }
    }
    counts[0] = c1;
    counts[1] = c2;
    counts[2] = c3;
    counts[3] = c4;
    return n;
}
