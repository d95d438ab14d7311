"""Pins of the oracle's fp64 block-scaled GEMMs (CPU only).

Exact rational brute force (Python ``fractions``) on tiny shapes, exact
integer special cases, one-hot rows, and agreement with a different
formulation (dense dequantization followed by one matmul) at moderate size.
Between them a dropped block, a transposed operand, a wrong scale index or a
mishandled partial tail block fails at least one test.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _rand_codes(rng, shape):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x7E  # no NaN codes
    return c


def _rand_scales(rng, shape):
    return (rng.random(shape) * 2.0 ** rng.integers(-12, 4, size=shape)).astype(np.float32) + np.float32(1e-6)


def _frac_value(code: int) -> Fraction:
    sign = -1 if code & 0x80 else 1
    e, m = (code >> 3) & 15, code & 7
    if e == 0:
        return sign * Fraction(m, 2 ** 9)
    return sign * Fraction(8 + m, 8) * (Fraction(2) ** (e - 7))


def _exact_block_gemm(a, sa, b, sb):
    """Y[r,c] = sum over blocks of sa*sb*sum(a*b), all in rationals."""
    R, L = a.shape
    C = b.shape[0]
    out = [[Fraction(0)] * C for _ in range(R)]
    mag = [[Fraction(0)] * C for _ in range(R)]  # sum of |block terms|, for the rounding bound
    for r in range(R):
        for c in range(C):
            tot, tabs = Fraction(0), Fraction(0)
            for cb in range((L + 127) // 128):
                part = sum((_frac_value(int(a[r, j])) * _frac_value(int(b[c, j]))
                            for j in range(cb * 128, min(L, cb * 128 + 128))), Fraction(0))
                term = Fraction(float(sa[cb, r])) * Fraction(float(sb[cb, c])) * part
                tot += term
                tabs += abs(term)
            out[r][c], mag[r][c] = tot, tabs
    return out, mag


@pytest.mark.parametrize("R,C,L", [(3, 2, 128), (2, 3, 256), (2, 2, 200), (1, 1, 1)])
def test_block_gemm_exact_rational(R, C, L):
    rng = np.random.default_rng(R * 100 + C * 10 + L)
    a, b = _rand_codes(rng, (R, L)), _rand_codes(rng, (C, L))
    LB = (L + 127) // 128
    sa, sb = _rand_scales(rng, (LB, R)), _rand_scales(rng, (LB, C))
    y = oracle.block_scaled_gemm(a, sa, b, sb)
    ex, mag = _exact_block_gemm(a, sa, b, sb)
    for r in range(R):
        for c in range(C):
            # fp64 rounds only the per-block scaling and the sum over blocks:
            # at most (LB + 1) units of 2^-53 of the summed magnitudes
            err = abs(Fraction(float(y[r, c])) - ex[r][c])
            assert err <= (LB + 1) * Fraction(1, 2 ** 53) * mag[r][c]


def _int_codes(rng, shape, lim=16):
    vals = rng.integers(-lim, lim + 1, size=shape).astype(np.float32)
    return oracle.e4m3_encode(vals), vals.astype(np.int64)


def test_fprop_integer_exact():
    rng = np.random.default_rng(21)
    M, N, K = 5, 256, 384
    qx, ix = _int_codes(rng, (M, K))
    qw, iw = _int_codes(rng, (N, K))
    sx = np.ones((K // 128, M), np.float32)
    sw = np.ones((N // 128, K // 128), np.float32)
    y = oracle.gemm_fprop(qx, sx, qw, sw)
    assert np.array_equal(y, (ix @ iw.T).astype(np.float64))


def test_dgrad_integer_exact():
    rng = np.random.default_rng(22)
    M, N, K = 7, 384, 256
    qdy, idy = _int_codes(rng, (M, N))
    qw, iw = _int_codes(rng, (N, K))
    sdy = np.ones((N // 128, M), np.float32)
    sw = np.ones((N // 128, K // 128), np.float32)
    y = oracle.gemm_dgrad(qdy, sdy, qw, sw)
    assert np.array_equal(y, (idy @ iw).astype(np.float64))


def test_wgrad_integer_exact_with_tail():
    rng = np.random.default_rng(23)
    M, N, K = 200, 128, 256  # partial last token block
    qdyT, idyT = _int_codes(rng, (N, M))
    qxT, ixT = _int_codes(rng, (K, M))
    MB = (M + 127) // 128
    y = oracle.gemm_wgrad(qdyT, np.ones((MB, N), np.float32), qxT, np.ones((MB, K), np.float32))
    assert np.array_equal(y, (idyT @ ixT.T).astype(np.float64))


def test_fprop_one_hot_rows_give_dequantized_weight_rows():
    rng = np.random.default_rng(24)
    N, K = 256, 256
    w = oracle.f32_to_bf16(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    qw, sw, _ = oracle.quant_weight_128x128(w)
    x = np.zeros((4, K), np.float32)
    hot = [0, 77, 128, 255]
    for i, k in enumerate(hot):
        x[i, k] = 1.0
    qx, sx = oracle.quant_rows_1x128(oracle.f32_to_bf16(x))
    y = oracle.gemm_fprop(qx, sx, qw, sw)
    wd = oracle.dequant_weight(qw, sw)
    for i, k in enumerate(hot):
        # x = 1 alone in its group: code 448 and s = fl32(1/448), so row i of Y is
        # column k of the dequantized W times 448 * s (exact in fp64)
        assert qx[i, k] == 0x7E
        assert np.array_equal(y[i], wd[:, k] * (448.0 * np.float64(sx[k // 128, i])))


def test_three_gemms_agree_with_dense_dequantized_matmul():
    rng = np.random.default_rng(25)
    M, N, K = 200, 384, 512
    x = oracle.f32_to_bf16(rng.standard_normal((M, K), dtype=np.float32))
    w = oracle.f32_to_bf16(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    dy = oracle.f32_to_bf16(rng.standard_normal((M, N), dtype=np.float32) * np.float32(1e-3))
    qx, sx = oracle.quant_rows_1x128(x)
    qw, sw, _ = oracle.quant_weight_128x128(w)
    qdy, sdy = oracle.quant_rows_1x128(dy)
    qdyT, sdyc = oracle.quant_cols_128x1(dy)
    qxT, sxc = oracle.quant_cols_128x1(x)
    wd = oracle.dequant_weight(qw, sw)

    y = oracle.gemm_fprop(qx, sx, qw, sw)
    assert np.allclose(y, oracle.dequant_rows(qx, sx) @ wd.T, rtol=1e-12, atol=1e-12)

    dx = oracle.gemm_dgrad(qdy, sdy, qw, sw)
    assert np.allclose(dx, oracle.dequant_rows(qdy, sdy) @ wd, rtol=1e-12, atol=1e-15)

    def deq_cols(qT, sc):  # [K, M] codes with [MB, K] scales -> [M, K] values
        v = oracle.dequant_codes(qT).T
        return v * np.repeat(sc.astype(np.float64), 128, axis=0)[:v.shape[0]]

    dw = oracle.gemm_wgrad(qdyT, sdyc, qxT, sxc)
    assert np.allclose(dw, deq_cols(qdyT, sdyc).T @ deq_cols(qxT, sxc), rtol=1e-12, atol=1e-15)

    # sampled rows / columns select the same entries
    rows, cols = np.array([0, 5, 199]), np.array([1, 130, 383])
    assert np.array_equal(oracle.gemm_fprop(qx, sx, qw, sw, rows=rows, cols=cols), y[np.ix_(rows, cols)])
    cols_k = np.array([0, 257, 511])
    assert np.array_equal(oracle.gemm_dgrad(qdy, sdy, qw, sw, rows=rows, cols=cols_k), dx[np.ix_(rows, cols_k)])
    assert np.array_equal(oracle.gemm_wgrad(qdyT, sdyc, qxT, sxc, rows=cols, cols=cols_k), dw[np.ix_(cols, cols_k)])

    # and the quantized product is close to the unquantized one (E4M3 relative error ~2^-4)
    yf = oracle.bf16_to_f32(x).astype(np.float64) @ oracle.bf16_to_f32(w).astype(np.float64).T
    assert np.linalg.norm(y - yf) / np.linalg.norm(yf) < 0.05
