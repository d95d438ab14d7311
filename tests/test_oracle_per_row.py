"""Pins of the oracle's per-token / per-channel FP8 path (CPU only).

QuRL notes, "损失函数 / 训练策略": weights quantized per output channel and
activations per token.  Here one group is a whole row over all K columns, with
the same scale rule (amax / 448, 1 for an all-zero row) and encoding as the
128-groups.  Independent restatements: a NumPy loop with torch's float8
conversion as the encoder, the K = 128 special case (which is the 1x128
quantizer, pinned elsewhere), invariants, and for the GEMM exact rationals and
the block-scaled oracle with the scales replicated over the K-blocks.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _bf16(rng, shape, std=1.0):
    return oracle.f32_to_bf16((rng.standard_normal(shape, dtype=np.float32) * np.float32(std)))


def _enc_torch(v: np.ndarray) -> np.ndarray:
    v = np.clip(v, -448.0, 448.0).astype(np.float32)  # torch is not satfinite
    return torch.from_numpy(np.ascontiguousarray(v)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("M,K", [(1, 1), (3, 7), (17, 640), (5, 4096)])
def test_per_row_matches_independent_loop(M, K):
    rng = np.random.default_rng(M * 31 + K)
    x = _bf16(rng, (M, K), std=0.02)
    if M > 2:
        x[2] = 0  # an all-zero row
    q, s = oracle.quant_per_row(x)
    xf = oracle.bf16_to_f32(x)
    for m in range(M):
        amax = np.float32(np.max(np.abs(xf[m])))
        sm = np.float32(1.0) if amax == 0 else amax / np.float32(448.0)
        assert s[m] == sm
        assert np.array_equal(q[m], _enc_torch(xf[m] / sm))
    if M > 2:
        assert s[2] == 1.0 and np.all(q[2] == 0)


def test_k128_reduces_to_1x128_groups():
    rng = np.random.default_rng(5)
    x = _bf16(rng, (300, 128))
    q, s = oracle.quant_per_row(x)
    q1, s1 = oracle.quant_rows_1x128(x)
    assert np.array_equal(q, q1) and np.array_equal(s, s1[0])


def test_every_nonzero_row_reaches_448_and_scales_are_covariant():
    rng = np.random.default_rng(6)
    x = _bf16(rng, (64, 1000), std=3.0)
    q, s = oracle.quant_per_row(x)
    assert np.all((q & 0x7F).max(axis=1) == 0x7E)  # |code| = 448 somewhere in every row
    for j in (-20, 7):
        xs = oracle.f32_to_bf16(oracle.bf16_to_f32(x) * np.float32(2.0 ** j))  # exact
        q2, s2 = oracle.quant_per_row(xs)
        assert np.array_equal(q2, q) and np.array_equal(s2, s * np.float32(2.0 ** j))


def _frac_value(code: int) -> Fraction:
    sign = -1 if code & 0x80 else 1
    e, m = (code >> 3) & 15, code & 7
    if e == 0:
        return sign * Fraction(m, 2 ** 9)
    return sign * Fraction(8 + m, 8) * (Fraction(2) ** (e - 7))


def _codes(rng, shape):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x7E
    return c


@pytest.mark.parametrize("M,N,K", [(2, 3, 5), (3, 2, 300)])
def test_gemm_per_channel_exact_rational(M, N, K):
    rng = np.random.default_rng(M + N + K)
    qx, qw = _codes(rng, (M, K)), _codes(rng, (N, K))
    sx = (rng.random(M) * 2.0 ** -8).astype(np.float32) + np.float32(1e-9)
    sw = (rng.random(N) * 2.0 ** -3).astype(np.float32) + np.float32(1e-9)
    y = oracle.gemm_per_channel(qx, sx, qw, sw)
    for m in range(M):
        for n in range(N):
            p = sum((_frac_value(int(qx[m, k])) * _frac_value(int(qw[n, k])) for k in range(K)), Fraction(0))
            exact = Fraction(float(sx[m])) * p * Fraction(float(sw[n]))
            # two roundings of an exact product in fp64
            assert abs(Fraction(float(y[m, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 51)


def test_gemm_per_channel_equals_block_gemm_with_replicated_scales():
    rng = np.random.default_rng(9)
    M, N, K = 40, 24, 640
    qx, qw = _codes(rng, (M, K)), _codes(rng, (N, K))
    sx = (rng.random(M) + 0.5).astype(np.float32)
    sw = (rng.random(N) + 0.5).astype(np.float32) * np.float32(2.0 ** -10)
    y = oracle.gemm_per_channel(qx, sx, qw, sw)
    KB = K // 128
    yb = oracle.block_scaled_gemm(qx, np.tile(sx, (KB, 1)), qw, np.tile(sw, (KB, 1)))
    assert np.allclose(y, yb, rtol=1e-12, atol=0)
    # and a transposed operand or swapped scale vectors would not match
    assert not np.allclose(oracle.gemm_per_channel(qx, sx[::-1].copy(), qw, sw), y, rtol=1e-6)


def test_gemm_per_channel_integer_special_case():
    rng = np.random.default_rng(10)
    lut = oracle.e4m3_lut()
    ints = [c for c in range(0x7F) if lut[c] == int(lut[c]) and abs(lut[c]) <= 16]  # 0x7F is NaN
    qx = rng.choice(ints, size=(7, 384)).astype(np.uint8) | (rng.integers(0, 2, (7, 384)) << 7).astype(np.uint8)
    qw = rng.choice(ints, size=(5, 384)).astype(np.uint8)
    y = oracle.gemm_per_channel(qx, np.ones(7, np.float32), qw, np.ones(5, np.float32))
    ref = lut[qx].astype(np.int64) @ lut[qw].astype(np.int64).T
    assert np.array_equal(y, ref.astype(np.float64))
