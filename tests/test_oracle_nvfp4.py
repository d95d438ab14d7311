"""Pins of the oracle's NVFP4 weight quantizer (CPU only).

QeRL news article: NVFP4 is a hardware 4-bit float with two-level scaling, FP8
E4M3 block scales and an FP32 tensor scale, used for the policy weights.
Readings: E2M1 elements (RN-even, saturating to +-6), blocks of 16 consecutive
elements along K, tensor scale amax / (6 * 448) so that every block scale fits
E4M3.  Independent restatements: the closed-form E2M1 table, a vectorised
nearest-value search with ties to even, torch's float8 conversion for the block
scales, invariants and the closed-form dequantization error bound.
"""
import numpy as np
import pytest
import torch

import oracle

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _nearest_e2m1(v: np.ndarray) -> np.ndarray:
    """Vectorised RN-even onto the E2M1 grid with saturation, sign kept."""
    a = np.abs(v.astype(np.float64))
    d = np.abs(a[:, None] - E2M1[None, :])
    best = np.argmin(d, axis=1)
    # ties: argmin takes the lower code; move to the even one where the upper ties
    up = np.minimum(best + 1, 7)
    tie = np.isclose(d[np.arange(len(a)), up], d[np.arange(len(a)), best], rtol=0, atol=0) & (up != best)
    best = np.where(tie & (best % 2 == 1), up, best)
    best = np.where(a >= 6.0, 7, best)
    return (best | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def _enc_e4m3_torch(v: np.ndarray) -> np.ndarray:
    v = np.clip(v, -448.0, 448.0).astype(np.float32)
    return torch.from_numpy(np.ascontiguousarray(v)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e2m1_table():
    vals = [oracle.e2m1_decode(c) for c in range(16)]
    assert vals[:8] == list(E2M1) and vals[8:] == list(-E2M1)
    assert all(oracle.e2m1_encode(v) == c for c, v in enumerate(vals) if c != 8)
    assert oracle.e2m1_encode(-0.0) == 8


def test_e2m1_encode_against_independent_search():
    grid = np.concatenate([np.linspace(-8, 8, 200001, dtype=np.float32),
                           (E2M1[:-1] + E2M1[1:]).astype(np.float32) / 2,      # every midpoint
                           -(E2M1[:-1] + E2M1[1:]).astype(np.float32) / 2,
                           np.array([6.0, 6.5, 1e30, -1e30, 1e-40], np.float32)])
    got = np.array([oracle.e2m1_encode(float(v)) for v in grid], np.uint8)
    assert np.array_equal(got, _nearest_e2m1(grid))
    mids = (E2M1[:-1] + E2M1[1:]) / 2
    assert all(oracle.e2m1_encode(m) % 2 == 0 for m in mids)  # ties go to the even code


def _independent_nvfp4(w_bits):
    x = oracle.bf16_to_f32(w_bits)
    amax = np.float32(np.abs(x).max())
    st = np.float32(1.0) if amax == 0 else amax / np.float32(6.0 * 448.0)
    N, K = x.shape
    xb = x.reshape(N, K // 16, 16)
    ab = np.abs(xb).max(axis=2).astype(np.float32)
    sb = _enc_e4m3_torch((ab / np.float32(6.0)) / st)
    S = (oracle.dequant_codes(sb).astype(np.float32) * st).astype(np.float32)
    with np.errstate(invalid="ignore", divide="ignore"):  # all-zero blocks are set below
        r = (xb / S[:, :, None]).astype(np.float32)
    q = _nearest_e2m1(r.reshape(-1)).reshape(N, K)
    q = np.where(np.repeat(S == 0, 16, axis=1), np.where(np.signbit(x), 8, 0), q).astype(np.uint8)
    return q, sb, float(st)


@pytest.mark.parametrize("N,K,std", [(8, 64, 0.02), (33, 160, 1.0), (128, 512, 3e-3)])
def test_quant_nvfp4_matches_independent_loop(N, K, std):
    rng = np.random.default_rng(N + K)
    w = oracle.f32_to_bf16((rng.standard_normal((N, K)) * std).astype(np.float32))
    w[1, 16:32] = 0  # an all-zero block
    q, sb, st = oracle.quant_nvfp4(w)
    iq, isb, ist = _independent_nvfp4(w)
    assert st == ist and np.array_equal(sb, isb) and np.array_equal(q, iq)
    assert sb[1, 1] == 0 and np.all(q[1, 16:32] == 0)


def test_nvfp4_invariants_and_error_bound():
    rng = np.random.default_rng(5)
    w = oracle.f32_to_bf16((rng.standard_normal((64, 256)) * 0.05).astype(np.float32))
    q, sb, st = oracle.quant_nvfp4(w)
    assert (sb & 0x7F).max() <= 0x7E                       # block scales stay within E4M3 (<= 448)
    x = oracle.bf16_to_f32(w).astype(np.float64)
    blk = np.abs(x).reshape(64, 16, 16).max(axis=2)
    i, j = np.unravel_index(np.argmax(blk), blk.shape)
    assert sb[i, j] == 0x7E                                # the tensor's largest block maps to 448
    S = oracle.dequant_codes(sb).repeat(16, axis=1) * st
    xh = oracle.dequant_nvfp4(q, sb, st)
    r = np.abs(x) / S
    gap = np.where(r < 2, 0.5, np.where(r < 4, 1.0, 2.0))  # E2M1 spacing around |x/S|
    bound = np.where(r <= 6, 0.5 * gap, r - 6) * S
    assert np.all(np.abs(x - xh) <= bound * (1 + 1e-6) + 1e-30)
    assert np.all(r <= 6 * (1 + 2.0 ** -4) + 1e-6)         # block scale rounding can push a block max past 6 by <= 1/16


def test_nvfp4_scale_covariance_and_zero():
    rng = np.random.default_rng(6)
    w = oracle.f32_to_bf16((rng.standard_normal((16, 128)) * 0.1).astype(np.float32))
    q, sb, st = oracle.quant_nvfp4(w)
    for j in (-10, 5):
        w2 = oracle.f32_to_bf16(oracle.bf16_to_f32(w) * np.float32(2.0 ** j))
        q2, sb2, st2 = oracle.quant_nvfp4(w2)
        assert np.array_equal(q2, q) and np.array_equal(sb2, sb) and st2 == np.float32(st * 2.0 ** j)
    qz, sbz, stz = oracle.quant_nvfp4(np.zeros((4, 32), np.uint16))
    assert stz == 1.0 and np.all(qz == 0) and np.all(sbz == 0)


def _frac_e2m1(c):
    from fractions import Fraction
    v = Fraction(E2M1[c & 7]).limit_denominator(2)
    return -v if c & 8 else v


def test_weight_only_gemm_exact_rationals():
    """Tiny shapes in exact rationals: sum_k x[m,k] * e2m1(q) * e4m3(sb), times st."""
    from fractions import Fraction
    rng = np.random.default_rng(8)
    M, N, K = 3, 4, 48
    x = oracle.f32_to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    w = oracle.f32_to_bf16((rng.standard_normal((N, K)) * 0.3).astype(np.float32))
    q, sb, st = oracle.quant_nvfp4(w)
    y = oracle.gemm_nvfp4_weight_only(x, q, sb, st)
    xf = oracle.bf16_to_f32(x)
    lut = oracle.e4m3_lut()
    for m in range(M):
        for n in range(N):
            acc = sum((Fraction(float(xf[m, k])) * _frac_e2m1(int(q[n, k])) * Fraction(float(lut[sb[n, k // 16]]))
                       for k in range(K)), Fraction(0))
            exact = acc * Fraction(st)
            assert abs(Fraction(float(y[m, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 51) + Fraction(1, 2 ** 1074)


def test_weight_only_gemm_matches_dequantized_weight_and_integer_case():
    rng = np.random.default_rng(9)
    x = oracle.f32_to_bf16(rng.standard_normal((20, 64)).astype(np.float32))
    w = oracle.f32_to_bf16((rng.standard_normal((12, 64)) * 0.1).astype(np.float32))
    q, sb, st = oracle.quant_nvfp4(w)
    y = oracle.gemm_nvfp4_weight_only(x, q, sb, st)
    ref = oracle.bf16_to_f32(x).astype(np.float64) @ oracle.dequant_nvfp4(q, sb, st).T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-300)
    # integers: x in {-2..2}, every block scale 1 and st 1 -> exact integer products
    xi = rng.integers(-2, 3, size=(5, 32)).astype(np.float32)
    qi = rng.integers(0, 16, size=(6, 32)).astype(np.uint8)
    sbi = np.full((6, 2), 0x38, np.uint8)  # E4M3 code of 1.0
    yi = oracle.gemm_nvfp4_weight_only(oracle.f32_to_bf16(xi), qi, sbi, 1.0)
    lut4 = np.array([oracle.e2m1_decode(c) for c in range(16)])
    assert np.array_equal(yi, xi.astype(np.float64) @ lut4[qi].T)
    assert oracle.dequant_codes(np.array([0x38], np.uint8))[0] == 1.0
