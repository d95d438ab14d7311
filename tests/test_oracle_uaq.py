"""Pins of the oracle's UAQ fold and of the s^2 argument behind it (CPU only).

QuRL notes, 关键设计 §1: WX = (W/s)(sX), s applied per column of W and per row
of the previous activation; folding s > 1 divides the weight quantization error
by s and multiplies the (activation-side) update by s, an s^2 gain in
signal-to-noise.  Page figures are read from tests/golden/uaq.txt.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from golden_util import load

U = load("uaq.txt")


def test_invariant_scaling_identity_exact_rationals():
    rng = np.random.default_rng(31)
    N, K, M = 3, 5, 4
    W = [[Fraction(int(v), 97) for v in row] for row in rng.integers(-50, 50, (N, K))]
    X = [[Fraction(int(v), 89) for v in row] for row in rng.integers(-50, 50, (M, K))]
    s = [Fraction(3, 2), Fraction(7, 3), Fraction(4), Fraction(5, 4), Fraction(11, 7)]
    Wf = [[W[n][k] / s[k] for k in range(K)] for n in range(N)]  # per input channel (column of W)
    Xf = [[X[m][k] * s[k] for k in range(K)] for m in range(M)]  # same channel of the activation
    for m in range(M):
        for n in range(N):
            assert sum(X[m][k] * W[n][k] for k in range(K)) == sum(Xf[m][k] * Wf[n][k] for k in range(K))


def test_fold_matches_independent_fp32_and_torch_bf16():
    rng = np.random.default_rng(32)
    N, K, R = 64, 384, 3
    w = oracle.f32_to_bf16(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    p = oracle.f32_to_bf16(rng.standard_normal((R, K), dtype=np.float32))
    s = rng.uniform(1.5, 4.0, K).astype(np.float32)
    wf, pf = oracle.uaq_fold(w, s, p)
    # independent: numpy fp32 arithmetic, torch's bf16 rounding
    w32 = oracle.bf16_to_f32(w) / s[None, :]
    p32 = oracle.bf16_to_f32(p) * s[None, :]
    ref_w = torch.from_numpy(w32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref_p = torch.from_numpy(p32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wf, ref_w) and np.array_equal(pf, ref_p)
    # the input arrays are untouched (the oracle folds copies)
    assert not np.array_equal(wf, w)


def test_fold_rounding_bound_and_power_of_two_exactness():
    rng = np.random.default_rng(33)
    N, K = 32, 256
    w = oracle.f32_to_bf16(rng.standard_normal((N, K), dtype=np.float32))
    s = rng.uniform(1.5, 4.0, K).astype(np.float32)
    wf, _ = oracle.uaq_fold(w, s)
    exact = oracle.bf16_to_f32(w).astype(np.float64) / s.astype(np.float64)
    got = oracle.bf16_to_f32(wf).astype(np.float64)
    assert np.all(np.abs(got - exact) <= np.abs(exact) * 2.0 ** -8 * (1 + 1e-6))  # bf16 half-ulp + fp32
    s4 = np.full(K, 4.0, np.float32)
    wf4, _ = oracle.uaq_fold(w, s4)
    assert np.array_equal(oracle.bf16_to_f32(wf4), oracle.bf16_to_f32(w) / np.float32(4))


def test_fold_by_power_of_two_commutes_with_quantization():
    """s = 4 on every channel (the tiny single-linear workload): quantizing the
    folded tensors gives the same codes, activation scales x4 and weight
    scales /4 exactly, hence the same block-scaled FProp output."""
    rng = np.random.default_rng(0)
    x = oracle.f32_to_bf16(rng.standard_normal((128, 256), dtype=np.float32))
    w = oracle.f32_to_bf16(rng.standard_normal((256, 256), dtype=np.float32) * np.float32(0.02))
    s = np.full(256, 4.0, np.float32)
    wf, xf = oracle.uaq_fold(w, s, x)
    qx, sx = oracle.quant_rows_1x128(x)
    qxf, sxf = oracle.quant_rows_1x128(xf)
    qw, sw, _ = oracle.quant_weight_128x128(w)
    qwf, swf, _ = oracle.quant_weight_128x128(wf)
    assert np.array_equal(qx, qxf) and np.array_equal(sxf, sx * np.float32(4))
    assert np.array_equal(qw, qwf) and np.array_equal(swf, sw / np.float32(4))
    assert np.array_equal(oracle.gemm_fprop(qx, sx, qw, sw), oracle.gemm_fprop(qxf, sxf, qwf, swf))


def _quant_blocks_f32(w32: np.ndarray):
    """128x128 block quantization of an fp32 weight (the master copy), using the
    oracle's element map and scale rule.  Returns (codes, per-element scale)."""
    N, K = w32.shape
    blk = w32.reshape(N // 128, 128, K // 128, 128)
    amax = np.abs(blk).max(axis=(1, 3))
    s = np.where(amax == 0, np.float32(1), amax / np.float32(448)).astype(np.float32)
    sfull = np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)
    return oracle.quant_element(w32, sfull), sfull


def test_s_squared_identity_exact_for_power_of_two_s():
    """With s a power of two, quantizing W/s + s*d equals quantizing W + s^2*d
    code for code: the update the quantized model sees grows by s^2."""
    rng = np.random.default_rng(34)
    N, K = 256, 512
    W = rng.standard_normal((N, K)) * 0.02
    d = U["update_lr"] * rng.standard_normal((N, K)) * U["update_grad_hi"]
    for s in (2.0, 4.0):
        lhs, _ = _quant_blocks_f32((W / s + s * d).astype(np.float32))
        rhs, _ = _quant_blocks_f32((W + s * s * d).astype(np.float32))
        assert np.array_equal(lhs, rhs)


@pytest.mark.slow
def test_s_squared_transmitted_update_statistics():
    """The update that survives quantization grows by s^2 (QuRL's SNR argument).

    Measured in the original frame: T(s) = sum_i sign(d_i) * (deq Q(W/s + s d)
    - deq Q(W/s))_i * s, i.e. the dequantized change of the folded weight seen
    through the s-scaled activation, projected on the update's direction.  In
    expectation over the weights' position inside a code cell this equals
    sum |s^2 d_i|, so T(2)/T(1) = 4 within 5 standard deviations estimated
    from the per-element contributions."""
    rng = np.random.default_rng(35)
    N, K = 2048, 4096
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32).astype(np.float64)
    lo, hi = U["update_grad_lo"], U["update_grad_hi"]
    G = rng.standard_normal((N, K)) * rng.uniform(lo, hi, (N, 1))
    d = U["update_lr"] * G
    assert 0.1 * U["update_magnitude"] < np.median(np.abs(d)) < 10 * U["update_magnitude"]
    T, V = {}, {}
    for s in (1.0, 2.0):
        q0, s0 = _quant_blocks_f32((W / s).astype(np.float32))
        q1, s1 = _quant_blocks_f32((W / s + s * d).astype(np.float32))
        change = (oracle.dequant_codes(q1) * s1 - oracle.dequant_codes(q0) * s0) * s
        t = np.sign(d) * change
        T[s], V[s] = float(t.sum()), float((t ** 2).sum())
    ratio = T[2.0] / T[1.0]
    expect = 2.0 ** U["snr_gain_power"]
    sigma = ratio * np.sqrt(V[1.0] / T[1.0] ** 2 + V[2.0] / T[2.0] ** 2)
    assert abs(ratio - expect) < 5 * sigma, (T, ratio, sigma)
    assert sigma < 0.1 * expect  # the test has power to tell s^2 from s
    # the quantized model's error in the original frame is unchanged by folding
    # (power-of-two s commutes with quantization), so the SNR gain is the s^2 above
    qa, sa = _quant_blocks_f32(W.astype(np.float32))
    qb, sb = _quant_blocks_f32((W / 2.0).astype(np.float32))
    assert np.array_equal(qa, qb) and np.array_equal(sb * 2, sa)


def test_quantization_error_scale_matches_pages():
    """The weight quantization error of N(0,0.02) weights under 128x128 E4M3
    blocks sits inside the range the pages quote (1e-3 .. 1e-1 is the norm of
    the error; elementwise it is far above the ~1e-7 update)."""
    rng = np.random.default_rng(36)
    w = oracle.f32_to_bf16(rng.standard_normal((256, 256), dtype=np.float32) * np.float32(0.02))
    q, s, _ = oracle.quant_weight_128x128(w)
    err = oracle.dequant_weight(q, s) - oracle.bf16_to_f32(w)
    rms_err = float(np.sqrt(np.mean(err ** 2)))
    assert rms_err > 100 * U["update_magnitude"]
    row_err_norm = float(np.linalg.norm(err) / np.sqrt(256))  # per 256-wide row
    assert U["quant_err_lo"] <= row_err_norm <= U["quant_err_hi"]
