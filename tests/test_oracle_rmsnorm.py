"""Pins of the oracle's RMSNorm (the activation, with the UAQ scale folded into
the norm weight, that the 1x128 quantizer takes; QuRL notes, 关键设计 §1).

Reading (the pages give no formula for the norm): x = h / sqrt(mean(h^2) + eps)
* gamma with fp32 steps, the sum of squares accumulated by fused multiply-adds
in index order, one rounding to bf16.  Pinned against:

* closed forms: constant rows of +-2^j give rstd = 2^-j and x = +-gamma exactly;
* exact arithmetic: where the sum of squares is exact (small integers), every
  later step is one correctly rounded operation, reproduced here in fp64 and
  rounded once to fp32 (for +, /, sqrt that double rounding is exact, since
  53 >= 2 * 24 + 2);
* the index order of the sum: a row whose squares are [2^24, 1, 1, ...] keeps
  2^24 (each +1 is a tie to even), which no other order gives;
* an error bound against the exact value (50-digit decimal arithmetic): within
  half a bf16 ulp plus the fp32 steps' error, and mostly the correctly rounded bf16;
* invariants: 2^j scaling of h leaves x unchanged (eps = 0); a power-of-two fold
  of gamma scales x exactly, so the 1x128 codes are unchanged and the scales scale;
* torch's rms_norm (an independent library) agrees to within one bf16 ulp.
"""
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_quantize_gb300 import inputs as I


def _f32(bits):
    return oracle.bf16_to_f32(bits)


def _bf(v):
    return I.to_bf16_bits(np.asarray(v, np.float32))


def _gamma(K, seed=0):
    return _bf(np.random.default_rng(seed).uniform(0.5, 2.0, K))


@pytest.mark.parametrize("j", [-10, 0, 3])
def test_constant_rows_closed_form(j):
    K = 256
    c = 2.0 ** j
    h = _bf(np.stack([np.full(K, c), np.full(K, -c)]))
    g = _gamma(K)
    x, rstd = oracle.rmsnorm(h, g, 0.0)
    assert np.all(rstd == np.float32(2.0 ** -j))
    assert np.array_equal(x[0], g)
    assert np.array_equal(x[1], g ^ np.uint16(0x8000))


@pytest.mark.parametrize("eps", [0.0, 1e-5, 0.25])
def test_rstd_of_exact_sums(eps):
    """Small integers: the fp32 sum of squares is exact (<= 64 * 4096 < 2^24),
    so rstd is fl32(1 / fl32(sqrt(fl32(fl32(S / K) + eps)))) with each step
    correctly rounded, reproduced in fp64 with one rounding per step."""
    K = 4096
    rng = np.random.default_rng(1)
    h = _bf(rng.integers(-8, 9, size=(64, K)).astype(np.float32))
    _, rstd = oracle.rmsnorm(h, _gamma(K), eps)
    S = (_f32(h).astype(np.float64) ** 2).sum(axis=1)  # exact: integers below 2^53
    f = np.float32
    ms = f(S / K)
    d = f(np.sqrt(np.float64(f(np.float64(ms) + np.float64(f(eps))))))
    r = f(1.0 / np.float64(d))
    assert np.array_equal(rstd, r)


def test_sum_runs_in_index_order():
    """Squares [2^24, 1, 1, ...]: in index order every +1 is a tie that rounds
    back to 2^24; ones-first or pairwise orders give a larger sum."""
    K = 128
    row = np.ones(K, np.float32)
    row[0] = 4096.0  # 4096^2 = 2^24
    h = _bf(row[None, :])
    _, rstd = oracle.rmsnorm(h, _bf(np.ones(K)), 0.0)
    f = np.float32
    expect = f(1.0 / np.float64(f(np.sqrt(np.float64(f(2.0 ** 24 / K))))))
    assert rstd[0] == expect
    larger = f(1.0 / np.float64(f(np.sqrt(np.float64(f((2.0 ** 24 + K - 1) / K))))))
    assert expect != larger  # the test separates the orders


def _ulp_bf16(v):
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
    return 2.0 ** (e - 7)


@pytest.mark.parametrize("K,eps", [(128, 1e-6), (4096, 1e-6), (4096, 0.25), (3584, 1e-5)])
def test_error_bound_against_exact_values(K, eps):
    getcontext().prec = 50
    rng = np.random.default_rng(K)
    M = 6
    hf = rng.standard_normal((M, K)).astype(np.float32) * np.array([1e-3, 0.1, 1, 3, 50, 1e3], np.float32)[:, None]
    h = _bf(hf)
    g = _gamma(K, 2)
    x, _ = oracle.rmsnorm(h, g, eps)
    hv, gv = _f32(h), _f32(g)
    exact = np.empty((M, K))
    for m in range(M):
        hd = [Decimal(float(v)) for v in hv[m]]
        ms = sum(v * v for v in hd) / K + Decimal(float(np.float32(eps)))
        inv = 1 / ms.sqrt()
        exact[m] = [float(v * inv * Decimal(float(gk))) for v, gk in zip(hd, gv)]
    got = _f32(x).astype(np.float64)
    # fp32 steps: the sum of K squares (<= K * 2^-24 relative), a few roundings
    slack = (K + 8) * 2.0 ** -24 * np.abs(exact)
    assert np.all(np.abs(got - exact) <= 0.5 * _ulp_bf16(exact) + slack)
    nearest = _f32(_bf(exact.astype(np.float32)))  # fp64 -> fp32 -> bf16: a further rounding, enough here
    assert np.mean(got == nearest) > 0.99


@pytest.mark.parametrize("j", [-4, 5])
def test_power_of_two_scaling_of_h_is_invisible(j):
    K = 512
    h = _bf(np.random.default_rng(3).standard_normal((16, K)))
    g = _gamma(K, 3)
    x0, r0 = oracle.rmsnorm(h, g, 0.0)
    x1, r1 = oracle.rmsnorm(_bf(_f32(h) * 2.0 ** j), g, 0.0)
    assert np.array_equal(x0, x1)
    assert np.array_equal(r1, r0 * np.float32(2.0 ** -j))


def test_power_of_two_fold_into_gamma_scales_x_and_keeps_codes():
    """QuRL notes, 关键设计 §1: s folded into the norm weight.  With s = 4 the
    folded gamma is exactly 4 gamma, so x is exactly 4 x: the 1x128 and 128x1
    codes are unchanged and every scale is multiplied by 4."""
    M, K = 200, 384
    h = _bf(np.random.default_rng(4).standard_normal((M, K)))
    g = _gamma(K, 4)
    s = np.full(K, 4.0, np.float32)
    _, g4 = oracle.uaq_fold(np.zeros((0, K), np.uint16), s, g[None, :])
    x0, _ = oracle.rmsnorm(h, g, 1e-6)
    x1, _ = oracle.rmsnorm(h, g4[0], 1e-6)
    assert np.array_equal(_f32(x1), 4 * _f32(x0))
    q0, s0 = oracle.quant_rows_1x128(x0)
    q1, s1 = oracle.quant_rows_1x128(x1)
    assert np.array_equal(q0, q1) and np.array_equal(s1, 4 * s0)
    c0, t0 = oracle.quant_cols_128x1(x0)
    c1, t1 = oracle.quant_cols_128x1(x1)
    assert np.array_equal(c0, c1) and np.array_equal(t1, 4 * t0)


def test_torch_rms_norm_agrees_within_one_ulp():
    if not hasattr(torch.nn.functional, "rms_norm"):
        pytest.skip("torch without rms_norm")
    M, K, eps = 64, 4096, 1e-6
    h = _bf(np.random.default_rng(5).standard_normal((M, K)) * 2)
    g = _gamma(K, 5)
    x, _ = oracle.rmsnorm(h, g, eps)
    ht = torch.from_numpy(_f32(h))
    ref = torch.nn.functional.rms_norm(ht, (K,), weight=torch.from_numpy(_f32(g)), eps=eps)
    rb = ref.to(torch.bfloat16).float().numpy().astype(np.float64)
    got = _f32(x).astype(np.float64)
    assert np.all(np.abs(got - rb) <= _ulp_bf16(rb) * 1.0001)
    assert np.mean(got == rb) > 0.99
