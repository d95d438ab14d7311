"""Pins of the oracle's group quantizers (CPU only).

Independent restatement used here: per-group loops in NumPy (fp32 IEEE
division) with torch's float8_e4m3fn conversion as the encoder — a different
library and a different loop structure from the C oracle — plus exhaustive
enumeration, invariants and closed-form bounds.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from golden_util import load
from pins_c import build as pins_build

GR = load("granularity.txt")
E = load("e4m3.txt")


def _bf16(rng, shape, std=1.0):
    v = (rng.standard_normal(shape, dtype=np.float32) * np.float32(std))
    return oracle.f32_to_bf16(v)


def _enc_torch(v: np.ndarray) -> np.ndarray:
    v = np.clip(v, -448.0, 448.0).astype(np.float32)  # torch is not satfinite
    return torch.from_numpy(np.ascontiguousarray(v)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _group(vals_f32: np.ndarray):
    amax = np.float32(np.max(np.abs(vals_f32))) if vals_f32.size else np.float32(0)
    s = np.float32(1.0) if amax == 0 else np.float32(amax) / np.float32(E["max_normal"])
    return s, _enc_torch(vals_f32 / s)


def test_rowwise_matches_independent_loop():
    rng = np.random.default_rng(1)
    M, K = 37, 512
    x = _bf16(rng, (M, K))
    x[3, 128:256] = 0  # an all-zero group
    q, s = oracle.quant_rows_1x128(x)
    assert q.shape == (M, K) and s.shape == (K // 128, M)
    xf = oracle.bf16_to_f32(x)
    g = int(GR["act_group_cols"])
    for m in range(M):
        for kb in range(K // g):
            sg, cg = _group(xf[m, kb * g:(kb + 1) * g])
            assert s[kb, m] == sg
            assert np.array_equal(q[m, kb * g:(kb + 1) * g], cg)
    assert s[1, 3] == 1.0 and np.all(q[3, 128:256] == 0)


@pytest.mark.parametrize("M", [1, 16, 127, 128, 200, 300])
def test_colwise_matches_independent_loop(M):
    rng = np.random.default_rng(M)
    K = 256
    x = _bf16(rng, (M, K), std=1e-3)
    qT, sc = oracle.quant_cols_128x1(x)
    g = int(GR["wgrad_second_group_rows"])
    MB = (M + g - 1) // g
    assert qT.shape == (K, M) and sc.shape == (MB, K)
    xf = oracle.bf16_to_f32(x)
    for k in range(K):
        for mb in range(MB):
            sg, cg = _group(xf[mb * g:min(M, (mb + 1) * g), k])
            assert sc[mb, k] == sg
            assert np.array_equal(qT[k, mb * g:min(M, (mb + 1) * g)], cg)


def test_weight_blocks_match_independent_loop():
    rng = np.random.default_rng(3)
    N, K = 384, 256
    w = _bf16(rng, (N, K), std=0.02)
    w[128:256, 0:128] = 0
    q, s, qT = oracle.quant_weight_128x128(w, transposed=True)
    assert s.shape == (N // 128, K // 128)
    wf = oracle.bf16_to_f32(w)
    br, bc = int(GR["weight_block_rows"]), int(GR["weight_block_cols"])
    for nb in range(N // br):
        for kb in range(K // bc):
            blk = wf[nb * br:(nb + 1) * br, kb * bc:(kb + 1) * bc]
            sg, cg = _group(blk.reshape(-1))
            assert s[nb, kb] == sg
            assert np.array_equal(q[nb * br:(nb + 1) * br, kb * bc:(kb + 1) * bc].reshape(-1), cg)
    assert np.array_equal(qT, q.T)
    assert s[1, 0] == 1.0


@pytest.mark.slow
def test_element_map_exhaustive_over_bf16_pairs():
    """Every (x, amax) bf16 pair with |x| <= amax: scale rule, fp32 division,
    the 448 invariant and the dequantization error bound."""
    lib = pins_build.load()
    counts = (ctypes.c_uint64 * 4)()
    n = lib.pin_quant_pairs(counts)
    assert n > 2 * 10 ** 9 // 2
    assert list(counts) == [0, 0, 0, 0], list(counts)


def test_element_map_matches_torch_division_sample():
    rng = np.random.default_rng(5)
    amax_bits = rng.integers(1, 0x7F80, size=1 << 18).astype(np.uint16)
    amax = oracle.bf16_to_f32(amax_bits)
    frac = rng.random(1 << 18).astype(np.float32) * (2 * rng.integers(0, 2, 1 << 18) - 1).astype(np.float32)
    x = oracle.bf16_to_f32(oracle.f32_to_bf16(amax * frac))
    s = np.where(amax == 0, np.float32(1), amax / np.float32(448)).astype(np.float32)
    ours = oracle.quant_element(x, s)
    xt = torch.from_numpy(x)
    st = torch.from_numpy(s)
    ref = torch.clamp(xt / st, -448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_every_nonzero_group_hits_448():
    """For each of the 32639 positive finite bf16 amax values the amax element
    itself quantizes to +-448 (subnormal scales included)."""
    amax = oracle.bf16_to_f32(np.arange(1, 0x7F80, dtype=np.uint16))
    s = np.array([oracle.group_scale(float(a)) for a in amax[::97]], np.float32)
    assert np.all(oracle.quant_element(amax[::97], s) == 0x7E)
    s_all = (amax / np.float32(448)).astype(np.float32)
    assert np.all(oracle.quant_element(amax, s_all) == E["max_normal_code"])
    assert np.all(oracle.quant_element(-amax, s_all) == 0xFE)
    assert int((s_all < np.float32(2.0 ** -126)).sum()) > 1000  # subnormal scales are exercised


@pytest.mark.parametrize("j", [-24, -3, 5, 20])
def test_scale_covariance_under_powers_of_two(j):
    rng = np.random.default_rng(11)
    x = _bf16(rng, (64, 384))
    xf = oracle.bf16_to_f32(x)
    x2 = oracle.f32_to_bf16(xf * np.float32(2.0 ** j))
    assert np.array_equal(oracle.bf16_to_f32(x2), xf * np.float32(2.0 ** j))  # exact scaling
    q, s = oracle.quant_rows_1x128(x)
    q2, s2 = oracle.quant_rows_1x128(x2)
    assert np.array_equal(q, q2)
    assert np.array_equal(s2, s * np.float32(2.0 ** j))
    qT, sc = oracle.quant_cols_128x1(x)
    qT2, sc2 = oracle.quant_cols_128x1(x2)
    assert np.array_equal(qT, qT2) and np.array_equal(sc2, sc * np.float32(2.0 ** j))


def test_special_scales():
    # a group whose amax is 448 has scale 1 and its codes are plain encodes
    rng = np.random.default_rng(4)
    v = np.clip(rng.standard_normal(128).astype(np.float32) * 100, -447, 447)
    v[17] = -448.0
    x = oracle.f32_to_bf16(v)[None, :]
    q, s = oracle.quant_rows_1x128(x)
    assert s[0, 0] == 1.0
    assert np.array_equal(q[0], oracle.e4m3_encode(oracle.bf16_to_f32(x[0])))
    # all-zero group: scale 1, codes are signed zeros
    z = oracle.f32_to_bf16(np.array([0.0, -0.0] * 64, np.float32))[None, :]
    qz, sz = oracle.quant_rows_1x128(z)
    assert sz[0, 0] == 1.0 and qz[0].tolist() == [0x00, 0x80] * 64


def test_dequant_error_bound_random():
    rng = np.random.default_rng(8)
    x = _bf16(rng, (256, 1024))
    q, s = oracle.quant_rows_1x128(x)
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    deq = oracle.dequant_rows(q, s)
    srep = np.repeat(s.T.astype(np.float64), 128, axis=1)
    err = np.abs(xf - deq)
    # relative 2^-4 for E4M3 normals (half of the 2^-3 mantissa step), 2^-10 * s below 2^-6 * s
    bound = np.maximum(np.abs(xf) * 2.0 ** -4, 2.0 ** -10 * srep) * (1 + 2.0 ** -20)
    assert np.all(err <= bound)
