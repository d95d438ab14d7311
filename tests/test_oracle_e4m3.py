"""Pins of the oracle's E4M3 codec and bf16 rounding (CPU only).

The E4M3 format facts come from the OCP OFP8 specification (tests/golden/e4m3.txt);
torch's and ml_dtypes' float8_e4m3fn conversions serve as independent libraries
(both are RN-even but return NaN past the format's range instead of saturating,
so they are compared only where |v| < 464).
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from golden_util import load
from pins_c import build as pins_build

G = load("e4m3.txt")


def test_decode_table_matches_ocp_parameters():
    v = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.isnan(v[G["nan_code_pos"]]) and np.isnan(v[G["nan_code_neg"]])
    assert int(np.isfinite(v).sum()) == int(G["finite_codes"])
    assert v[G["max_normal_code"]] == G["max_normal"]
    assert v[G["min_normal_code"]] == G["min_normal"]
    assert v[0x07] == G["max_subnormal"]
    assert v[0x01] == G["min_subnormal"]
    assert v[0x00] == 0.0 and math.copysign(1.0, v[0x80]) == -1.0
    # bias: code with exponent field 7 and mantissa 0 is 1.0
    assert v[int(G["exponent_bias"]) << 3] == 1.0
    # magnitudes strictly increase with the code index; negative half mirrors
    mags = v[:0x7F]
    assert np.all(np.diff(mags) > 0)
    assert np.array_equal(v[0x80:0xFF], -v[:0x7F])


def test_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(ours), fin)
    assert np.array_equal(ours[fin], ref[fin])


def test_decode_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    ref = np.arange(256, dtype=np.uint8).view(ml.float8_e4m3fn).astype(np.float64)
    ours = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    fin = np.isfinite(ref)
    assert np.array_equal(ours[fin], ref[fin])


def test_encode_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_encode_saturates_at_448():
    big = np.array([448.0, 449.0, 463.99, 464.0, 480.0, 1e30, np.inf], np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    # just below 448: between 416 (0x7D) and 448 (0x7E), midpoint 432 ties to even 0x7E
    assert oracle.e4m3_encode(np.array([431.99, 432.0, 432.01], np.float32)).tolist() == [0x7D, 0x7E, 0x7E]


def test_encode_signed_zero_and_nan():
    vals = np.array([0.0, -0.0, 1e-30, -1e-30, 2.0 ** -10, -(2.0 ** -10)], np.float32)
    # 2^-10 is the midpoint between 0 and 2^-9: ties to even -> zero
    assert oracle.e4m3_encode(vals).tolist() == [0x00, 0x80, 0x00, 0x80, 0x00, 0x80]
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


def test_encode_ties_to_even_at_every_midpoint():
    v = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    for i in range(0x7E):
        mid = np.float32((v[i] + v[i + 1]) / 2)  # exact: a midpoint of two E4M3 values
        assert float(mid) == (v[i] + v[i + 1]) / 2
        even = i if i % 2 == 0 else i + 1
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(np.inf))
        got = oracle.e4m3_encode(np.array([below, mid, above], np.float32)).tolist()
        assert got == [i, even, i + 1], (i, got)


def _torch_e4m3(vals: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(vals).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_encode_matches_torch_on_all_bf16_and_random_fp32():
    rng = np.random.default_rng(12345)
    all_bf16 = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    rnd = rng.integers(0, 2 ** 32, size=1 << 22, dtype=np.uint64).astype(np.uint32).view(np.float32)
    # dense sample around the E4M3 grid: every code value times (1 + small offsets)
    grid = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float32)
    ulps = np.arange(-64, 65, dtype=np.int32)
    near = (grid.view(np.int32)[:, None] + ulps[None, :]).reshape(-1).view(np.float32)
    vals = np.concatenate([all_bf16, rnd, near, -near])
    vals = vals[np.isfinite(vals) & (np.abs(vals) < 464.0)]
    assert np.array_equal(oracle.e4m3_encode(vals), _torch_e4m3(vals))


def test_encode_matches_ml_dtypes_random():
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(7)
    vals = (rng.standard_normal(1 << 20) * rng.choice([1e-3, 1.0, 100.0], 1 << 20)).astype(np.float32)
    vals = vals[np.abs(vals) < 464.0]
    ref = vals.astype(ml.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(oracle.e4m3_encode(vals), ref)


@pytest.mark.slow
def test_encode_exhaustive_nearest_ties_even_satfinite():
    """All 2^32 fp32 patterns: the code is the nearest E4M3 value (ties to the
    even mantissa), clamped to +-448, sign kept; NaN -> 0x7F."""
    lib = pins_build.load()
    first = ctypes.c_uint32(0)
    bad = lib.pin_encode_exhaustive(ctypes.byref(first))
    assert bad == 0, f"{bad} mismatches, first pattern 0x{first.value:08x}"


# ------------------------------------------------------------- bf16 RN ---

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(99)
    bits = rng.integers(0, 2 ** 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    # ties: low half exactly 0x8000 with both parities of the kept half
    ties = (rng.integers(0, 2 ** 16, size=1 << 14, dtype=np.uint32) << 16) | 0x8000
    vals = np.concatenate([bits, ties]).view(np.float32)
    vals = vals[~np.isnan(vals)]
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f32_to_bf16(vals), ref)


def test_bf16_roundtrip_exact():
    b = np.arange(65536, dtype=np.uint16)
    f = oracle.bf16_to_f32(b)
    keep = ~np.isnan(f)
    assert np.array_equal(oracle.f32_to_bf16(f[keep]), b[keep])
