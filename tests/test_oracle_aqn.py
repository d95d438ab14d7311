"""Pins of the oracle's AQN step (CPU only).

QeRL news article: adaptive quantization noise (AQN) adds channel-wise Gaussian
perturbations to the LayerNorm scale and decays them on an exponential
schedule.  Reading: gamma'[k] = bf16_RN(fl32(gamma[k] + fl32(sigma_t * z[k]))),
z[k] ~ N(0, 1) drawn by the caller, sigma_t geometric from sigma_start (t = 0)
to sigma_end (t = T - 1).  Independent restatements: NumPy fp32 arithmetic with
torch's bf16 conversion, closed forms of the schedule, the identities at zero
noise, and the noise statistics.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _bf16_bits_torch(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_zero_noise_is_the_identity():
    rng = np.random.default_rng(1)
    g = oracle.f32_to_bf16(rng.standard_normal(1000).astype(np.float32))
    z = rng.standard_normal(1000).astype(np.float32)
    assert np.array_equal(oracle.aqn_perturb(g, z, 0.0), g)
    assert np.array_equal(oracle.aqn_perturb(g, np.zeros(1000, np.float32), 0.3), g)


@pytest.mark.parametrize("sigma", [1e-3, 0.05, 2.0])
def test_matches_numpy_fp32_and_torch_bf16(sigma):
    rng = np.random.default_rng(2)
    K = 5000
    g = oracle.f32_to_bf16((1.0 + 0.1 * rng.standard_normal(K)).astype(np.float32))
    z = rng.standard_normal(K).astype(np.float32)
    noise = np.float32(sigma) * z                       # one fp32 rounding
    ref = _bf16_bits_torch(oracle.bf16_to_f32(g) + noise)  # one fp32 rounding, then bf16 RN
    assert np.array_equal(oracle.aqn_perturb(g, z, sigma), ref)


def test_schedule_endpoints_and_geometric_decay():
    s0, s1, T = 1e-2, 5e-4, 11
    sig = [oracle.aqn_sigma(s0, s1, t, T) for t in range(T)]
    assert sig[0] == np.float32(s0) and sig[-1] == np.float32(s1)
    ratio = (s1 / s0) ** (1.0 / (T - 1))
    for a, b in zip(sig[:-1], sig[1:]):
        assert math.isclose(b / a, ratio, rel_tol=1e-6)       # constant ratio: exponential decay
    assert oracle.aqn_sigma(s0, s1, 0, 1) == np.float32(s0)   # a single step
    assert oracle.aqn_sigma(s0, s0, 5, 9) == np.float32(s0)   # flat schedule


def test_noise_statistics():
    """gamma = 0 (so that bf16 resolves the noise): the perturbation has mean 0 and
    standard deviation sigma (5-sigma bounds over 10^6 channels)."""
    rng = np.random.default_rng(3)
    K, sigma = 1_000_000, 0.02
    z = rng.standard_normal(K).astype(np.float32)
    d = oracle.bf16_to_f32(oracle.aqn_perturb(np.zeros(K, np.uint16), z, sigma)).astype(np.float64)
    assert abs(d.mean()) < 5 * sigma / math.sqrt(K)
    assert abs(d.std() / sigma - 1.0) < 5 * math.sqrt(0.5 / K) + 2.0 ** -8  # sampling + bf16 rounding
