"""GPU parity of the AQN step (QeRL news article: channel-wise Gaussian noise
in the LayerNorm scale) through the C ABI: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_quantize_gb300 import rlq

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("K", [1, 127, 3584, 18944, 1_000_003])
@pytest.mark.parametrize("sigma", [0.0, 1e-3, 0.05])
def test_aqn_perturb_bit_exact(K, sigma):
    rng = np.random.default_rng(K)
    g = oracle.f32_to_bf16((1.0 + 0.05 * rng.standard_normal(K)).astype(np.float32))
    z = rng.standard_normal(K).astype(np.float32)
    gd = torch.from_numpy(g.view(np.int16)).cuda().view(torch.bfloat16)
    rlq.aqn_perturb_(gd, torch.from_numpy(z).cuda(), sigma)
    rlq.check()
    got = gd.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle.aqn_perturb(g, z, sigma))


def test_aqn_schedule_then_perturb_over_steps():
    """Steps of a schedule applied in sequence to the same norm scale (fresh noise
    each step), as a training loop would."""
    rng = np.random.default_rng(7)
    K, T = 4096, 6
    g = oracle.f32_to_bf16(np.ones(K, np.float32))
    gd = torch.from_numpy(g.view(np.int16)).cuda().view(torch.bfloat16)
    for t in range(T):
        z = rng.standard_normal(K).astype(np.float32)
        sigma = rlq.rlq_aqn_sigma(1e-2, 1e-3, t, T)
        rlq.aqn_perturb_(gd, torch.from_numpy(z).cuda(), sigma)
        g = oracle.aqn_perturb(g, z, sigma)
    rlq.check()
    assert np.array_equal(gd.view(torch.int16).cpu().numpy().view(np.uint16), g)
