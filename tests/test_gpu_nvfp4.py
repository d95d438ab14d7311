"""GPU parity of the NVFP4 weight quantizer (QeRL news article: 4-bit floats,
E4M3 block scales, FP32 tensor scale) through the C ABI: element codes, block
codes and the tensor scale bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_quantize_gb300 import inputs as I
from fp8_block_scaled_quantize_gb300 import rlq
from gpu_util import normal_bits, np_, to_dev

pytestmark = pytest.mark.gpu


def _unpack(qp: np.ndarray) -> np.ndarray:
    lo, hi = qp & 0xF, qp >> 4
    return np.stack([lo, hi], axis=-1).reshape(qp.shape[0], -1)


def _check(w_bits, q, sb, st):
    oq, osb, ost = oracle.quant_nvfp4(w_bits)
    assert np_(st)[0] == np.float32(ost), "tensor scale differs"
    assert np.array_equal(np_(sb), osb), "block scales differ"
    assert np.array_equal(_unpack(np_(q)), oq), "element codes differ"


@pytest.mark.parametrize("N,K,std", [(1, 16, 1.0), (7, 48, 0.02), (128, 512, 3e-3), (14336, 4096, 0.02)])
def test_nvfp4_parity(N, K, std):
    w = normal_bits(70, (N, K), std=std)
    q, sb, st = rlq.quant_nvfp4(to_dev(w))
    rlq.check()
    _check(w, q, sb, st)


def test_nvfp4_edge_blocks():
    """Blocks 2^-40 .. 2^20 apart (the smallest flush to zero), all-zero and
    signed-zero blocks, exact E2M1 midpoints, and the zero tensor."""
    rng = np.random.default_rng(71)
    N, K = 64, 256
    v = rng.standard_normal((N, K)).astype(np.float32)
    v *= np.exp2(rng.integers(-40, 21, size=(N, K // 16))).repeat(16, axis=1).astype(np.float32)
    v[0, :16] = 0.0
    v[0, 16:32] = -0.0
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32)
    v[1, :16] = np.concatenate([mids, -mids])  # block amax 6: block scale 1 * st when st makes it exact
    w = I.to_bf16_bits(v)
    q, sb, st = rlq.quant_nvfp4(to_dev(w))
    rlq.check()
    _check(w, q, sb, st)
    z = np.zeros((16, 64), np.uint16)
    qz, sbz, stz = rlq.quant_nvfp4(to_dev(z))
    rlq.check()
    _check(z, qz, sbz, stz)


def test_nvfp4_pitched():
    N, K = 40, 96
    w = normal_bits(72, (N, K), std=0.5)
    dev = "cuda"
    wb = torch.zeros((N, K + 8), dtype=torch.bfloat16, device=dev)
    wb[:, :K] = to_dev(w)
    qb = torch.full((N, K // 2 + 16), 0xA5, dtype=torch.uint8, device=dev)
    sbb = torch.full((N, K // 16 + 3), 0x5A, dtype=torch.uint8, device=dev)
    st = torch.empty(1, dtype=torch.float32, device=dev)
    rlq.rlq_quant_nvfp4(wb.data_ptr(), N, K, K + 8, qb.data_ptr(), K // 2 + 16, sbb.data_ptr(), K // 16 + 3,
                        st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    rlq.check()
    _check(w, qb[:, :K // 2], sbb[:, :K // 16], st)
    assert torch.all(qb[:, K // 2:] == 0xA5) and torch.all(sbb[:, K // 16:] == 0x5A)


def test_nvfp4_midpoint_quotients_under_non_power_of_two_block_scales():
    """Blocks whose scale decodes to 1.125, 1.25, 1.5 or 1.75 (amax 6.75, 7.5, 9,
    10.5 with a tensor scale of 1) holding x = m * S for every E2M1 midpoint m:
    x / S is exactly a midpoint (a tie, to the even code), while x * RN(1 / S) lands
    an ulp away from it; the codes must still equal the oracle's, which divides."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    blocks = []
    for S in (1.125, 1.25, 1.5, 1.75):
        v = np.zeros(16, np.float32)
        v[0] = 6.0 * S                    # block amax: its scale code decodes to S exactly
        v[1:8] = mids * S
        v[8:15] = -mids * S
        v[15] = 0.375 * S                 # below the first midpoint
        blocks.append(v)
    row = np.concatenate(blocks + [np.zeros(16 * 4, np.float32)])
    row[-1] = 2688.0                      # tensor amax 6 * 448: tensor scale exactly 1
    w = I.to_bf16_bits(np.tile(row, (4, 1)))
    assert np.array_equal(oracle.bf16_to_f32(w)[0], row)  # every value exact in bf16
    q, sb, st = rlq.quant_nvfp4(to_dev(w))
    rlq.check()
    _check(w, q, sb, st)


def test_nvfp4_block_scales_on_e4m3_grid_points_and_midpoints():
    """Tensor scale 1 (tensor amax 2688) and block maxima 6 * c for c on the E4M3
    grid and halfway between grid neighbours: amax_b / 6 / st is then exactly a code
    or a rounding tie (to the even code), where the block scale's reciprocal-based
    estimate brackets a rounding point and the kernel must fall back to the IEEE
    divisions.  Block maxima that are not bf16-exact are skipped."""
    codes = np.arange(0x08, 0x7F, dtype=np.uint8)  # normal positive E4M3 values up to 448
    vals = oracle.e4m3_decode(codes).astype(np.float64)
    cands = np.concatenate([vals, (vals[:-1] + vals[1:]) / 2]) * 6.0
    bf = oracle.bf16_to_f32(I.to_bf16_bits(cands.astype(np.float32))).astype(np.float64)
    cands = cands[bf == cands]  # block maxima exact in bf16
    assert cands.size > 100
    rng = np.random.default_rng(88)
    blocks = []
    for a in cands:
        v = (rng.uniform(-1.0, 1.0, 16) * a).astype(np.float32)
        v[int(rng.integers(0, 16))] = a * (1 if rng.random() < 0.5 else -1)
        blocks.append(v)
    row = np.concatenate(blocks)
    pad = (-row.size) % 128
    row = np.concatenate([row, np.zeros(pad, np.float32)])
    row[-1] = 2688.0  # tensor amax 6 * 448: tensor scale exactly 1
    w = I.to_bf16_bits(np.tile(row, (3, 1)))
    q, sb, st = rlq.quant_nvfp4(to_dev(w))
    rlq.check()
    _check(w, q, sb, st)
