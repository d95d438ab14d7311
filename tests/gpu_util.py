"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch

import oracle
from fp8_block_scaled_quantize_gb300 import inputs as I
from fp8_block_scaled_quantize_gb300 import rlq

DEV = "cuda"

# GEMM tolerance: relative Frobenius error and per-element bound,
# measured on the bf16 output against the fp64 oracle.
REL_FRO = 2e-3
ELEM_ABS = 1e-2


def to_dev(bits: np.ndarray) -> torch.Tensor:
    return I.to_torch(bits, DEV)


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def np_(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def assert_gemm_close(got: torch.Tensor, ref: np.ndarray, what: str = ""):
    g = got.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    err = g - ref
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(err) / nref if nref > 0 else np.linalg.norm(err)
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3e} > {REL_FRO}"
    bad = np.abs(err) > ELEM_ABS * (np.abs(ref) + 1)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond 1e-2*(|ref|+1)"
    return rel


def normal_bits(seed, shape, std=1.0, tag="x"):
    return I.to_bf16_bits(I.normal(seed, tag, shape, std, *shape))


def strata(n, blk, rng):
    """One random index in every block of `blk` indices of range(n), plus 0 and n - 1."""
    starts = np.arange(0, n, blk)
    picks = np.minimum(starts + rng.integers(0, blk, size=starts.size), n - 1)
    return np.unique(np.concatenate([picks, [0, n - 1]]))


def idx(a) -> torch.Tensor:
    return torch.from_numpy(np.asarray(a)).cuda()


def assert_equal_to_oracle(got: torch.Tensor, ref: np.ndarray, what: str):
    g = np_(got)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.array_equal(g, ref), f"{what}: GPU quantizer output differs from the oracle"


def quant_act_checked(bits: np.ndarray, colwise: bool):
    """1x128 (+ 128x1) quantization on the GPU, asserted bit for bit equal to
    the oracle's; returns (GPU tensors, oracle arrays) in quant_act_1x128's order."""
    g = rlq.quant_act_1x128(to_dev(bits), colwise=colwise)
    o = oracle.quant_rows_1x128(bits)
    assert_equal_to_oracle(g[0], o[0], "1x128 codes")
    assert_equal_to_oracle(g[1], o[1], "1x128 scales")
    if colwise:
        o = o + oracle.quant_cols_128x1(bits)
        assert_equal_to_oracle(g[2], o[2], "128x1 codes (transposed)")
        assert_equal_to_oracle(g[3], o[3], "128x1 scales")
    return g, o


def quant_weight_checked(bits: np.ndarray, transposed: bool):
    """128x128 quantization on the GPU, asserted equal to the oracle's."""
    g = rlq.quant_weight_128x128(to_dev(bits), transposed=transposed)
    o = oracle.quant_weight_128x128(bits, transposed=transposed)
    assert_equal_to_oracle(g[0], o[0], "128x128 codes")
    assert_equal_to_oracle(g[1], o[1], "128x128 scales")
    if transposed:
        assert_equal_to_oracle(g[2], o[2], "128x128 codes (transposed copy)")
    return g, o
