"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch

from fp8_block_scaled_quantize_gb300 import inputs as I

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
