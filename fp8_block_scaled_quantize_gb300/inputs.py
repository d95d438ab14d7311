"""Seeded synthetic inputs for the quantized actor linear layer.

This module only draws random tensors (NumPy ``default_rng``, fp32, rounded
to bf16 by torch) in the shapes and distributions of the workloads below.  It
holds none of the method's arithmetic and serves both the CUDA path's tests /
bench and the oracle's tests.  Arrays are returned as uint16 bf16 bit patterns
(use ``to_torch`` for a ``torch.bfloat16`` view).

Workloads (shapes of the models the pages run: Llama-3.1-8B, Qwen2.5-7B and a
32B model; Jet-RL notes Tables 2-4, QuRL notes main table).  No weights or
datasets are used: every tensor is drawn here.

* ``tiny_single_linear``   X [128,256] N(0,1), W [256,256] N(0,0.02), s = 4 on all K
* ``decode_upproj_8b``     X [256,4096] N(0,1) with 1% of K channels x20, W [14336,4096] N(0,0.02)
* ``train_step_8b``        X [8192,4096] N(0,1), W [14336,4096] N(0,0.02), dY [8192,14336] N(0,1e-3)
* ``qwen7b_layer``         gate/up W [18944,3584] or down W [3584,18944] N(0,0.02); X [M,K] N(0,1)
                           with 1% of K channels drawn from Student-t(3); s ~ U[1.5,4] per K
* ``sweep_32b``            (N,K) = (27648,5120) or (5120,27648), W N(0,0.015); X [M,K] N(0,1) with
                           0.5% of K channels x50; dY [M,N] N(0,1e-3)

Each tensor draws from its own stream ``default_rng([seed, tag])`` so that a
tensor does not depend on the sizes of the others.
"""
from __future__ import annotations

import numpy as np
import torch

SEEDS = {"tiny_single_linear": 0, "decode_upproj_8b": 1, "train_step_8b": 2,
         "qwen7b_layer": 3, "sweep_32b": 4}

_TAG = {"x": 1, "w": 2, "dy": 3, "outlier_idx": 4, "outlier_val": 5, "s": 6}


def _rng(seed: int, tag: str, *extra: int) -> np.random.Generator:
    return np.random.default_rng([seed, _TAG[tag], *extra])


def to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), rounded by torch."""
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def to_torch(bits: np.ndarray, device=None) -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor (on ``device``)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device is not None else t


def normal(seed: int, tag: str, shape, std: float, *extra: int) -> np.ndarray:
    v = _rng(seed, tag, *extra).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    return v


def with_outlier_channels(seed: int, x: np.ndarray, frac: float, factor: float, *extra: int) -> np.ndarray:
    """Scale a seeded random choice of ceil(frac*K) columns of x by ``factor``."""
    K = x.shape[1]
    n = int(np.ceil(frac * K))
    idx = _rng(seed, "outlier_idx", *extra).choice(K, n, replace=False)
    x[:, idx] *= np.float32(factor)
    return x


def with_student_t_channels(seed: int, x: np.ndarray, frac: float, dof: float, *extra: int) -> np.ndarray:
    """Replace a seeded random choice of ceil(frac*K) columns of x by i.i.d. Student-t draws."""
    M, K = x.shape
    n = int(np.ceil(frac * K))
    idx = _rng(seed, "outlier_idx", *extra).choice(K, n, replace=False)
    x[:, idx] = _rng(seed, "outlier_val", *extra).standard_t(dof, (M, n)).astype(np.float32)
    return x


# ----------------------------------------------------------- workloads ---

def tiny_single_linear():
    seed = SEEDS["tiny_single_linear"]
    x = to_bf16_bits(normal(seed, "x", (128, 256), 1.0))
    w = to_bf16_bits(normal(seed, "w", (256, 256), 0.02))
    s = np.full(256, 4.0, np.float32)
    return {"x": x, "w": w, "s": s}


def decode_upproj_8b():
    seed = SEEDS["decode_upproj_8b"]
    x = with_outlier_channels(seed, normal(seed, "x", (256, 4096), 1.0), 0.01, 20.0)
    return {"x": to_bf16_bits(x), "w": to_bf16_bits(normal(seed, "w", (14336, 4096), 0.02))}


def train_step_8b(M: int = 8192, N: int = 14336, K: int = 4096, with_dy: bool = True):
    """The 8B-shaped training step; smaller M / N / K give the same recipe at
    other sizes (used by tests)."""
    seed = SEEDS["train_step_8b"]
    out = {"x": to_bf16_bits(normal(seed, "x", (M, K), 1.0, M, K)),
           "w": to_bf16_bits(normal(seed, "w", (N, K), 0.02, N, K))}
    if with_dy:
        out["dy"] = to_bf16_bits(normal(seed, "dy", (M, N), 1e-3, M, N))
    return out


def qwen7b_layer(M: int, which: str = "gate_up"):
    seed = SEEDS["qwen7b_layer"]
    N, K = {"gate_up": (18944, 3584), "down": (3584, 18944)}[which]
    wid = 0 if which == "gate_up" else 1
    x = with_student_t_channels(seed, normal(seed, "x", (M, K), 1.0, M, wid), 0.01, 3.0, wid)
    s = _rng(seed, "s", wid).uniform(1.5, 4.0, K).astype(np.float32)
    return {"x": to_bf16_bits(x), "w": to_bf16_bits(normal(seed, "w", (N, K), 0.02, wid)), "s": s}


def sweep_32b(M: int, orient: str = "up", with_dy: bool = True, with_w: bool = True):
    seed = SEEDS["sweep_32b"]
    N, K = {"up": (27648, 5120), "down": (5120, 27648)}[orient]
    oid = 0 if orient == "up" else 1
    x = with_outlier_channels(seed, normal(seed, "x", (M, K), 1.0, M, oid), 0.005, 50.0, oid)
    out = {"x": to_bf16_bits(x)}
    if with_w:
        out["w"] = to_bf16_bits(normal(seed, "w", (N, K), 0.015, oid))
    if with_dy:
        out["dy"] = to_bf16_bits(normal(seed, "dy", (M, N), 1e-3, M, oid))
    return out


SWEEP_32B_M = (1, 16, 64, 256, 1024, 4096, 16384)
QWEN7B_M = (64, 512, 4096)
