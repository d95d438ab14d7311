"""GPU parity on every workload the benchmark times, at full size, through the
C ABI, against the fp64 oracle.

For each workload the inputs are quantized on the GPU and by the oracle; the
GPU's codes and scales (row-wise, the transposed column-wise ones and the
weight blocks) must equal the oracle's bit for bit, and the GEMMs are then
compared with the oracle's fp64 GEMMs over the oracle's own codes, on outputs
sampled in every 128-row (and, where the contraction is long, 128-column)
stratum, at the tolerance of the other GEMM tests: relative Frobenius error
<= 2e-3 and per element |err| <= 1e-2 * (|ref| + 1) after bf16 rounding.

Workloads (granularities: Jet-RL notes, section "细粒度 GEMM 量化方案", Fig. 6;
the fold: QuRL notes, 关键设计 §1):

* Llama-3.1-8B decode up-projection: X [256, 4096] with 1% outlier channels,
  W [14336, 4096]; FProp on every output, single pass and split-K.
* Qwen2.5-7B layer set: gate/up [18944, 3584] and down [3584, 18944] at
  M in {64, 512, 4096}: the UAQ fold with per-channel s ~ U[1.5, 4] (folded
  tensors bit-exact), then quantization, then FProp (single pass and split-K).
* 32B-shaped sweep, both orientations: M in {4096, 16384} for FProp, DGrad
  (transposed and untransposed weight codes) and WGrad; the down orientation
  at every smaller M as well (single pass and split-K wherever the library's
  plan splits).
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_quantize_gb300 import inputs as I
from fp8_block_scaled_quantize_gb300 import rlq
from gpu_util import (assert_gemm_close, idx as _idx, quant_act_checked as _quant_act,
                      quant_weight_checked as _quant_weight, strata as _strata, to_dev, u16)

pytestmark = pytest.mark.gpu


def _splits(kind, M, N, K):
    return rlq.rlq_gemm_splitk_workspace_bytes(kind, M, N, K) > 0


# -------------------------------------------------- 8B decode up-proj ---

def test_decode_upproj_8b_full_size_fprop():
    d = I.decode_upproj_8b()
    M, K = d["x"].shape
    N = d["w"].shape[0]
    (qx, sx, _, _), (oqx, osx) = _quant_act(d["x"], colwise=False)
    (qw, sw, _), (oqw, osw, _) = _quant_weight(d["w"], transposed=False)
    ref = oracle.gemm_fprop(oqx, osx, oqw, osw)  # every one of the 256 x 14336 outputs
    assert_gemm_close(rlq.gemm_fprop(qx, sx, qw, sw), ref, "FProp 8B decode")
    if _splits(rlq.GEMM_FPROP, M, N, K):
        assert_gemm_close(rlq.gemm_fprop(qx, sx, qw, sw, split_k=True), ref, "FProp 8B decode, split-K")
    rlq.check()


# ------------------------------------------------ Qwen2.5-7B layer set ---

@pytest.mark.parametrize("which", ["gate_up", "down"])
@pytest.mark.parametrize("M", list(I.QWEN7B_M))
def test_qwen7b_fold_quant_fprop(which, M):
    """The fold with per-channel s, then quantization, then FProp."""
    d = I.qwen7b_layer(M, which)
    N, K = d["w"].shape
    xg, wg = to_dev(d["x"]), to_dev(d["w"])
    rlq.uaq_fold_(wg, torch.from_numpy(d["s"]).cuda(), xg)
    w_f, x_f = oracle.uaq_fold(d["w"], d["s"], d["x"])
    rlq.check()
    assert np.array_equal(u16(wg), w_f), "folded W"
    assert np.array_equal(u16(xg), x_f), "folded X"
    del xg, wg
    (qx, sx, _, _), (oqx, osx) = _quant_act(x_f, colwise=False)
    (qw, sw, _), (oqw, osw, _) = _quant_weight(w_f, transposed=False)
    rng = np.random.default_rng(M + N)
    rows = np.arange(M) if M <= 512 else _strata(M, 32, rng)
    ref = oracle.gemm_fprop(oqx, osx, oqw, osw, rows=rows)
    y = rlq.gemm_fprop(qx, sx, qw, sw)
    assert_gemm_close(y[_idx(rows)], ref, f"FProp qwen7b {which} M={M}")
    if _splits(rlq.GEMM_FPROP, M, N, K):
        y = rlq.gemm_fprop(qx, sx, qw, sw, split_k=True)
        assert_gemm_close(y[_idx(rows)], ref, f"FProp qwen7b {which} M={M}, split-K")
    rlq.check()


# --------------------------------------------------------- 32B sweep ---

_W32 = {}


def _weight_32b(orient):
    """The 32B weight of one orientation, quantized on the GPU (with the
    transposed copy) and by the oracle; built once per orientation."""
    if orient not in _W32:
        _W32.clear()  # keep one orientation resident at a time
        w = I.sweep_32b(1, orient, with_dy=False)["w"]
        _W32[orient] = _quant_weight(w, transposed=True)
    return _W32[orient]


def _check_32b(orient, M, single=True, split=True):
    (qw, sw, qwT), (oqw, osw, _) = _weight_32b(orient)
    d = I.sweep_32b(M, orient, with_w=False)
    N, K = oqw.shape
    (qx, sx, qxT, sxc), (oqx, osx, oqxT, osxc) = _quant_act(d["x"], colwise=True)
    (qdy, sdy, qdyT, sdyc), (oqdy, osdy, oqdyT, osdyc) = _quant_act(d["dy"], colwise=True)
    del d
    rng = np.random.default_rng(17 * M + N)
    rows_m = _strata(M, 128, rng) if M > 256 else np.arange(M)
    rows_n = _strata(N, 128, rng)
    cols_k = _strata(K, 32, rng) if K > 8192 else np.arange(K)
    tag = f"32B {orient} M={M}"
    ref_y = oracle.gemm_fprop(oqx, osx, oqw, osw, rows=rows_m)
    ref_dx = oracle.gemm_dgrad(oqdy, osdy, oqw, osw, rows=rows_m)
    ref_dw = oracle.gemm_wgrad(oqdyT, osdyc, oqxT, osxc, rows=rows_n, cols=cols_k)
    modes = ([False] if single else []) + ([True] if split else [])
    for sk in modes:
        # the split-K entry points are checked where the library's plan splits
        if not sk or _splits(rlq.GEMM_FPROP, M, N, K):
            y = rlq.gemm_fprop(qx, sx, qw, sw, split_k=sk)
            assert_gemm_close(y[_idx(rows_m)], ref_y, f"FProp {tag} split_k={sk}")
            del y
        if not sk or _splits(rlq.GEMM_DGRAD, M, N, K):
            dx = rlq.gemm_dgrad(qdy, sdy, qwT, sw, transposed=True, split_k=sk)
            assert_gemm_close(dx[_idx(rows_m)], ref_dx, f"DGrad {tag} split_k={sk}")
            dx = rlq.gemm_dgrad(qdy, sdy, qw, sw, transposed=False, split_k=sk, out=dx)
            assert_gemm_close(dx[_idx(rows_m)], ref_dx, f"DGrad (untransposed codes) {tag} split_k={sk}")
            del dx
        if not sk or _splits(rlq.GEMM_WGRAD, M, N, K):
            dw = rlq.gemm_wgrad(qdyT, sdyc, qxT, sxc, split_k=sk)
            assert_gemm_close(dw[_idx(rows_n)][:, _idx(cols_k)], ref_dw, f"WGrad {tag} split_k={sk}")
            del dw
    rlq.check()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("orient", ["up", "down"])
@pytest.mark.parametrize("M", [4096, 16384])
def test_sweep_32b_large_M_all_gemms(orient, M):
    """K = 5120 / N = 27648 and the transposed shape, at the two token counts
    where the GEMMs are bound by the tensor cores: the longest contractions of
    the suite (216 promoted blocks in DGrad of the up orientation and FProp of
    the down one; 128 token blocks in WGrad at M = 16384)."""
    _check_32b(orient, M)


@pytest.mark.parametrize("M", [1, 16, 64, 256, 1024])
def test_sweep_32b_down_small_and_mid_M(M):
    """The down orientation (N = 5120, K = 27648) at the decode-to-prefill token
    counts: FProp and DGrad single pass and split-K, WGrad at every M."""
    _check_32b("down", M)
