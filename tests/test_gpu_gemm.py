"""GPU parity of the block-scaled FP8 GEMMs (FProp, DGrad, WGrad through the
C ABI) against the oracle's fp64 GEMMs over the same codes and scales.

* Tolerance: relative Frobenius error <= 2e-3 and per element
  |err| <= 1e-2 * (|ref| + 1), on the bf16 output.
* Integer pins: integer-valued codes with scales 1 (or one power of two) give
  exact fp32 accumulations; the bf16 outputs must then match the oracle's
  result rounded to bf16 bit for bit — this catches any layout, transpose,
  scale-index or tail mistake that a tolerance could hide.
* Full-size workloads are checked on sampled output rows / columns.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_quantize_gb300 import inputs as I
from fp8_block_scaled_quantize_gb300 import rlq
from gpu_util import (assert_gemm_close, idx, normal_bits, np_, quant_act_checked, quant_weight_checked,
                      strata, to_dev, u16)

pytestmark = pytest.mark.gpu

SHAPES = [(1, 128, 128), (5, 256, 256), (128, 256, 128), (200, 384, 512), (257, 512, 384),
          (1000, 1280, 1024), (129, 640, 896)]


def _quantized_operands(M, N, K, seed):
    x = normal_bits(seed, (M, K), 1.0, "x")
    w = normal_bits(seed, (N, K), 0.02, "w")
    dy = normal_bits(seed, (M, N), 1e-3, "dy")
    xg, wg, dyg = to_dev(x), to_dev(w), to_dev(dy)
    g = {}
    g["qx"], g["sx"], g["qxT"], g["sxc"] = rlq.quant_act_1x128(xg, colwise=True)
    g["qdy"], g["sdy"], g["qdyT"], g["sdyc"] = rlq.quant_act_1x128(dyg, colwise=True)
    g["qw"], g["sw"], g["qwT"] = rlq.quant_weight_128x128(wg, transposed=True)
    o = {}
    o["qx"], o["sx"] = oracle.quant_rows_1x128(x)
    o["qxT"], o["sxc"] = oracle.quant_cols_128x1(x)
    o["qdy"], o["sdy"] = oracle.quant_rows_1x128(dy)
    o["qdyT"], o["sdyc"] = oracle.quant_cols_128x1(dy)
    o["qw"], o["sw"], _ = oracle.quant_weight_128x128(w)
    for k in ("qx", "sx", "qdy", "sdy", "qw", "sw"):
        assert np.array_equal(np_(g[k]), o[k]), k
    return g, o


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_fprop_parity(M, N, K):
    g, o = _quantized_operands(M, N, K, 20)
    y = rlq.gemm_fprop(g["qx"], g["sx"], g["qw"], g["sw"])
    rlq.check()
    assert_gemm_close(y, oracle.gemm_fprop(o["qx"], o["sx"], o["qw"], o["sw"]), "FProp")


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("transposed", [True, False])
def test_dgrad_parity(M, N, K, transposed):
    """DGrad from the transposed weight codes, or from the FProp codes read
    MN-major; both must match the oracle (and each other)."""
    g, o = _quantized_operands(M, N, K, 21)
    w = g["qwT"] if transposed else g["qw"]
    dx = rlq.gemm_dgrad(g["qdy"], g["sdy"], w, g["sw"], transposed=transposed)
    rlq.check()
    assert_gemm_close(dx, oracle.gemm_dgrad(o["qdy"], o["sdy"], o["qw"], o["sw"]), "DGrad")


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_wgrad_parity(M, N, K):
    g, o = _quantized_operands(M, N, K, 22)
    dw = rlq.gemm_wgrad(g["qdyT"], g["sdyc"], g["qxT"], g["sxc"])
    rlq.check()
    assert_gemm_close(dw, oracle.gemm_wgrad(o["qdyT"], o["sdyc"], o["qxT"], o["sxc"]), "WGrad")


# ------------------------------------------------------------ exact pins ---

def _int_codes(rng, shape, lim=16):
    return oracle.e4m3_encode(rng.integers(-lim, lim + 1, size=shape).astype(np.float32))


def _bf16_of(ref: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(ref.astype(np.float32))  # exact: |integers| < 2^24
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("M,N,K", [(3, 128, 128), (130, 256, 384), (300, 640, 256), (1024, 512, 1024)])
@pytest.mark.parametrize("scale", [1.0, 2.0 ** -7])
def test_integer_gemms_bit_exact(M, N, K, scale):
    rng = np.random.default_rng(M + N + K)
    qx, qw, qdy = _int_codes(rng, (M, K)), _int_codes(rng, (N, K)), _int_codes(rng, (M, N))
    sx = np.full((K // 128, M), scale, np.float32)
    sw = np.full((N // 128, K // 128), 1.0, np.float32)
    sdy = np.full((N // 128, M), scale, np.float32)
    y = rlq.gemm_fprop(_dev(qx), _dev(sx), _dev(qw), _dev(sw))
    dx = rlq.gemm_dgrad(_dev(qdy), _dev(sdy), _dev(np.ascontiguousarray(qw.T)), _dev(sw), transposed=True)
    dx_mn = rlq.gemm_dgrad(_dev(qdy), _dev(sdy), _dev(qw), _dev(sw), transposed=False)
    # WGrad operands: 128x1 codes of dY and X, transposed, with a partial last token block
    MB = (M + 127) // 128
    ldm = (M + 15) // 16 * 16
    qdyT = np.zeros((N, ldm), np.uint8)
    qdyT[:, :M] = qdy.T
    qxT = np.zeros((K, ldm), np.uint8)
    qxT[:, :M] = qx.T
    sdyc = np.full((MB, N), scale, np.float32)
    sxc = np.full((MB, K), 1.0, np.float32)
    dw = rlq.gemm_wgrad(_dev(qdyT)[:, :M], _dev(sdyc), _dev(qxT)[:, :M], _dev(sxc))
    rlq.check()
    ry = oracle.gemm_fprop(qx, sx, qw, sw)
    rdx = oracle.gemm_dgrad(qdy, sdy, qw, sw)
    rdw = oracle.gemm_wgrad(qdyT[:, :M], sdyc, qxT[:, :M], sxc)
    assert np.array_equal(u16(y), _bf16_of(ry)), "FProp integer pin"
    assert np.array_equal(u16(dx), _bf16_of(rdx)), "DGrad integer pin"
    assert np.array_equal(u16(dx_mn), _bf16_of(rdx)), "DGrad (untransposed weight codes) integer pin"
    assert np.array_equal(u16(dw), _bf16_of(rdw)), "WGrad integer pin"


def test_one_hot_rows_select_weight_columns():
    """One-hot X rows (value 448, so the row scale is exactly 1) against W whose
    128x128 blocks each hold one element 448 * 2^-10 (block scale exactly
    2^-10): every output is 448 * decode(code) * 2^-10, at most 7 significant
    bits, so the bf16 result is exact and must match the oracle bit for bit."""
    N, K = 512, 384
    rng = np.random.default_rng(31)
    wf = np.clip(rng.standard_normal((N, K)).astype(np.float32) * 0.02, -0.4, 0.4)
    wf[::128, ::128] = 0.4375  # 448 * 2^-10 in every block
    w = I.to_bf16_bits(wf)
    xf = np.zeros((6, K), np.float32)
    hot = [0, 1, 127, 128, 255, 383]
    for i, k in enumerate(hot):
        xf[i, k] = 448.0
    x = I.to_bf16_bits(xf)
    qx, sx, _, _ = rlq.quant_act_1x128(to_dev(x))
    qw, sw, _ = rlq.quant_weight_128x128(to_dev(w))
    y = rlq.gemm_fprop(qx, sx, qw, sw)
    rlq.check()
    oqx, osx = oracle.quant_rows_1x128(x)
    oqw, osw, _ = oracle.quant_weight_128x128(w)
    assert np.all(osw == 2.0 ** -10)
    ref = oracle.gemm_fprop(oqx, osx, oqw, osw)
    wd = oracle.dequant_weight(oqw, osw)
    for i, k in enumerate(hot):
        assert np.array_equal(ref[i], 448.0 * wd[:, k])
    assert np.array_equal(u16(y), I.to_bf16_bits(ref.astype(np.float32)))


# ------------------------------------------------------- degenerate cases ---

def test_empty_and_degenerate_shapes():
    dev = "cuda"
    # WGrad over zero tokens: dW = 0
    dw = torch.full((256, 128), 3.0, dtype=torch.bfloat16, device=dev)
    e = torch.empty((256, 16), dtype=torch.uint8, device=dev)
    rlq.rlq_gemm_wgrad(e.data_ptr(), 16, 0, 256, e.data_ptr(), 16, 0, 128, dw.data_ptr(), 128, 0, 256, 128,
                       torch.cuda.current_stream().cuda_stream)
    rlq.check()
    assert torch.all(dw == 0)
    # FProp with M = 0 launches nothing and succeeds
    y = torch.empty((0, 256), dtype=torch.bfloat16, device=dev)
    rlq.gemm_fprop(torch.empty((0, 128), dtype=torch.uint8, device=dev), torch.empty((1, 1), device=dev),
                   torch.empty((256, 128), dtype=torch.uint8, device=dev), torch.empty((2, 1), device=dev), out=y)
    rlq.check()


def test_all_zero_operands_give_zero():
    M, N, K = 130, 256, 256
    x = np.zeros((M, K), np.uint16)
    w = normal_bits(40, (N, K), 0.02, "w")
    qx, sx, qxT, sxc = rlq.quant_act_1x128(to_dev(x), colwise=True)
    qw, sw, _ = rlq.quant_weight_128x128(to_dev(w))
    y = rlq.gemm_fprop(qx, sx, qw, sw)
    rlq.check()
    assert torch.all(y == 0)


# ---------------------------------------------------- full-size, sampled ---

def test_full_size_train_step_8b_sampled():
    """The 8B-shaped training step (M=8192, N=14336, K=4096): all three GEMMs
    in the bench's launch configuration, checked on outputs sampled in every
    128-row stratum against the oracle's GEMMs over the oracle's own codes
    (the GPU's codes, column-wise ones included, are asserted equal first)."""
    d = I.train_step_8b()
    (qx, sx, qxT, sxc), (oqx, osx, oqxT, osxc) = quant_act_checked(d["x"], colwise=True)
    (qdy, sdy, qdyT, sdyc), (oqdy, osdy, oqdyT, osdyc) = quant_act_checked(d["dy"], colwise=True)
    (qw, sw, qwT), (oqw, osw, _) = quant_weight_checked(d["w"], transposed=True)
    del d
    y = rlq.gemm_fprop(qx, sx, qw, sw)
    dx = rlq.gemm_dgrad(qdy, sdy, qwT, sw, transposed=True)
    dw = rlq.gemm_wgrad(qdyT, sdyc, qxT, sxc)
    rlq.check()
    rng = np.random.default_rng(5)
    M, N, K = 8192, 14336, 4096
    rows = strata(M, 128, rng)
    rows_n = strata(N, 128, rng)
    assert_gemm_close(y[idx(rows)], oracle.gemm_fprop(oqx, osx, oqw, osw, rows=rows), "FProp 8B")
    assert_gemm_close(dx[idx(rows)], oracle.gemm_dgrad(oqdy, osdy, oqw, osw, rows=rows), "DGrad 8B")
    assert_gemm_close(dw[idx(rows_n)], oracle.gemm_wgrad(oqdyT, osdyc, oqxT, osxc, rows=rows_n), "WGrad 8B")


@pytest.mark.parametrize("M", [1, 16, 64, 256, 1024])
def test_sweep_32b_small_and_mid_M(M):
    d = I.sweep_32b(M, "up")
    (qx, sx, qxT, sxc), (oqx, osx, oqxT, osxc) = quant_act_checked(d["x"], colwise=True)
    (qdy, sdy, qdyT, sdyc), (oqdy, osdy, oqdyT, osdyc) = quant_act_checked(d["dy"], colwise=True)
    (qw, sw, qwT), (oqw, osw, _) = quant_weight_checked(d["w"], transposed=True)
    del d
    y = rlq.gemm_fprop(qx, sx, qw, sw)
    dx = rlq.gemm_dgrad(qdy, sdy, qwT, sw, transposed=True)
    dw = rlq.gemm_wgrad(qdyT, sdyc, qxT, sxc)
    rlq.check()
    rng = np.random.default_rng(M)
    rows = np.arange(M) if M <= 256 else strata(M, 16, rng)
    assert_gemm_close(y[idx(rows)], oracle.gemm_fprop(oqx, osx, oqw, osw, rows=rows), f"FProp 32B M={M}")
    assert_gemm_close(dx[idx(rows)], oracle.gemm_dgrad(oqdy, osdy, oqw, osw, rows=rows), f"DGrad 32B M={M}")
    rows_n = strata(27648, 128, rng)
    assert_gemm_close(dw[idx(rows_n)], oracle.gemm_wgrad(oqdyT, osdyc, oqxT, osxc, rows=rows_n),
                      f"WGrad 32B M={M}")


_MODE_SCRIPT = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
from fp8_block_scaled_quantize_gb300 import rlq
from gpu_util import normal_bits, to_dev
M, N, K = 512, 768, 1024
qx, sx, qxT, sxc = rlq.quant_act_1x128(to_dev(normal_bits(60, (M, K), 1.0, "x")), colwise=True)
qdy, sdy, qdyT, sdyc = rlq.quant_act_1x128(to_dev(normal_bits(60, (M, N), 1e-3, "dy")), colwise=True)
qw, sw, qwT = rlq.quant_weight_128x128(to_dev(normal_bits(60, (N, K), 0.02, "w")), transposed=True)
outs = [rlq.gemm_fprop(qx, sx, qw, sw), rlq.gemm_dgrad(qdy, sdy, qwT, sw), rlq.gemm_dgrad(qdy, sdy, qw, sw, transposed=False),
        rlq.gemm_wgrad(qdyT, sdyc, qxT, sxc)]
acc = torch.full((N, K), 0.25, dtype=torch.float32, device="cuda")
rlq.gemm_wgrad_accumulate_(acc, qdyT, sdyc, qxT, sxc)  # no workspace: the epilogue adds (pairs: TMA reduce-adds)
rlq.check()
np.savez(sys.argv[2], *[o.view(torch.int16).cpu().numpy() for o in outs], acc.view(torch.int32).cpu().numpy())
"""


def test_pair_and_single_cta_modes_agree_bitwise(tmp_path):
    """Tiles of 256 output rows run on CTA pairs (cta_group::2); RLQ_GEMM_PAIR=0
    forces one CTA per 128 rows.  The per-element arithmetic is the same, so the
    two modes must give identical bits for FProp, both DGrad forms, WGrad, and
    WGrad added into an fp32 gradient (pairs add by TMA reduce at L2, single CTAs
    by a read-modify-write: both one fp32 addition per element)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = {}
    for mode in ("0", "1"):
        out = str(tmp_path / f"mode{mode}.npz")
        env = dict(os.environ, RLQ_GEMM_PAIR=mode)
        r = subprocess.run([sys.executable, "-c", _MODE_SCRIPT, root, out], env=env, capture_output=True, text=True,
                           timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        res[mode] = np.load(out)
    for key in res["0"].files:
        assert np.array_equal(res["0"][key], res["1"][key]), key
