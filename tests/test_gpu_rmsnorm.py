"""GPU parity of the fused RMSNorm + 1x128 (+ 128x1) quantizer, through the C
ABI, against the oracle: rstd, codes and scales bit for bit equal to
oracle.rmsnorm followed by the oracle's 1x128 / 128x1 quantizers.

QuRL notes, 关键设计 §1: the UAQ scale folded into the norm weight; Jet-RL
notes, 细粒度 GEMM 量化方案: the activation's 1x128 and 128x1 FP8 codes.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_quantize_gb300 import inputs as I
from fp8_block_scaled_quantize_gb300 import rlq
from gpu_util import assert_gemm_close, assert_equal_to_oracle, np_, quant_weight_checked, to_dev, u16

pytestmark = pytest.mark.gpu


def _gamma(K, seed):
    return I.to_bf16_bits(np.random.default_rng(seed).uniform(0.5, 2.0, K).astype(np.float32))


def _check(h, g, eps, colwise, what=""):
    q, s, qT, sc, rstd = rlq.rmsnorm_quant_act_1x128(to_dev(h), to_dev(g), eps, colwise=colwise)
    rlq.check()
    x, orstd = oracle.rmsnorm(h, g, eps)
    assert_equal_to_oracle(rstd, orstd, f"rstd {what}")
    oq, os_ = oracle.quant_rows_1x128(x)
    assert_equal_to_oracle(q, oq, f"1x128 codes {what}")
    assert_equal_to_oracle(s, os_, f"1x128 scales {what}")
    if colwise:
        oqT, osc = oracle.quant_cols_128x1(x)
        assert_equal_to_oracle(qT, oqT, f"128x1 codes {what}")
        assert_equal_to_oracle(sc, osc, f"128x1 scales {what}")
    return x, (q, s, qT, sc, rstd)


@pytest.mark.parametrize("M", [1, 7, 31, 33, 129, 200, 1000])
@pytest.mark.parametrize("K", [128, 384, 4096])
@pytest.mark.parametrize("colwise", [False, True])
def test_ragged_shapes(M, K, colwise):
    h = I.to_bf16_bits(I.normal(80, "x", (M, K), 1.0, M, K))
    _check(h, _gamma(K, K), 1e-6, colwise, f"M={M} K={K}")


@pytest.mark.parametrize("K", [256, 640, 768, 896, 1664])
def test_row_factor_ring_boundaries(K):
    """Row lengths of 2, 5, 6, 7 and 13 chunks of 128 columns around the row-factor
    kernel's six-slot ring (fewer chunks than slots, exactly the lookahead, one
    full ring, one past it, two wraps), on 70 rows (a partial last CTA)."""
    h = I.to_bf16_bits(I.normal(87, "x", (70, K), 1.0, 70, K))
    _check(h, _gamma(K, K + 1), 1e-6, True, f"K={K}")
    _check(h, _gamma(K, K + 1), 1e-6, False, f"K={K}")


def test_rows_of_different_magnitude_and_crafted_rows():
    """Rows spanning 2^-40 .. 2^20 (each row's factor must go to its own row),
    constant +-2^j rows (closed form, eps = 0 exact), the index-order row
    [4096, 1, 1, ...] whose ones are all lost to ties, and signed zeros."""
    K = 512
    rng = np.random.default_rng(81)
    rows = [rng.standard_normal(K) * 2.0 ** e for e in (-40, -12, 0, 7, 20)]
    rows += [np.full(K, 0.25), np.full(K, -8.0)]
    r = np.ones(K)
    r[0] = 4096.0
    rows.append(r)
    z = np.full(K, 1.5)
    z[::3] = -0.0
    rows.append(z)
    h = I.to_bf16_bits(np.stack(rows).astype(np.float32))
    g = _gamma(K, 82)
    _check(h, g, 0.0, True, "crafted, eps=0")
    _check(h, g, 1e-5, True, "crafted, eps=1e-5")


def test_tiny_rows_with_subnormal_partial_sums():
    """Rows of magnitude 2^-64 .. 2^-75, whose squares and early partial sums are
    fp32 subnormals (the sum of squares must not flush them), and rows of bf16
    subnormals, whose squares all round to zero (then eps alone sets rstd)."""
    K = 384
    rng = np.random.default_rng(86)
    rows = [rng.standard_normal(K) * 2.0 ** e for e in (-64, -66, -70, -75)]
    rows.append(rng.standard_normal(K) * 2.0 ** -130)
    mixed = rng.standard_normal(K) * 2.0 ** -70
    mixed[200:] *= 2.0 ** 40
    rows.append(mixed)
    h = I.to_bf16_bits(np.stack(rows).astype(np.float32))
    g = _gamma(K, 86)
    _check(h[:3], g, 0.0, True, "tiny rows, eps=0")
    _check(h, g, 1e-30, True, "tiny and subnormal rows, eps=1e-30")


def test_pitched_hidden_state():
    M, K, pad = 130, 384, 40
    h = I.to_bf16_bits(I.normal(83, "x", (M, K), 1.0))
    buf = torch.full((M, K + pad), 9.0, dtype=torch.bfloat16, device="cuda")
    buf[:, :K] = to_dev(h)
    g = _gamma(K, 83)
    gd = to_dev(g)
    q = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    s = torch.empty((K // 128, M), dtype=torch.float32, device="cuda")
    rstd = torch.empty(M, dtype=torch.float32, device="cuda")
    rlq.rlq_rmsnorm_quant_act_1x128(buf.data_ptr(), M, K, K + pad, gd.data_ptr(), 1e-6, rstd.data_ptr(),
                                    q.data_ptr(), K, s.data_ptr(), M, None, 0, None, 0,
                                    torch.cuda.current_stream().cuda_stream)
    rlq.check()
    x, orstd = oracle.rmsnorm(h, g, 1e-6)
    oq, os_ = oracle.quant_rows_1x128(x)
    assert np.array_equal(np_(rstd), orstd) and np.array_equal(np_(q), oq) and np.array_equal(np_(s), os_)


@pytest.mark.parametrize("which,M", [("llama8b", 8192), ("qwen7b", 4096), ("32b", 16384)])
def test_full_size_hidden_states(which, M):
    """The hidden sizes the norm precedes (4096, 3584, 5120) at full token counts."""
    K = {"llama8b": 4096, "qwen7b": 3584, "32b": 5120}[which]
    h = I.to_bf16_bits(I.normal(84, "x", (M, K), 1.0, M, K))
    _check(h, _gamma(K, 84), 1e-5, True, which)


def test_folded_gamma_then_fprop_matches_the_unfused_chain():
    """QuRL notes, 关键设计 §1: gamma' = gamma * s and W' = W / s (per-channel
    s ~ U[1.5, 4], folded on the GPU); the fused norm + quant of the hidden state
    with gamma', then FProp with W', against the oracle's fold -> rmsnorm ->
    quant -> fp64 GEMM chain."""
    d = I.qwen7b_layer(512, "gate_up")
    N, K = d["w"].shape
    M = 512
    h = I.to_bf16_bits(I.normal(85, "x", (M, K), 1.0))
    g = _gamma(K, 85)
    gg, wg = to_dev(g)[None, :].contiguous(), to_dev(d["w"])
    sg = torch.from_numpy(d["s"]).cuda()
    rlq.uaq_fold_(wg, sg, gg)
    w_f, g_f = oracle.uaq_fold(d["w"], d["s"], g[None, :])
    rlq.check()
    assert np.array_equal(u16(gg), g_f) and np.array_equal(u16(wg), w_f)
    x, (qx, sx, _, _, _) = _check(h, g_f[0], 1e-6, False, "folded gamma")
    (qw, sw, _), (oqw, osw, _) = quant_weight_checked(w_f, transposed=False)
    oqx, osx = oracle.quant_rows_1x128(x)
    y = rlq.gemm_fprop(qx, sx, qw, sw)
    rlq.check()
    assert_gemm_close(y, oracle.gemm_fprop(oqx, osx, oqw, osw), "FProp after the fused norm")


def test_validation():
    K = 256
    h = torch.zeros((4, K), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(K + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rlq.RlqError) as e:
        rlq.rlq_rmsnorm_quant_act_1x128(h.data_ptr(), 4, K, K, g[1:].data_ptr(), 1e-6, 0x10000, 0x10000, K,
                                        0x10000, 4, None, 0, None, 0, 0)
    assert e.value.status == 3  # gamma misaligned
    with pytest.raises(rlq.RlqError) as e:
        rlq.rmsnorm_quant_act_1x128(h, g[:K], float("nan"))
    assert e.value.status == 1
    rlq.check()
