"""GPU parity of the UAQ fold, the fold-commutes-with-quantization invariant,
and the bounded-wait failure path (no fault, trap or hang: a wait that nothing
satisfies runs out, the error is reported and the context stays usable)."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_quantize_gb300 import inputs as I
from fp8_block_scaled_quantize_gb300 import rlq
from gpu_util import normal_bits, np_, to_dev, u16

pytestmark = pytest.mark.gpu


def test_fold_tiny_single_linear_bit_exact():
    d = I.tiny_single_linear()
    wg, xg = to_dev(d["w"]), to_dev(d["x"])
    sg = torch.from_numpy(d["s"]).cuda()
    rlq.uaq_fold_(wg, sg, xg)
    rlq.check()
    w_f, x_f = oracle.uaq_fold(d["w"], d["s"], d["x"])
    assert np.array_equal(u16(wg), w_f) and np.array_equal(u16(xg), x_f)


@pytest.mark.parametrize("which", ["gate_up", "down"])
def test_fold_qwen7b_per_channel_bit_exact(which):
    d = I.qwen7b_layer(512, which)
    wg, xg = to_dev(d["w"]), to_dev(d["x"])
    sg = torch.from_numpy(d["s"]).cuda()
    rlq.uaq_fold_(wg, sg, xg)
    gamma = I.to_bf16_bits(np.ones((1, d["w"].shape[1]), np.float32))
    gg = to_dev(gamma)
    rlq.uaq_fold_(torch.empty((0, d["w"].shape[1]), dtype=torch.bfloat16, device="cuda"), sg, gg)  # R = 1 norm weight
    rlq.check()
    w_f, x_f = oracle.uaq_fold(d["w"], d["s"], d["x"])
    _, g_f = oracle.uaq_fold(np.zeros((0, d["w"].shape[1]), np.uint16), d["s"], gamma)
    assert np.array_equal(u16(wg), w_f) and np.array_equal(u16(xg), x_f) and np.array_equal(u16(gg), g_f)


def _fold_gpu(w_bits, s):
    wg = to_dev(w_bits)
    rlq.uaq_fold_(wg, torch.from_numpy(s).cuda())
    rlq.check()
    return u16(wg)


def test_fold_bit_exact_over_wide_ranges():
    """W / s must equal the oracle's bf16_RN(fl32(w / s)) for every element.

    Part 1: 4M random finite bf16 patterns (every exponent, both signs,
    subnormals) against per-column scales log-uniform over 2^-126 .. 2^127 plus
    special ones (1, 3, 7, 0.1, 1/3, 2^-100, 2^101, a subnormal scale, the
    largest floats): quotients that overflow, underflow to subnormals or zero.
    Part 2: N(0, 1) weights against scales in [0.5, 8], every quotient normal."""
    rng = np.random.default_rng(77)
    N, K = 2048, 2048
    w = rng.integers(0, 1 << 16, size=(N, K), dtype=np.uint32).astype(np.uint16)
    nonfinite = ((w >> 7) & 0xFF) == 0xFF
    w[nonfinite] &= np.uint16(0x807F)  # exponent field cleared: a finite subnormal
    s = np.exp2(rng.uniform(-126.0, 127.0, size=K)).astype(np.float32)
    special = [1.0, 3.0, 7.0, 0.1, 1.0 / 3.0, 2.0 ** -100, 2.0 ** -100 * 0.999, 2.0 ** 101, 2.0 ** 101 * 0.999,
               2.0 ** -126, 1e-40, 3.4e38, 2.0 ** 50]
    s[:len(special)] = np.array(special, np.float32)
    want, _ = oracle.uaq_fold(w, s)
    assert np.array_equal(_fold_gpu(w, s), want)
    w2 = normal_bits(78, (N, K), 1.0, "w")
    s2 = rng.uniform(0.5, 8.0, size=K).astype(np.float32)
    want2, _ = oracle.uaq_fold(w2, s2)
    assert np.array_equal(_fold_gpu(w2, s2), want2)


def test_fold_pitched_rows_untouched_padding():
    N, K = 64, 256
    w = I.to_bf16_bits(I.normal(9, "w", (N, K), 0.02))
    buf = torch.full((N, K + 24), 5.0, dtype=torch.bfloat16, device="cuda")
    buf[:, :K] = to_dev(w)
    s = np.random.default_rng(9).uniform(1.5, 4.0, K).astype(np.float32)
    rlq.rlq_uaq_fold(buf.data_ptr(), N, K, K + 24, torch.from_numpy(s).cuda().data_ptr(), None, 0, 0,
                     torch.cuda.current_stream().cuda_stream)
    rlq.check()
    w_f, _ = oracle.uaq_fold(w, s)
    assert np.array_equal(u16(buf[:, :K]), w_f)
    assert torch.all(buf[:, K:] == 5.0)


def test_fold_then_quant_power_of_two_invariance_on_gpu():
    """s = 4 on every channel: the folded tensors quantize to the same codes,
    activation scales x4, weight scales /4, and FProp is bitwise unchanged."""
    d = I.tiny_single_linear()
    xg, wg = to_dev(d["x"]), to_dev(d["w"])
    qx, sx, _, _ = rlq.quant_act_1x128(xg)
    qw, sw, _ = rlq.quant_weight_128x128(wg)
    y0 = rlq.gemm_fprop(qx, sx, qw, sw)
    rlq.uaq_fold_(wg, torch.from_numpy(d["s"]).cuda(), xg)
    qx2, sx2, _, _ = rlq.quant_act_1x128(xg)
    qw2, sw2, _ = rlq.quant_weight_128x128(wg)
    y1 = rlq.gemm_fprop(qx2, sx2, qw2, sw2)
    rlq.check()
    assert torch.equal(qx, qx2) and torch.equal(qw, qw2)
    assert torch.equal(sx2, sx * 4) and torch.equal(sw2, sw / 4)
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


def test_bounded_wait_reports_timeout_and_context_survives():
    rlq.check()  # nothing pending
    rlq.rlq_diag_bounded_wait(2000, torch.cuda.current_stream().cuda_stream)
    with pytest.raises(rlq.RlqError) as e:
        rlq.check()
    assert e.value.status == 5 and "diagnostic" in str(e.value)
    rlq.check()  # the error word was cleared
    # the context still works: a quantizer and a GEMM run and match the oracle
    x = I.to_bf16_bits(I.normal(3, "x", (64, 256), 1.0))
    w = I.to_bf16_bits(I.normal(3, "w", (256, 256), 0.02))
    qx, sx, _, _ = rlq.quant_act_1x128(to_dev(x))
    qw, sw, _ = rlq.quant_weight_128x128(to_dev(w))
    y = rlq.gemm_fprop(qx, sx, qw, sw)
    rlq.check()
    oqx, osx = oracle.quant_rows_1x128(x)
    assert np.array_equal(np_(qx), oqx)
    ref = oracle.gemm_fprop(oqx, osx, *oracle.quant_weight_128x128(w)[:2])
    assert np.linalg.norm(y.float().cpu().numpy() - ref) <= 2e-3 * np.linalg.norm(ref)


def test_invalid_arguments_raise_before_launch():
    x = torch.zeros((4, 100), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rlq.RlqError) as e:
        rlq.quant_act_1x128(x)
    assert e.value.status == 2
    rlq.check()


@pytest.mark.parametrize("kind", ["fprop", "wgrad"])
def test_gemm_abort_path_reports_timeout_and_context_survives(kind):
    """The block-scaled GEMM's own bounded waits: with the stall diagnostic
    armed, the next GEMM runs on single CTAs whose producer withholds its first
    stage's loads.  The MMA warp's wait runs out, the CTA raises its abort flag,
    drains its copies, frees its tensor memory and exits; rlq_check reports the
    timeout, the error word clears, and the same GEMM then matches the oracle."""
    M, N, K = 1024, 512, 1024  # 8 contraction blocks per tile either way: one stage withheld, three in flight
    x = I.to_bf16_bits(I.normal(11, "x", (M, K), 1.0))
    w = I.to_bf16_bits(I.normal(11, "w", (N, K), 0.02))
    qx, sx, qxT, sxc = rlq.quant_act_1x128(to_dev(x), colwise=True)
    qw, sw, _ = rlq.quant_weight_128x128(to_dev(w))
    rlq.check()

    def run():
        if kind == "fprop":
            return rlq.gemm_fprop(qx, sx, qw, sw)
        return rlq.gemm_wgrad(qxT, sxc, qxT, sxc)  # dX^T X-shaped: [K, K] over M tokens

    rlq.rlq_diag_arm_gemm_stall()
    run()
    with pytest.raises(rlq.RlqError) as e:
        rlq.check()
    assert e.value.status == 5 and "device-side wait ran out" in str(e.value)
    rlq.check()  # cleared
    got = run()
    rlq.check()
    oqx, osx = oracle.quant_rows_1x128(x)
    if kind == "fprop":
        oqw, osw, _ = oracle.quant_weight_128x128(w)
        ref = oracle.gemm_fprop(oqx, osx, oqw, osw)
    else:
        oqxT, osxc = oracle.quant_cols_128x1(x)
        assert np.array_equal(np_(qxT), oqxT)
        ref = oracle.gemm_wgrad(oqxT, osxc, oqxT, osxc)
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.linalg.norm(g - ref) <= 2e-3 * np.linalg.norm(ref)
    assert not (np.abs(g - ref) > 1e-2 * (np.abs(ref) + 1)).any()
