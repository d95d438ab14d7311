"""GPU parity of the per-token / per-channel FP8 path (QuRL notes, "损失函数 /
训练策略": channel-wise weights, token-wise activations) through the C ABI:
codes and scales bit-exact against the oracle, the replicated scale layout, and
the per-channel FProp within the GEMM tolerance (bit-exact on integer inputs)."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_quantize_gb300 import inputs as I
from fp8_block_scaled_quantize_gb300 import rlq
from gpu_util import assert_gemm_close, normal_bits, np_, to_dev

pytestmark = pytest.mark.gpu


def _check(x_bits, q, s, s_rep):
    oq, os_ = oracle.quant_per_row(x_bits)
    assert np.array_equal(np_(q), oq), "per-row codes differ"
    assert np.array_equal(np_(s), os_), "per-row scales differ"
    if s_rep is not None:
        assert np.array_equal(np_(s_rep), np.tile(os_, (x_bits.shape[1] // 128, 1))), "replicated scales differ"


# Few rows run one CTA per row, many rows (more than 64 per SM) one warp per row:
# the last two shapes take the warp path on GPUs of up to 312 SMs.
@pytest.mark.parametrize("M,K", [(1, 128), (7, 256), (300, 640), (4096, 4096), (64, 27648), (20000, 128),
                                 (20011, 1152), (33, 5120), (17, 16384), (9, 16512), (3, 32768), (5, 32896),
                                 (300, 3584), (1000, 18944), (40, 20480), (41, 24576), (42, 27648)])
def test_per_row_parity(M, K):
    """Rows held by one warp (K <= 4096), by one CTA (K <= 32768, 8 or 16 loads per
    thread, ragged ends) and streamed twice (longer rows)."""
    x = normal_bits(41, (M, K), std=0.02)
    q, s, s_rep = rlq.quant_per_row(to_dev(x))
    _check(x, q, s, s_rep)


def test_per_row_edge_rows():
    """All-zero and signed-zero rows, subnormal rows, rows scaled 2^-120 and
    2^100, and rows whose magnitudes differ by up to 2^60 from their neighbours."""
    rng = np.random.default_rng(42)
    M, K = 96, 384
    v = rng.standard_normal((M, K)).astype(np.float32)
    v *= np.exp2(rng.integers(-30, 31, size=(M, 1))).astype(np.float32)
    v[0] = 0.0
    v[1] = -0.0
    v[2, :128] = (np.arange(1, 129, dtype=np.uint32) << 16).view(np.float32)  # bf16 subnormals
    v[2, 128:] = 0.0
    v[3] *= np.float32(2.0 ** -120)
    v[4] = v[4] / np.abs(v[4]).max() * np.float32(2.0 ** 100)
    x = I.to_bf16_bits(v)
    q, s, s_rep = rlq.quant_per_row(to_dev(x))
    _check(x, q, s, s_rep)
    assert np_(s)[0] == 1.0 and np.all(np_(q)[0] == 0) and np.all(np_(q)[1] == 0x80)


def test_per_row_pitched_with_guard_bands():
    M, K = 130, 256
    x = normal_bits(43, (M, K))
    dev = "cuda"
    xb = torch.zeros((M, K + 64), dtype=torch.bfloat16, device=dev)
    xb[:, :K] = to_dev(x)
    qb = torch.full((M, K + 32), 0xA5, dtype=torch.uint8, device=dev)
    sb = torch.full((M + 8,), -7.0, dtype=torch.float32, device=dev)
    rb = torch.full((K // 128 + 1, M + 6), -9.0, dtype=torch.float32, device=dev)
    st = torch.cuda.current_stream().cuda_stream
    rlq.rlq_quant_per_row(xb.data_ptr(), M, K, K + 64, qb.data_ptr(), K + 32, sb.data_ptr(), rb.data_ptr(), M + 6, st)
    rlq.check()
    _check(x, qb[:, :K], sb[:M], rb[:K // 128, :M])
    assert torch.all(qb[:, K:] == 0xA5) and torch.all(sb[M:] == -7.0)
    assert torch.all(rb[:, M:] == -9.0) and torch.all(rb[K // 128:] == -9.0)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (200, 384, 640), (1000, 256, 4096), (300, 512, 27648)])
def test_per_channel_fprop_parity(M, N, K):
    x = normal_bits(44, (M, K))
    w = normal_bits(45, (N, K), std=0.02)
    qx, sx, sx_rep = rlq.quant_per_row(to_dev(x))
    qw, sw, sw_rep = rlq.quant_per_row(to_dev(w))
    y = rlq.gemm_fprop_per_channel(qx, sx_rep, qw, sw_rep)
    rlq.check()
    ref = oracle.gemm_per_channel(np_(qx), np_(sx), np_(qw), np_(sw))
    assert_gemm_close(y, ref, f"per-channel FProp {M}x{N}x{K}")


def test_per_channel_fprop_integer_bit_exact():
    """Unit scales and small-integer codes: every partial and sum is exact in fp32,
    so the output must be the exact integer product rounded once to bf16."""
    rng = np.random.default_rng(46)
    lut = oracle.e4m3_lut()
    ints = np.array([c for c in range(0x7F) if lut[c] == int(lut[c]) and abs(lut[c]) <= 4], np.uint8)
    M, N, K = 96, 256, 512
    qx = rng.choice(ints, size=(M, K)) | (rng.integers(0, 2, (M, K)) << 7).astype(np.uint8)
    qw = rng.choice(ints, size=(N, K)).astype(np.uint8)
    ones_x = torch.ones((K // 128, M), dtype=torch.float32, device="cuda")
    ones_w = torch.ones((K // 128, N), dtype=torch.float32, device="cuda")
    y = rlq.gemm_fprop_per_channel(torch.from_numpy(qx).cuda(), ones_x, torch.from_numpy(qw).cuda(), ones_w)
    rlq.check()
    exact = (lut[qx].astype(np.int64) @ lut[qw].astype(np.int64).T).astype(np.float32)
    assert np.array_equal(y.float().cpu().numpy(), oracle.bf16_round(exact))


def test_per_channel_fprop_qwen7b_gate_up_sampled():
    """Qwen2.5-7B gate/up shape at M=4096 (Student-t channels as in the layer set),
    compared on sampled rows and columns."""
    cfg = I.qwen7b_layer(4096, "gate_up")
    qx, sx, sx_rep = rlq.quant_per_row(to_dev(cfg["x"]))
    qw, sw, sw_rep = rlq.quant_per_row(to_dev(cfg["w"]))
    y = rlq.gemm_fprop_per_channel(qx, sx_rep, qw, sw_rep)
    rlq.check()
    rng = np.random.default_rng(47)
    rows = np.sort(rng.choice(qx.shape[0], 64, replace=False))
    cols = np.sort(rng.choice(qw.shape[0], 256, replace=False))
    ref = oracle.gemm_per_channel(np_(qx), np_(sx), np_(qw), np_(sw), rows=rows, cols=cols)
    assert_gemm_close(y[rows][:, cols], ref, "per-channel FProp qwen7b gate_up")



@pytest.mark.parametrize("M,N,K", [(64, 3584, 18944), (5, 1024, 4096)])
def test_per_channel_fprop_splitk_parity(M, N, K):
    """Decode-sized per-channel FProp through the split-K entry (the library's plan)."""
    x = normal_bits(48, (M, K))
    w = normal_bits(49, (N, K), std=0.02)
    qx, sx, sx_rep = rlq.quant_per_row(to_dev(x))
    qw, sw, sw_rep = rlq.quant_per_row(to_dev(w))
    if K >= 16384:  # a 148-block contraction over 14 tiles: the plan splits on any GB300-sized GPU
        assert rlq.rlq_gemm_splitk_workspace_bytes(rlq.GEMM_FPROP, M, N, K) > 0
    y = rlq.gemm_fprop_per_channel(qx, sx_rep, qw, sw_rep, split_k=True)
    y1 = rlq.gemm_fprop_per_channel(qx, sx_rep, qw, sw_rep)
    rlq.check()
    ref = oracle.gemm_per_channel(np_(qx), np_(sx), np_(qw), np_(sw))
    assert_gemm_close(y, ref, f"per-channel split-K FProp {M}x{N}x{K}")
    assert_gemm_close(y1, ref, f"per-channel FProp {M}x{N}x{K}")
