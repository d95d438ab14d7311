"""GPU parity of the NVFP4 weight-only GEMM (QeRL news article: the rollout's
FP4 x BF16 GEMM with NVFP4 weights) through the C ABI, against the oracle's fp64
gemm_nvfp4_weight_only over the oracle's own codes.

* Tolerance of the other GEMM tests: relative Frobenius <= 2e-3 and per element
  |err| <= 1e-2 * (|ref| + 1) on the bf16 output.
* Exact pin: integer activations, block scales that are powers of two and a tensor
  scale of 1 give fp32 sums that are exact: the GPU output must equal the exact
  result rounded to bf16, bit for bit.
* The weights come from the GPU quantizer, whose codes are first asserted equal to
  the oracle's; then the workloads' shapes (8B decode, Qwen2.5-7B layers, 32B at
  decode sizes), ragged M, a pitched layout and the empty contraction.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_quantize_gb300 import inputs as I
from fp8_block_scaled_quantize_gb300 import rlq
from gpu_util import assert_gemm_close, idx, normal_bits, np_, strata, to_dev, u16

pytestmark = pytest.mark.gpu

DECODE_MAX_M = 4        # batches of up to this many tokens run the CUDA-core kernel ...
DECODE_SPLIT_MAX_M = 2  # ... also through the split-K entry point (no workspace planned)


def _unpack(qp: np.ndarray) -> np.ndarray:
    lo, hi = qp & 0xF, qp >> 4
    return np.stack([lo, hi], axis=-1).reshape(qp.shape[0], -1)


def _pack(q: np.ndarray) -> np.ndarray:
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)


def _padded(a: np.ndarray) -> torch.Tensor:
    """A device view of `a` whose rows start 16 bytes apart (the pitch rule for
    codes and block scales)."""
    rows, cols = a.shape
    buf = torch.zeros((rows, (cols + 15) // 16 * 16), dtype=torch.uint8, device="cuda")
    buf[:, :cols] = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return buf[:, :cols]


def _quantized_weight(w_bits):
    """GPU NVFP4 quantization, asserted equal to the oracle's; returns both."""
    q, sb, st = rlq.quant_nvfp4(to_dev(w_bits))
    rlq.check()
    oq, osb, ost = oracle.quant_nvfp4(w_bits)
    assert np_(st)[0] == np.float32(ost)
    assert np.array_equal(np_(sb), osb)
    assert np.array_equal(_unpack(np_(q)), oq)
    return (q, sb, st), (oq, osb, ost)


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (5, 256, 128), (128, 256, 256), (200, 384, 320),
                                   (300, 640, 1024), (129, 128, 2048)])
def test_parity_small_shapes(M, N, K):
    x = normal_bits(90, (M, K), 1.0, "x")
    w = normal_bits(90, (N, K), 0.02, "w")
    (q, sb, st), (oq, osb, ost) = _quantized_weight(w)
    y = rlq.gemm_nvfp4_weight_only(to_dev(x), q, sb, st)
    rlq.check()
    assert_gemm_close(y, oracle.gemm_nvfp4_weight_only(x, oq, osb, ost), f"NVFP4 GEMM {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(3, 128, 64), (130, 256, 512), (64, 512, 1280)])
def test_integer_case_bit_exact(M, N, K):
    """x integers in [-4, 4], E2M1 codes at random, block scales 1/2, 1 and 2 (E4M3
    codes 0x30, 0x38, 0x40), st = 1: every product is a multiple of 1/4 of at most
    48 in magnitude and every partial sum a multiple of 1/4 below 2^17, so the fp32
    sum is exact whatever its order; the GPU's bf16 output must then be the exact
    result rounded to bf16, bit for bit."""
    rng = np.random.default_rng(M + N + K)
    x = I.to_bf16_bits(rng.integers(-4, 5, size=(M, K)).astype(np.float32))
    q = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    sb = rng.choice(np.array([0x30, 0x38, 0x40], np.uint8), size=(N, K // 16))
    ref = oracle.gemm_nvfp4_weight_only(x, q, sb, 1.0)
    assert np.all(ref * 4 == np.round(ref * 4)) and np.all(np.abs(ref) < 2 ** 17)
    qp = _padded(_pack(q))
    sbd = _padded(sb)
    st = torch.ones(1, dtype=torch.float32, device="cuda")
    y = rlq.gemm_nvfp4_weight_only(to_dev(x), qp, sbd, st)
    rlq.check()
    assert np.array_equal(u16(y), I.to_bf16_bits(ref.astype(np.float32)))


def test_decode_upproj_8b_full_size():
    d = I.decode_upproj_8b()
    (q, sb, st), (oq, osb, ost) = _quantized_weight(d["w"])
    y = rlq.gemm_nvfp4_weight_only(to_dev(d["x"]), q, sb, st)
    rlq.check()
    rng = np.random.default_rng(91)
    cols = strata(14336, 64, rng)
    ref = oracle.gemm_nvfp4_weight_only(d["x"], oq, osb, ost, cols=cols)
    assert_gemm_close(y[:, idx(cols)], ref, "NVFP4 GEMM, 8B decode up-projection")


@pytest.mark.parametrize("which", ["gate_up", "down"])
@pytest.mark.parametrize("M", [64, 512])
def test_qwen7b_layers(which, M):
    d = I.qwen7b_layer(M, which)
    (q, sb, st), (oq, osb, ost) = _quantized_weight(d["w"])
    y = rlq.gemm_nvfp4_weight_only(to_dev(d["x"]), q, sb, st)
    rlq.check()
    N = d["w"].shape[0]
    rng = np.random.default_rng(M + N)
    rows = np.arange(M) if M <= 64 else strata(M, 16, rng)
    cols = strata(N, 32, rng)
    ref = oracle.gemm_nvfp4_weight_only(d["x"], oq, osb, ost, rows=rows, cols=cols)
    assert_gemm_close(y[idx(rows)][:, idx(cols)], ref, f"NVFP4 GEMM qwen7b {which} M={M}")


@pytest.mark.parametrize("orient", ["up", "down"])
@pytest.mark.parametrize("M", [1, 16, 64])
def test_sweep_32b_decode(orient, M):
    d = I.sweep_32b(M, orient, with_dy=False)
    (q, sb, st), (oq, osb, ost) = _quantized_weight(d["w"])
    y = rlq.gemm_nvfp4_weight_only(to_dev(d["x"]), q, sb, st)
    rlq.check()
    N = d["w"].shape[0]
    cols = strata(N, 64, np.random.default_rng(M))
    ref = oracle.gemm_nvfp4_weight_only(d["x"], oq, osb, ost, cols=cols)
    assert_gemm_close(y[:, idx(cols)], ref, f"NVFP4 GEMM 32B {orient} M={M}")


def test_pitched_operands_and_guard_bands():
    M, N, K = 70, 256, 512
    x = normal_bits(92, (M, K), 1.0, "x")
    w = normal_bits(92, (N, K), 0.02, "w")
    oq, osb, ost = oracle.quant_nvfp4(w)
    dev = "cuda"
    xb = torch.zeros((M, K + 24), dtype=torch.bfloat16, device=dev)
    xb[:, :K] = to_dev(x)
    qb = torch.zeros((N, K // 2 + 48), dtype=torch.uint8, device=dev)
    qb[:, :K // 2] = torch.from_numpy(_pack(oq)).cuda()
    sbb = torch.zeros((N, K // 16 + 16), dtype=torch.uint8, device=dev)
    sbb[:, :K // 16] = torch.from_numpy(osb).cuda()
    st = torch.tensor([ost], dtype=torch.float32, device=dev)
    yb = torch.full((M, N + 40), 3.0, dtype=torch.bfloat16, device=dev)
    rlq.rlq_gemm_nvfp4_weight_only(xb.data_ptr(), K + 24, qb.data_ptr(), K // 2 + 48, sbb.data_ptr(), K // 16 + 16,
                                   st.data_ptr(), yb.data_ptr(), N + 40, M, N, K,
                                   torch.cuda.current_stream().cuda_stream)
    rlq.check()
    assert_gemm_close(yb[:, :N], oracle.gemm_nvfp4_weight_only(x, oq, osb, ost), "pitched NVFP4 GEMM")
    assert torch.all(yb[:, N:] == 3.0)


def test_empty_contraction_and_validation():
    dev = "cuda"
    y = torch.full((4, 128), 5.0, dtype=torch.bfloat16, device=dev)
    st = torch.ones(1, dtype=torch.float32, device=dev)
    rlq.rlq_gemm_nvfp4_weight_only(None, 0, None, 0, None, 0, st.data_ptr(), y.data_ptr(), 128, 4, 128, 0,
                                   torch.cuda.current_stream().cuda_stream)
    rlq.check()
    assert torch.all(y == 0)
    x = torch.zeros((4, 96), dtype=torch.bfloat16, device=dev)
    with pytest.raises(rlq.RlqError) as e:  # K % 64
        rlq.rlq_gemm_nvfp4_weight_only(x.data_ptr(), 96, x.data_ptr(), 48, x.data_ptr(), 16, st.data_ptr(),
                                       y.data_ptr(), 128, 4, 128, 96, 0)
    assert e.value.status == 2
    rlq.check()


def _ws(M, N, K):
    nb = rlq.rlq_gemm_splitk_workspace_bytes(rlq.GEMM_NVFP4_WEIGHT_ONLY, M, N, K)
    return nb, (torch.empty(nb, dtype=torch.uint8, device="cuda") if nb else None)


@pytest.mark.parametrize("M,N,K", [(5, 128, 4096), (16, 256, 8192), (130, 384, 2048), (5, 128, 4288),
                                   (7, 640, 3392)])
def test_splitk_parity(M, N, K):
    """Shapes whose output has far fewer tiles than the GPU has SMs: the plan
    splits K (asserted), including splits whose last range is not a whole raw
    chunk (K / 64 = 67 and 53 stages)."""
    nb, ws = _ws(M, N, K)
    assert nb > 0 and nb % (4 * M * N) == 0, nb
    x = normal_bits(93, (M, K), 1.0, "x")
    w = normal_bits(93, (N, K), 0.02, "w")
    (q, sb, st), (oq, osb, ost) = _quantized_weight(w)
    y = rlq.gemm_nvfp4_weight_only(to_dev(x), q, sb, st, split_k=True, workspace=ws)
    y1 = rlq.gemm_nvfp4_weight_only(to_dev(x), q, sb, st)
    rlq.check()
    ref = oracle.gemm_nvfp4_weight_only(x, oq, osb, ost)
    assert_gemm_close(y, ref, f"split-K NVFP4 GEMM {M}x{N}x{K} ({nb // (4 * M * N)} splits)")
    assert_gemm_close(y1, ref, f"NVFP4 GEMM {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(5, 128, 4288), (64, 256, 8192)])
def test_splitk_integer_case_bit_exact(M, N, K):
    """The exact integer case of test_integer_case_bit_exact under a split plan:
    every split sum and their total are exact, so the split and single-pass
    outputs both equal the exact result rounded to bf16."""
    nb, ws = _ws(M, N, K)
    assert nb > 0
    rng = np.random.default_rng(M * 7 + K)
    x = I.to_bf16_bits(rng.integers(-4, 5, size=(M, K)).astype(np.float32))
    q = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    sb = rng.choice(np.array([0x30, 0x38, 0x40], np.uint8), size=(N, K // 16))
    ref = oracle.gemm_nvfp4_weight_only(x, q, sb, 1.0)
    assert np.all(ref * 4 == np.round(ref * 4)) and np.all(np.abs(ref) < 2 ** 17)
    qp, sbd = _padded(_pack(q)), _padded(sb)
    st = torch.ones(1, dtype=torch.float32, device="cuda")
    y = rlq.gemm_nvfp4_weight_only(to_dev(x), qp, sbd, st, split_k=True, workspace=ws)
    y1 = rlq.gemm_nvfp4_weight_only(to_dev(x), qp, sbd, st)
    rlq.check()
    exact = I.to_bf16_bits(ref.astype(np.float32))
    assert np.array_equal(u16(y), exact)
    assert np.array_equal(u16(y1), exact)


@pytest.mark.parametrize("case", ["32b_down_m1", "32b_down_m16", "qwen7b_down_m64"])
def test_splitk_down_projections(case):
    """The down projections at decode sizes (few output tiles, long contraction:
    the case the split plan is for; a single token runs the CUDA-core kernel in
    one pass, with no workspace)."""
    if case.startswith("32b"):
        M = int(case.split("_m")[1])
        d = I.sweep_32b(M, "down", with_dy=False)
    else:
        M = 64
        d = I.qwen7b_layer(M, "down")
    N, K = d["w"].shape
    nb, ws = _ws(M, N, K)
    assert (nb == 0) if M <= DECODE_SPLIT_MAX_M else (nb > 0)
    (q, sb, st), (oq, osb, ost) = _quantized_weight(d["w"])
    y = rlq.gemm_nvfp4_weight_only(to_dev(d["x"]), q, sb, st, split_k=True, workspace=ws)
    rlq.check()
    cols = strata(N, 64, np.random.default_rng(5))
    ref = oracle.gemm_nvfp4_weight_only(d["x"], oq, osb, ost, cols=cols)
    assert_gemm_close(y[:, idx(cols)], ref, f"split-K NVFP4 GEMM {case} ({nb // (4 * M * N)} splits)")


def test_splitk_workspace_limits():
    """A workspace smaller than the plan's lowers the split count (still within
    tolerance); none runs the single pass, bit-equal to the plain call; a
    misaligned workspace is rejected before any launch."""
    M, N, K = 16, 256, 8192
    nb, ws = _ws(M, N, K)
    splits = nb // (4 * M * N)
    assert splits >= 3
    x = normal_bits(94, (M, K), 1.0, "x")
    w = normal_bits(94, (N, K), 0.02, "w")
    (q, sb, st), (oq, osb, ost) = _quantized_weight(w)
    xd = to_dev(x)
    ref = oracle.gemm_nvfp4_weight_only(x, oq, osb, ost)
    small = torch.empty(2 * 4 * M * N, dtype=torch.uint8, device="cuda")
    y2 = rlq.gemm_nvfp4_weight_only(xd, q, sb, st, split_k=True, workspace=small)
    y1 = rlq.gemm_nvfp4_weight_only(xd, q, sb, st)
    y0 = torch.empty_like(y1)
    rlq.rlq_gemm_nvfp4_weight_only_splitk(xd.data_ptr(), K, q.data_ptr(), q.stride(0), sb.data_ptr(), sb.stride(0),
                                          st.data_ptr(), y0.data_ptr(), N, M, N, K, None, 0,
                                          torch.cuda.current_stream().cuda_stream)
    rlq.check()
    assert_gemm_close(y2, ref, "split-K NVFP4 GEMM with a 2-split workspace")
    assert torch.equal(y0, y1)
    with pytest.raises(rlq.RlqError) as e:
        rlq.rlq_gemm_nvfp4_weight_only_splitk(xd.data_ptr(), K, q.data_ptr(), q.stride(0), sb.data_ptr(),
                                              sb.stride(0), st.data_ptr(), y0.data_ptr(), N, M, N, K,
                                              ws.data_ptr() + 4, nb - 16, torch.cuda.current_stream().cuda_stream)
    assert e.value.status == 3
    rlq.check()


def _integer_case(M, N, K, seed):
    """Operands whose fp32 sums are exact in any order (see test_integer_case_bit_exact)."""
    rng = np.random.default_rng(seed)
    x = I.to_bf16_bits(rng.integers(-4, 5, size=(M, K)).astype(np.float32))
    q = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    sb = rng.choice(np.array([0x30, 0x38, 0x40], np.uint8), size=(N, K // 16))
    ref = oracle.gemm_nvfp4_weight_only(x, q, sb, 1.0)
    assert np.all(ref * 4 == np.round(ref * 4)) and np.all(np.abs(ref) < 2 ** 17)
    return x, q, sb, ref


@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K", [(128, 64), (256, 1088), (384, 4288), (128, 27648)])
def test_decode_kernel_parity(M, N, K):
    """Batches of up to four tokens (the CUDA-core kernel): contractions of 2 block
    pairs (two lanes busy), 34 pairs (past one warp's 32 lanes), 134 pairs (a
    ragged last step of loads) and the 32B down projection's 864 on 128 rows (the
    row group then shared by several warps); M = 3 leaves one token of the
    four-token kernel unused.  Through the split-K entry point one or two tokens
    plan no workspace and return the same bits; three or four take the split
    tensor-core path, within the same tolerance."""
    x = normal_bits(95 + M, (M, K), 1.0, "x")
    w = normal_bits(95, (N, K), 0.02, "w")
    (q, sb, st), (oq, osb, ost) = _quantized_weight(w)
    nb, ws = _ws(M, N, K)
    xd = to_dev(x)
    y = rlq.gemm_nvfp4_weight_only(xd, q, sb, st)
    y2 = rlq.gemm_nvfp4_weight_only(xd, q, sb, st, split_k=True, workspace=ws)
    rlq.check()
    ref = oracle.gemm_nvfp4_weight_only(x, oq, osb, ost)
    assert_gemm_close(y, ref, f"decode NVFP4 GEMM {M}x{N}x{K}")
    if M <= DECODE_SPLIT_MAX_M:
        assert nb == 0
        assert torch.equal(y, y2)
    else:
        assert_gemm_close(y2, ref, f"split-K NVFP4 GEMM {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1, 128, 4096), (2, 256, 1088), (3, 128, 4288), (4, 384, 2048)])
def test_decode_kernel_integer_case_bit_exact(M, N, K):
    """The exact integer case through the CUDA-core kernel: its fp32 sums run in
    another order than the tensor cores', and must still give the exact result
    rounded to bf16, bit for bit."""
    x, q, sb, ref = _integer_case(M, N, K, 17 * M + K)
    st = torch.ones(1, dtype=torch.float32, device="cuda")
    y = rlq.gemm_nvfp4_weight_only(to_dev(x), _padded(_pack(q)), _padded(sb), st)
    rlq.check()
    assert np.array_equal(u16(y), I.to_bf16_bits(ref.astype(np.float32)))


def test_decode_kernel_pitched_and_repeatable():
    """Pitched activations, codes, scales and output through the CUDA-core kernel
    (guard bands untouched), and a second call equal bit for bit (its additions run
    in a fixed order)."""
    M, N, K = 3, 256, 1024
    x = normal_bits(96, (M, K), 1.0, "x")
    w = normal_bits(96, (N, K), 0.02, "w")
    oq, osb, ost = oracle.quant_nvfp4(w)
    dev = "cuda"
    xb = torch.zeros((M, K + 40), dtype=torch.bfloat16, device=dev)
    xb[:, :K] = to_dev(x)
    qb = torch.zeros((N, K // 2 + 32), dtype=torch.uint8, device=dev)
    qb[:, :K // 2] = torch.from_numpy(_pack(oq)).cuda()
    sbb = torch.zeros((N, K // 16 + 32), dtype=torch.uint8, device=dev)
    sbb[:, :K // 16] = torch.from_numpy(osb).cuda()
    st = torch.tensor([ost], dtype=torch.float32, device=dev)
    outs = []
    for _ in range(2):
        yb = torch.full((M, N + 24), 3.0, dtype=torch.bfloat16, device=dev)
        rlq.rlq_gemm_nvfp4_weight_only(xb.data_ptr(), K + 40, qb.data_ptr(), K // 2 + 32, sbb.data_ptr(),
                                       K // 16 + 32, st.data_ptr(), yb.data_ptr(), N + 24, M, N, K,
                                       torch.cuda.current_stream().cuda_stream)
        rlq.check()
        assert torch.all(yb[:, N:] == 3.0)
        outs.append(yb[:, :N].clone())
    assert torch.equal(outs[0], outs[1])
    assert_gemm_close(outs[0], oracle.gemm_nvfp4_weight_only(x, oq, osb, ost), "pitched decode NVFP4 GEMM")


@pytest.mark.parametrize("M", [1, 3])
def test_decode_kernel_qwen7b_down(M):
    """The Qwen2.5-7B down projection (N 3584, K 18944) at one and three tokens:
    few row groups for the GPU's warps, so each group is shared by 4 (M = 1) or 8
    (M = 3) warps of a CTA whose partial sums meet in shared memory."""
    d = I.qwen7b_layer(M, "down")
    (q, sb, st), (oq, osb, ost) = _quantized_weight(d["w"])
    y = rlq.gemm_nvfp4_weight_only(to_dev(d["x"]), q, sb, st)
    rlq.check()
    N = d["w"].shape[0]
    cols = strata(N, 32, np.random.default_rng(M + 7))
    ref = oracle.gemm_nvfp4_weight_only(d["x"], oq, osb, ost, cols=cols)
    assert_gemm_close(y[:, idx(cols)], ref, f"decode NVFP4 GEMM qwen7b down M={M}")
