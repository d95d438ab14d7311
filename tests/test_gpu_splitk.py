"""GPU parity of the split-K GEMM entry points (caller-provided workspace).

Split-K changes only the order of the fp32 sum over contraction blocks (each
split sums a contiguous range, then the splits are added in order), so:

* against the fp64 oracle the usual GEMM tolerance holds;
* integer-valued operands (every partial sum exact in fp32) give bit-exact
  bf16 outputs, whatever the split;
* repeated calls give identical bits (no atomics);
* a workspace too small for any split runs the single-pass kernel and gives
  its bits exactly.
Every shape here is chosen so that the library's plan does split; the tests
assert that first.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_quantize_gb300 import inputs as I
from fp8_block_scaled_quantize_gb300 import rlq
from gpu_util import assert_gemm_close, normal_bits, np_, to_dev, u16

pytestmark = pytest.mark.gpu

# (M, N, K): FProp / DGrad contract over K / N, WGrad over M
SHAPES = [(1, 256, 4096), (200, 384, 2048), (129, 640, 3072), (64, 512, 4096)]
WGRAD_SHAPES = [(4096, 128, 256), (3000, 256, 384), (2049, 384, 128)]


def _splits(kind, M, N, K):
    return rlq.rlq_gemm_splitk_workspace_bytes(kind, M, N, K)


def _operands(M, N, K, seed):
    x = normal_bits(seed, (M, K), 1.0, "x")
    w = normal_bits(seed, (N, K), 0.02, "w")
    dy = normal_bits(seed, (M, N), 1e-3, "dy")
    g = {}
    g["qx"], g["sx"], g["qxT"], g["sxc"] = rlq.quant_act_1x128(to_dev(x), colwise=True)
    g["qdy"], g["sdy"], g["qdyT"], g["sdyc"] = rlq.quant_act_1x128(to_dev(dy), colwise=True)
    g["qw"], g["sw"], g["qwT"] = rlq.quant_weight_128x128(to_dev(w), transposed=True)
    return g


def test_plan_splits_few_tile_shapes_only():
    # 32B down projection at decode M: 20 output tiles, 216 contraction blocks
    assert _splits(rlq.GEMM_FPROP, 64, 5120, 27648) > 0
    # 8B training step: 1792 tiles fill every SM many times over
    assert _splits(rlq.GEMM_FPROP, 8192, 14336, 4096) == 0
    assert _splits(rlq.GEMM_DGRAD, 8192, 14336, 4096) == 0
    # too short a contraction to split
    assert _splits(rlq.GEMM_FPROP, 64, 256, 512) == 0
    for M, N, K in SHAPES:
        assert _splits(rlq.GEMM_FPROP, M, N, K) > 0
        assert _splits(rlq.GEMM_DGRAD, M, K, N) > 0  # DGrad contracts over N
    for M, N, K in WGRAD_SHAPES:
        assert _splits(rlq.GEMM_WGRAD, M, N, K) > 0
    # the workspace holds splits fp32 planes of the output
    b = _splits(rlq.GEMM_FPROP, 200, 384, 2048)
    assert b % (200 * 384 * 4) == 0 and 2 <= b // (200 * 384 * 4) <= 16


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_fprop_splitk_parity(M, N, K):
    g = _operands(M, N, K, 50)
    y = rlq.gemm_fprop(g["qx"], g["sx"], g["qw"], g["sw"], split_k=True)
    rlq.check()
    assert_gemm_close(y, oracle.gemm_fprop(np_(g["qx"]), np_(g["sx"]), np_(g["qw"]), np_(g["sw"])), "FProp split-K")


@pytest.mark.parametrize("M,N,K", [(1, 4096, 256), (200, 2048, 384), (129, 3072, 640), (64, 4096, 512)])
@pytest.mark.parametrize("transposed", [True, False])
def test_dgrad_splitk_parity(M, N, K, transposed):
    assert _splits(rlq.GEMM_DGRAD, M, N, K) > 0
    g = _operands(M, N, K, 51)
    w = g["qwT"] if transposed else g["qw"]
    dx = rlq.gemm_dgrad(g["qdy"], g["sdy"], w, g["sw"], transposed=transposed, split_k=True)
    rlq.check()
    ref = oracle.gemm_dgrad(np_(g["qdy"]), np_(g["sdy"]), np_(g["qw"]), np_(g["sw"]))
    assert_gemm_close(dx, ref, "DGrad split-K")


@pytest.mark.parametrize("M,N,K", WGRAD_SHAPES)
def test_wgrad_splitk_parity(M, N, K):
    g = _operands(M, N, K, 52)
    dw = rlq.gemm_wgrad(g["qdyT"], g["sdyc"], g["qxT"], g["sxc"], split_k=True)
    rlq.check()
    ref = oracle.gemm_wgrad(np_(g["qdyT"]), np_(g["sdyc"]), np_(g["qxT"]), np_(g["sxc"]))
    assert_gemm_close(dw, ref, "WGrad split-K")


def _int_codes(rng, shape, lim=16):
    return oracle.e4m3_encode(rng.integers(-lim, lim + 1, size=shape).astype(np.float32))


def _bf16_of(ref):
    return torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("M,N,K", [(3, 2048, 2048), (130, 2048, 1536)])
def test_integer_splitk_bit_exact(M, N, K):
    """Integer codes with power-of-two scales: every partial sum is exact in
    fp32, so the split outputs equal the oracle's rounded to bf16 bit for bit."""
    assert _splits(rlq.GEMM_FPROP, M, N, K) > 0 and _splits(rlq.GEMM_DGRAD, M, N, K) > 0
    rng = np.random.default_rng(M + N + K)
    qx, qw, qdy = _int_codes(rng, (M, K)), _int_codes(rng, (N, K)), _int_codes(rng, (M, N))
    sx = np.full((K // 128, M), 2.0 ** -7, np.float32)
    sw = np.full((N // 128, K // 128), 1.0, np.float32)
    sdy = np.full((N // 128, M), 2.0 ** -7, np.float32)
    y = rlq.gemm_fprop(_dev(qx), _dev(sx), _dev(qw), _dev(sw), split_k=True)
    dx = rlq.gemm_dgrad(_dev(qdy), _dev(sdy), _dev(qw.T), _dev(sw), transposed=True, split_k=True)
    dx_mn = rlq.gemm_dgrad(_dev(qdy), _dev(sdy), _dev(qw), _dev(sw), transposed=False, split_k=True)
    rlq.check()
    assert np.array_equal(u16(y), _bf16_of(oracle.gemm_fprop(qx, sx, qw, sw)))
    rdx = _bf16_of(oracle.gemm_dgrad(qdy, sdy, qw, sw))
    assert np.array_equal(u16(dx), rdx) and np.array_equal(u16(dx_mn), rdx)


@pytest.mark.parametrize("M,N,K", [(1500, 128, 256), (2049, 256, 128)])
def test_integer_wgrad_splitk_bit_exact(M, N, K):
    assert _splits(rlq.GEMM_WGRAD, M, N, K) > 0
    rng = np.random.default_rng(M + N + K + 1)
    qdy, qx = _int_codes(rng, (M, N)), _int_codes(rng, (M, K))
    MB, ldm = (M + 127) // 128, (M + 15) // 16 * 16
    qdyT = np.zeros((N, ldm), np.uint8)
    qdyT[:, :M] = qdy.T
    qxT = np.zeros((K, ldm), np.uint8)
    qxT[:, :M] = qx.T
    sdyc = np.full((MB, N), 2.0 ** -7, np.float32)
    sxc = np.full((MB, K), 1.0, np.float32)
    dw = rlq.gemm_wgrad(_dev(qdyT)[:, :M], _dev(sdyc), _dev(qxT)[:, :M], _dev(sxc), split_k=True)
    rlq.check()
    assert np.array_equal(u16(dw), _bf16_of(oracle.gemm_wgrad(qdyT[:, :M], sdyc, qxT[:, :M], sxc)))


def test_splitk_repeatable_and_close_to_single_pass():
    M, N, K = 200, 384, 2048
    g = _operands(M, N, K, 53)
    ys = [u16(rlq.gemm_fprop(g["qx"], g["sx"], g["qw"], g["sw"], split_k=True)) for _ in range(3)]
    y1 = rlq.gemm_fprop(g["qx"], g["sx"], g["qw"], g["sw"])
    rlq.check()
    assert all(np.array_equal(ys[0], y) for y in ys[1:])
    # the two sum orders differ by at most a few bf16 ulps
    a = torch.from_numpy(ys[0].view(np.int16)).view(torch.bfloat16).float()
    b = y1.float().cpu()
    assert torch.all((a - b).abs() <= 2.0 ** -6 * b.abs() + 1e-6)


def test_small_workspace_runs_single_pass_bits():
    M, N, K = 64, 512, 4096
    g = _operands(M, N, K, 54)
    y1 = rlq.gemm_fprop(g["qx"], g["sx"], g["qw"], g["sw"])
    tiny = torch.empty(1024, dtype=torch.uint8, device="cuda")  # too small for two fp32 planes
    y2 = rlq.gemm_fprop(g["qx"], g["sx"], g["qw"], g["sw"], split_k=True, workspace=tiny)
    y3 = torch.empty_like(y1)
    s = torch.cuda.current_stream().cuda_stream
    rlq.rlq_gemm_fprop_splitk(g["qx"].data_ptr(), K, g["sx"].data_ptr(), M, g["qw"].data_ptr(), K,
                              g["sw"].data_ptr(), K // 128, y3.data_ptr(), N, M, N, K, None, 0, s)
    # a workspace with room for two planes but not the full plan: still within tolerance
    two = torch.empty(2 * M * N * 4, dtype=torch.uint8, device="cuda")
    y4 = rlq.gemm_fprop(g["qx"], g["sx"], g["qw"], g["sw"], split_k=True, workspace=two)
    rlq.check()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))
    assert_gemm_close(y4, oracle.gemm_fprop(np_(g["qx"]), np_(g["sx"]), np_(g["qw"]), np_(g["sw"])), "2 planes")


def test_misaligned_or_negative_workspace_rejected():
    M, N, K = 64, 256, 2048
    g = _operands(M, N, K, 55)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    args = (g["qx"].data_ptr(), K, g["sx"].data_ptr(), M, g["qw"].data_ptr(), K, g["sw"].data_ptr(), K // 128,
            y.data_ptr(), N, M, N, K)
    with pytest.raises(rlq.RlqError) as e:
        rlq.rlq_gemm_fprop_splitk(*args, ws.data_ptr() + 4, (1 << 20) - 4, s)
    assert e.value.status == 3
    with pytest.raises(rlq.RlqError) as e:
        rlq.rlq_gemm_fprop_splitk(*args, ws.data_ptr(), -1, s)
    assert e.value.status == 1
    with pytest.raises(rlq.RlqError) as e:
        rlq.rlq_gemm_splitk_workspace_bytes(7, M, N, K)
    assert e.value.status == 1
    rlq.check()


@pytest.mark.parametrize("M", [1, 64, 256])
def test_sweep_32b_down_decode_splitk_sampled(M):
    """The 32B down projection (N=5120, K=27648) at decode-sized M, split-K
    FProp and DGrad as the sweep times them, against the oracle."""
    d = I.sweep_32b(M, "down")
    qx, sx, _, _ = rlq.quant_act_1x128(to_dev(d["x"]))
    qdy, sdy, _, _ = rlq.quant_act_1x128(to_dev(d["dy"]))
    qw, sw, qwT = rlq.quant_weight_128x128(to_dev(d["w"]), transposed=True)
    assert _splits(rlq.GEMM_FPROP, M, qw.shape[0], qw.shape[1]) > 0
    y = rlq.gemm_fprop(qx, sx, qw, sw, split_k=True)
    dx = rlq.gemm_dgrad(qdy, sdy, qwT, sw, transposed=True, split_k=True)
    rlq.check()
    rows = np.sort(np.random.default_rng(M).choice(M, size=min(M, 32), replace=False))
    hqw, hsw = np_(qw), np_(sw)
    ri = torch.from_numpy(rows).cuda()
    assert_gemm_close(y[ri], oracle.gemm_fprop(np_(qx), np_(sx), hqw, hsw, rows=rows), f"FProp 32B down M={M}")
    assert_gemm_close(dx[ri], oracle.gemm_dgrad(np_(qdy), np_(sdy), hqw, hsw, rows=rows), f"DGrad 32B down M={M}")
