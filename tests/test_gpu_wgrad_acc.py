"""GPU parity of WGrad accumulated into an fp32 gradient (micro-batch
accumulation) through the C ABI, against the oracle's fp64 WGrad."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_quantize_gb300 import rlq
from gpu_util import normal_bits, np_, to_dev

pytestmark = pytest.mark.gpu


def _operands(seed, M, N, K):
    x = normal_bits(seed, (M, K))
    dy = normal_bits(seed + 1, (M, N), std=1e-3)
    _, _, qxT, sxc = rlq.quant_act_1x128(to_dev(x), colwise=True)
    _, _, qdyT, sdyc = rlq.quant_act_1x128(to_dev(dy), colwise=True)
    return qdyT, sdyc, qxT, sxc


def _ref(qdyT, sdyc, qxT, sxc):
    return oracle.gemm_wgrad(np_(qdyT), np_(sdyc), np_(qxT), np_(sxc))


def _assert_fp32_close(got, want, what):
    """fp32 accumulation of 128-blocks: relative Frobenius error far below bf16's."""
    g = got.cpu().numpy().astype(np.float64)
    err = np.linalg.norm(g - want) / np.linalg.norm(want)
    assert err <= 1e-5, f"{what}: relative Frobenius error {err:.2e}"


@pytest.mark.parametrize("M,N,K", [(200, 256, 384), (1024, 384, 256), (8192, 1024, 512)])
def test_accumulate_onto_existing_gradient(M, N, K):
    qdyT, sdyc, qxT, sxc = _operands(60, M, N, K)
    rng = np.random.default_rng(61)
    acc0 = (rng.standard_normal((N, K)) * 1e-2).astype(np.float32)
    acc = torch.from_numpy(acc0.copy()).cuda()
    rlq.gemm_wgrad_accumulate_(acc, qdyT, sdyc, qxT, sxc)
    rlq.check()
    ref = _ref(qdyT, sdyc, qxT, sxc)
    _assert_fp32_close(acc - torch.from_numpy(acc0).cuda(), ref, f"increment {M}x{N}x{K}")
    _assert_fp32_close(acc, acc0.astype(np.float64) + ref, f"accumulated {M}x{N}x{K}")


def test_two_micro_batches_sum():
    N, K = 256, 384
    a = _operands(62, 640, N, K)
    b = _operands(64, 300, N, K)
    acc = torch.zeros((N, K), dtype=torch.float32, device="cuda")
    rlq.gemm_wgrad_accumulate_(acc, *a)
    rlq.gemm_wgrad_accumulate_(acc, *b)
    rlq.check()
    _assert_fp32_close(acc, _ref(*a) + _ref(*b), "two micro-batches")


@pytest.mark.parametrize("M,N,K", [(1, 256, 128), (100, 512, 256), (128, 256, 384), (4096, 2048, 1024)])
def test_accumulate_from_the_epilogue_without_workspace(M, N, K):
    """No workspace: the GEMM's epilogue adds each tile's fp32 result into the
    gradient (single CTAs and CTA pairs, one token block or many)."""
    qdyT, sdyc, qxT, sxc = _operands(68, M, N, K)
    rng = np.random.default_rng(69)
    acc0 = (rng.standard_normal((N, K)) * 1e-2).astype(np.float32)
    acc = torch.from_numpy(acc0.copy()).cuda()
    rlq.rlq_gemm_wgrad_accumulate(qdyT.data_ptr(), qdyT.stride(0), sdyc.data_ptr(), sdyc.stride(0), qxT.data_ptr(),
                                  qxT.stride(0), sxc.data_ptr(), sxc.stride(0), acc.data_ptr(), K, M, N, K, None, 0,
                                  torch.cuda.current_stream().cuda_stream)
    rlq.check()
    ref = _ref(qdyT, sdyc, qxT, sxc)
    _assert_fp32_close(acc - torch.from_numpy(acc0).cuda(), ref, f"increment {M}x{N}x{K}")


def test_epilogue_accumulate_from_zero_rounds_to_the_single_pass_wgrad():
    """From zero and without a workspace, the fp32 result rounded to bf16 equals the
    single-pass WGrad's output bit for bit (same promotion order)."""
    M, N, K = 1024, 512, 768
    qdyT, sdyc, qxT, sxc = _operands(70, M, N, K)
    acc = torch.zeros((N, K), dtype=torch.float32, device="cuda")
    rlq.rlq_gemm_wgrad_accumulate(qdyT.data_ptr(), qdyT.stride(0), sdyc.data_ptr(), sdyc.stride(0), qxT.data_ptr(),
                                  qxT.stride(0), sxc.data_ptr(), sxc.stride(0), acc.data_ptr(), K, M, N, K, None, 0,
                                  torch.cuda.current_stream().cuda_stream)
    dw = rlq.gemm_wgrad(qdyT, sdyc, qxT, sxc)
    rlq.check()
    assert torch.equal(acc.to(torch.bfloat16), dw)


def test_accumulate_from_zero_rounds_to_the_split_k_wgrad():
    """From a zero gradient with the split-K plan's workspace, the fp32 result rounded
    to bf16 is the split-K WGrad's output bit for bit (same splits, same order)."""
    M, N, K = 2048, 256, 384
    qdyT, sdyc, qxT, sxc = _operands(66, M, N, K)
    nbytes = rlq.rlq_gemm_splitk_workspace_bytes(rlq.GEMM_WGRAD, M, N, K)
    assert nbytes >= 2 * N * K * 4  # the plan splits this few-tile shape
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    acc = torch.zeros((N, K), dtype=torch.float32, device="cuda")
    rlq.gemm_wgrad_accumulate_(acc, qdyT, sdyc, qxT, sxc, workspace=ws)
    dw = rlq.gemm_wgrad(qdyT, sdyc, qxT, sxc, split_k=True, workspace=ws)
    rlq.check()
    assert torch.equal(acc.to(torch.bfloat16), dw)
