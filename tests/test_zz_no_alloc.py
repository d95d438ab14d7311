"""The allocation-free split-K FProp (library-owned static scratch), through
the C ABI, against the split-K entry point that takes a caller's workspace.

Collected last, so it runs both after every other test in the process and, on
its own, in a fresh process (the first call on the device sets up the scratch).
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_quantize_gb300 import rlq
from gpu_util import ELEM_ABS, REL_FRO, normal_bits, to_dev

pytestmark = pytest.mark.gpu


def _quantized(M, N, K, seed):
    qx, sx, _, _ = rlq.quant_act_1x128(to_dev(normal_bits(seed, (M, K), 1.0, "x")))
    qw, sw, _ = rlq.quant_weight_128x128(to_dev(normal_bits(seed, (N, K), 0.02, "w")))
    return qx, sx, qw, sw


def _static_fprop(qx, sx, qw, sw, y, stream=None):
    M, K = qx.shape
    N = qw.shape[0]
    st = (stream or torch.cuda.current_stream()).cuda_stream
    rlq.rlq_gemm_fprop_splitk_static(qx.data_ptr(), K, sx.data_ptr(), M, qw.data_ptr(), K, sw.data_ptr(), K // 128,
                                     y.data_ptr(), N, M, N, K, st)


def _assert_close(got, ref, what):
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    err = g - r
    assert np.linalg.norm(err) <= REL_FRO * np.linalg.norm(r), what
    assert not (np.abs(err) > ELEM_ABS * (np.abs(r) + 1)).any(), what


@pytest.mark.parametrize("M,N,K", [(64, 512, 4096), (129, 640, 3072)])
def test_static_scratch_matches_workspace_entry_point_twice(M, N, K):
    need = rlq.rlq_gemm_splitk_workspace_bytes(rlq.GEMM_FPROP, M, N, K)
    assert 0 < need <= rlq.STATIC_SCRATCH_BYTES  # the plan splits and uses the scratch
    # two calls in a row on different data: the second must not see the first's partials
    for seed in (70, 71):
        qx, sx, qw, sw = _quantized(M, N, K, seed)
        ref = rlq.gemm_fprop(qx, sx, qw, sw, split_k=True)
        y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
        _static_fprop(qx, sx, qw, sw, y)
        rlq.check()
        _assert_close(y, ref, f"static-scratch FProp, seed {seed}")


def test_static_scratch_on_a_side_stream_twice():
    """Two calls in a row on a stream other than the default one, each synced
    and checked: the scratch's address holds for every stream of the context."""
    M, N, K = 64, 512, 4096
    side = torch.cuda.Stream()
    for seed in (72, 73):
        qx, sx, qw, sw = _quantized(M, N, K, seed)
        ref = rlq.gemm_fprop(qx, sx, qw, sw, split_k=True)
        torch.cuda.synchronize()
        y = torch.full((M, N), -3.0, dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        _static_fprop(qx, sx, qw, sw, y, stream=side)
        rlq.check(side)
        torch.cuda.synchronize()
        _assert_close(y, ref, f"static-scratch FProp on a side stream, seed {seed}")


def test_plan_beyond_static_scratch_is_rejected():
    M, N, K = 1024, 5120, 27648  # the plan needs more than one 20 MiB fp32 plane
    need = rlq.rlq_gemm_splitk_workspace_bytes(rlq.GEMM_FPROP, M, N, K)
    assert need > rlq.STATIC_SCRATCH_BYTES
    y = torch.empty(1, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rlq.RlqError) as e:
        rlq.rlq_gemm_fprop_splitk_static(0x10000, K, 0x10000, M, 0x10000, K, 0x10000, K // 128, y.data_ptr(), N,
                                         M, N, K, torch.cuda.current_stream().cuda_stream)
    assert e.value.status == 2 and "static" in str(e.value)
    rlq.check()
