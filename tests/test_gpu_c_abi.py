"""The C ABI from C: tests/c_abi/example.c, compiled with gcc against
include/rlq.h and librlq.so (no Python in the caller), quantizes and runs
FProp and DGrad; its outputs must equal, bit for bit, what the Python binding
computes from the same inputs through the same entry points."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from fp8_block_scaled_quantize_gb300 import rlq

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
M, N, K, LDM = 200, 384, 512, 208


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def test_c_caller_matches_python_binding(tmp_path):
    lib = rlq.library_path()
    rlq.lib()
    cuda = _cuda_home()
    exe = str(tmp_path / "example")
    cmd = ["gcc", "-O2", "-std=c11", os.path.join(ROOT, "tests", "c_abi", "example.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           lib, "-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.dirname(lib),
           "-Wl,-rpath," + os.path.join(cuda, "lib64"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe, str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr

    def load(name, dtype, shape):
        return np.fromfile(tmp_path / f"{name}.bin", dtype=dtype).reshape(shape)

    x = torch.from_numpy(load("x", np.int16, (M, K))).view(torch.bfloat16).cuda()
    w = torch.from_numpy(load("w", np.int16, (N, K))).view(torch.bfloat16).cuda()
    dy = torch.from_numpy(load("dy", np.int16, (M, N))).view(torch.bfloat16).cuda()
    qx, sx, qxT, sxc = rlq.quant_act_1x128(x, colwise=True)
    qw, sw, qwT = rlq.quant_weight_128x128(w, transposed=True)
    qdy, sdy, _, _ = rlq.quant_act_1x128(dy)
    y = rlq.gemm_fprop(qx, sx, qw, sw)
    dx = rlq.gemm_dgrad(qdy, sdy, qwT, sw, transposed=True)
    rlq.check()
    np_ = lambda t: t.cpu().numpy()
    assert np.array_equal(np_(qx), load("qx", np.uint8, (M, K)))
    assert np.array_equal(np_(sx), load("sx", np.float32, (K // 128, M)))
    assert np.array_equal(np_(qxT), load("qxT", np.uint8, (K, LDM))[:, :M])
    assert np.array_equal(np_(sxc), load("sxc", np.float32, ((M + 127) // 128, K)))
    assert np.array_equal(np_(qw), load("qw", np.uint8, (N, K)))
    assert np.array_equal(np_(sw), load("sw", np.float32, (N // 128, K // 128)))
    assert np.array_equal(np_(y.view(torch.int16)), load("y", np.int16, (M, N)))
    assert np.array_equal(np_(dx.view(torch.int16)), load("dx", np.int16, (M, K)))
