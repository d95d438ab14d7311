"""CPU-side checks of the C ABI: the library builds, loads and exports every
entry point that include/rlq.h declares, and host-side validation returns the
documented status codes before anything is launched (no GPU needed)."""
import os
import re

import pytest

from fp8_block_scaled_quantize_gb300 import rlq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rlq.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rlq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ("rlq_quant_act_1x128", "rlq_quant_weight_128x128", "rlq_gemm_fprop", "rlq_gemm_dgrad",
              "rlq_gemm_wgrad", "rlq_uaq_fold", "rlq_check", "rlq_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = rlq.lib()
    for n in declared_functions():
        assert hasattr(L, n), f"librlq.so does not export {n}"
    assert rlq.rlq_version().count(".") == 2


def test_status_strings():
    for code, name in rlq.STATUS.items():
        assert rlq.rlq_status_string(code).startswith(name)
    assert "unknown" in rlq.rlq_status_string(99)


FAKE = 0x10000  # an aligned fake device address: validation never dereferences it


def _status(fn, *args):
    try:
        fn(*args)
        return 0
    except rlq.RlqError as e:
        return e.status


def test_quant_act_validation():
    q = rlq.rlq_quant_act_1x128
    assert _status(q, FAKE, 4, 100, 128, FAKE, 128, FAKE, 4, None, 0, None, 0, None) == 2  # K % 128
    assert _status(q, FAKE, -1, 128, 128, FAKE, 128, FAKE, 4, None, 0, None, 0, None) == 1
    assert _status(q, None, 4, 128, 128, FAKE, 128, FAKE, 4, None, 0, None, 0, None) == 1  # NULL x
    assert _status(q, FAKE, 4, 128, 64, FAKE, 128, FAKE, 4, None, 0, None, 0, None) == 1   # ldx < K
    assert _status(q, FAKE, 4, 128, 128, FAKE, 128, FAKE, 3, None, 0, None, 0, None) == 1  # lds < M
    assert _status(q, FAKE + 8, 4, 128, 128, FAKE, 128, FAKE, 4, None, 0, None, 0, None) == 3
    assert _status(q, FAKE, 4, 128, 132, FAKE, 128, FAKE, 4, None, 0, None, 0, None) == 3  # ldx % 8
    assert _status(q, FAKE, 4, 128, 128, FAKE, 136, FAKE, 4, None, 0, None, 0, None) == 3  # ldq % 16
    assert _status(q, FAKE, 4, 128, 128, FAKE, 128, FAKE, 4, FAKE, 16, None, 0, None) == 1  # qT without sc
    assert _status(q, FAKE, 4, 128, 128, FAKE, 128, FAKE, 4, FAKE, 8, FAKE, 128, None) == 3  # ldqT % 16
    assert "qT" in rlq.rlq_last_error()
    assert _status(q, FAKE, 40, 128, 128, FAKE, 128, FAKE, 40, FAKE, 32, FAKE, 128, None) == 1  # ldqT < M
    assert _status(q, FAKE, 4, 128, 128, FAKE, 128, FAKE, 4, FAKE, 16, FAKE, 64, None) == 1  # ldsc < K
    # empty extents are a no-op success without touching the pointers
    assert _status(q, None, 0, 128, 128, None, 128, None, 0, None, 0, None, 0, None) == 0
    assert _status(q, None, 5, 0, 0, None, 0, None, 0, None, 0, None, 0, None) == 0


def test_rmsnorm_quant_validation():
    r = rlq.rlq_rmsnorm_quant_act_1x128
    ok = (FAKE, 4, 128, 128, FAKE, 1e-6, FAKE, FAKE, 128, FAKE, 4, None, 0, None, 0, None)

    def with_(i, v):
        a = list(ok)
        a[i] = v
        return a

    assert _status(r, *with_(2, 100)) == 2            # K % 128
    assert _status(r, *with_(4, None)) == 1           # gamma NULL
    assert _status(r, *with_(4, FAKE + 8)) == 3       # gamma not 16-byte aligned
    assert _status(r, *with_(5, float("inf"))) == 1   # eps not finite
    assert _status(r, *with_(5, -1.0)) == 1           # eps negative
    assert _status(r, *with_(6, None)) == 1           # rstd NULL
    assert _status(r, *with_(6, FAKE + 2)) == 3       # rstd alignment
    assert _status(r, *with_(3, 64)) == 1             # ldh < K
    assert _status(r, *with_(11, FAKE)) == 1          # qT without sc
    assert _status(r, None, 0, 128, 128, None, 0.0, None, None, 0, None, 0, None, 0, None, 0, None) == 0


def test_weight_and_fold_validation():
    w = rlq.rlq_quant_weight_128x128
    assert _status(w, FAKE, 100, 128, 128, FAKE, 128, FAKE, 1, None, 0, None) == 2
    assert _status(w, FAKE, 128, 256, 256, FAKE, 256, FAKE, 1, None, 0, None) == 1  # lds < K/128
    assert _status(w, FAKE, 128, 128, 128, FAKE, 128, FAKE, 1, FAKE, 64, None) == 1  # ldqT < N
    f = rlq.rlq_uaq_fold
    assert _status(f, FAKE, 4, 12, 16, FAKE, None, 0, 0, None) == 2  # K % 8
    assert _status(f, FAKE, 4, 16, 16, None, None, 0, 0, None) == 1  # s NULL
    assert _status(f, FAKE, 4, 16, 16, FAKE + 4, None, 0, 0, None) == 3  # s alignment
    assert _status(f, None, 0, 16, 16, None, None, 0, 0, None) == 0


def test_gemm_validation():
    fp = rlq.rlq_gemm_fprop
    assert _status(fp, FAKE, 128, FAKE, 4, FAKE, 128, FAKE, 1, FAKE, 136, 4, 130, 128, None) == 2  # N % 128
    assert _status(fp, FAKE, 128, FAKE, 4, FAKE, 128, FAKE, 1, FAKE, 128, 4, 128, 100, None) == 2  # K % 128
    assert _status(fp, FAKE, 120, FAKE, 4, FAKE, 128, FAKE, 1, FAKE, 128, 4, 128, 128, None) == 1  # ldxq < K
    assert _status(fp, FAKE, 144, FAKE, 4, FAKE + 1, 128, FAKE, 1, FAKE, 128, 4, 128, 128, None) == 3
    assert _status(fp, FAKE, 128, FAKE, 3, FAKE, 128, FAKE, 1, FAKE, 128, 4, 128, 128, None) == 1  # ldxs < M
    assert _status(fp, None, 0, None, 0, None, 0, None, 0, None, 0, 0, 128, 128, None) == 0  # M == 0
    dg = rlq.rlq_gemm_dgrad
    assert _status(dg, FAKE, 128, FAKE, 4, FAKE, 128, 2, FAKE, 1, FAKE, 128, 4, 128, 128, None) == 1
    wg = rlq.rlq_gemm_wgrad
    # column scales of X must be 16-byte aligned rows
    assert _status(wg, FAKE, 16, FAKE, 128, FAKE, 16, FAKE + 4, 128, FAKE, 128, 4, 128, 128, None) == 3
    assert _status(wg, FAKE, 16, FAKE, 128, FAKE, 16, FAKE, 130, FAKE, 128, 4, 128, 128, None) == 3


def test_diag_validation():
    assert _status(rlq.rlq_diag_bounded_wait, 0, None) == 1
    assert _status(rlq.rlq_diag_bounded_wait, 10 ** 8, None) == 1


def test_splitk_and_static_validation():
    """Host-side checks of the split-K, workspace-query and static-scratch entry
    points, all made before any CUDA call."""
    fp = rlq.rlq_gemm_fprop_splitk
    args = (FAKE, 128, FAKE, 4, FAKE, 128, FAKE, 1, FAKE, 128, 4, 128, 128)
    assert _status(fp, *args, FAKE + 4, 1 << 20, None) == 3    # workspace not 16-byte aligned
    assert _status(fp, *args, FAKE, -1, None) == 1             # negative workspace size
    assert _status(fp, FAKE, 128, FAKE, 4, FAKE, 128, FAKE, 1, FAKE, 136, 4, 130, 128, FAKE, 0, None) == 2
    dg = rlq.rlq_gemm_dgrad_splitk
    assert _status(dg, FAKE, 128, FAKE, 4, FAKE, 128, 1, FAKE, 1, FAKE, 128, 4, 128, 128, FAKE + 8, 64, None) == 3
    wg = rlq.rlq_gemm_wgrad_splitk
    assert _status(wg, FAKE, 16, FAKE, 128, FAKE, 16, FAKE, 128, FAKE, 128, 4, 128, 128, FAKE, -8, None) == 1
    q = rlq.rlq_gemm_splitk_workspace_bytes
    assert _status(q, 7, 64, 256, 4096) == 1                   # unknown GEMM kind
    assert _status(q, rlq.GEMM_FPROP, -1, 256, 4096) == 1     # negative size
    assert _status(q, rlq.GEMM_FPROP, 64, 1 << 31, 4096) == 2  # dimension beyond 2^31
    st = rlq.rlq_gemm_fprop_splitk_static
    assert _status(st, FAKE, 128, FAKE, 4, FAKE, 128, FAKE, 1, FAKE, 128, -4, 128, 128, None) == 1
    assert _status(st, FAKE, 128, FAKE, 4, FAKE, 128, FAKE, 1, FAKE, 128, 4, 1 << 31, 128, None) == 2
    assert rlq.STATIC_SCRATCH_BYTES == 16 << 20
    header = open(HEADER).read()
    assert "#define RLQ_STATIC_SCRATCH_BYTES 16777216" in header


def test_per_row_and_per_channel_validation():
    """Per-token / per-channel entry points: host-side checks before any launch."""
    q = rlq.rlq_quant_per_row
    assert _status(q, FAKE, 4, 100, 128, FAKE, 128, FAKE, None, 0, None) == 2        # K % 128
    assert _status(q, FAKE, -1, 128, 128, FAKE, 128, FAKE, None, 0, None) == 1       # negative M
    assert _status(q, None, 4, 128, 128, FAKE, 128, FAKE, None, 0, None) == 1        # NULL x
    assert _status(q, FAKE, 4, 128, 128, FAKE, 128, None, None, 0, None) == 1        # NULL s
    assert _status(q, FAKE, 4, 128, 128, FAKE, 120, FAKE, None, 0, None) == 1        # ldq < K
    assert _status(q, FAKE, 4, 128, 128, FAKE, 128, FAKE, FAKE, 3, None) == 1        # ld_rep < M
    assert _status(q, FAKE + 2, 4, 128, 128, FAKE, 128, FAKE, None, 0, None) == 3    # x misaligned
    assert _status(q, FAKE, 0, 128, 128, None, 0, None, None, 0, None) == 0          # empty: no-op
    g = rlq.rlq_gemm_fprop_per_channel
    ok = (FAKE, 128, FAKE, 4, FAKE, 128, FAKE, 128, FAKE, 128, 4, 128, 128, None)
    assert _status(g, FAKE, 128, FAKE, 4, FAKE, 128, FAKE, 128, FAKE, 136, 4, 136, 128, None) == 2  # N % 128
    assert _status(g, FAKE, 128, FAKE, 4, FAKE, 128, FAKE + 4, 128, FAKE, 128, 4, 128, 128, None) == 3  # ws_rep
    assert _status(g, FAKE, 128, FAKE, 4, FAKE, 128, FAKE, 126, FAKE, 128, 4, 128, 128, None) == 1  # ldws < N
    assert _status(g, FAKE, 128, FAKE, 3, FAKE, 128, FAKE, 128, FAKE, 128, 4, 128, 128, None) == 1  # ldxs < M
    assert _status(g, *ok[:10], -1, *ok[11:]) == 1                                                 # negative M


def test_per_channel_splitk_validation():
    g = rlq.rlq_gemm_fprop_per_channel_splitk
    args = (FAKE, 128, FAKE, 4, FAKE, 128, FAKE, 128, FAKE, 128, 4, 128, 128)
    assert _status(g, *args, FAKE + 4, 1 << 20, None) == 3    # workspace not 16-byte aligned
    assert _status(g, *args, FAKE, -1, None) == 1             # negative workspace size


def test_aqn_validation_and_host_schedule():
    """AQN: host-side checks of the perturbation, and the host-only noise schedule
    against the oracle's."""
    import oracle
    p = rlq.rlq_aqn_perturb
    assert _status(p, FAKE, -1, FAKE, 0.1, None) == 1                 # negative K
    assert _status(p, None, 8, FAKE, 0.1, None) == 1                  # NULL gamma
    assert _status(p, FAKE + 1, 8, FAKE, 0.1, None) == 3              # gamma not 2-byte aligned
    assert _status(p, FAKE, 8, FAKE + 2, 0.1, None) == 3              # z not 4-byte aligned
    assert _status(p, FAKE, 8, FAKE, float("nan"), None) == 1         # sigma not finite
    assert _status(p, None, 0, None, 0.1, None) == 0                  # empty: no-op
    with pytest.raises(rlq.RlqError):
        rlq.rlq_aqn_sigma(1e-2, 5e-4, 10, 10)                         # t outside 0 .. T-1
    with pytest.raises(rlq.RlqError):
        rlq.rlq_aqn_sigma(0.0, 5e-4, 1, 10)                           # decaying from zero
    for s0, s1, T in ((1e-2, 5e-4, 11), (0.05, 1e-3, 100), (0.3, 0.3, 5), (0.02, 0.01, 1)):
        for t in range(T):
            a, b = rlq.rlq_aqn_sigma(s0, s1, t, T), oracle.aqn_sigma(s0, s1, t, T)
            assert abs(a - b) <= 1e-6 * b
        assert rlq.rlq_aqn_sigma(s0, s1, 0, T) == oracle.aqn_sigma(s0, s1, 0, T)
        assert rlq.rlq_aqn_sigma(s0, s1, T - 1, T) == oracle.aqn_sigma(s0, s1, T - 1, T)


def test_wgrad_accumulate_validation():
    g = rlq.rlq_gemm_wgrad_accumulate
    ok = (FAKE, 256, FAKE, 128, FAKE, 256, FAKE, 128, FAKE, 128, 256, 128, 128, FAKE, 2 * 128 * 128 * 4, None)
    assert _status(g, *ok[:13], FAKE + 8, 1 << 20, None) == 3       # workspace not 16-byte aligned
    assert _status(g, *ok[:14], -1, None) == 1                      # negative workspace size
    assert _status(g, *ok[:8], FAKE + 4, *ok[9:]) == 3              # dw_acc not 16-byte aligned
    assert _status(g, *ok[:9], 126, *ok[10:]) == 1                  # ld_acc < K
    assert _status(g, *ok[:10], 0, *ok[11:]) == 0                   # M = 0: nothing to add


def test_nvfp4_validation():
    f = rlq.rlq_quant_nvfp4
    assert _status(f, FAKE, 4, 24, 24, FAKE, 16, FAKE, 2, FAKE, None) == 2      # K % 16
    assert _status(f, FAKE, 4, 32, 32, FAKE, 16, FAKE, 2, None, None) == 1      # NULL st
    assert _status(f, FAKE, 4, 32, 32, FAKE, 12, FAKE, 2, FAKE, None) == 1      # ldq < K/2
    assert _status(f, FAKE, 4, 32, 32, FAKE + 4, 16, FAKE, 2, FAKE, None) == 3  # q rows not 8-byte aligned
    assert _status(f, FAKE, 4, 32, 32, FAKE, 16, FAKE, 1, FAKE, None) == 1      # ldsb < K/16
    assert _status(f, FAKE, 0, 32, 32, None, 0, None, 0, FAKE, None) == 0       # empty: no-op


def test_binding_covers_every_declared_function():
    """Every entry point of include/rlq.h has a ctypes signature in the binding
    (the string-returning ones are typed when the library loads)."""
    typed_at_load = {"rlq_status_string", "rlq_last_error", "rlq_version"}
    missing = [n for n in declared_functions() if n not in rlq._SIGS and n not in typed_at_load]
    assert not missing, f"no ctypes signature for {missing}"


def test_nvfp4_gemm_validation():
    """Host checks of the NVFP4 weight-only GEMM and its split-K form (no launch)."""
    g, gs = rlq.rlq_gemm_nvfp4_weight_only, rlq.rlq_gemm_nvfp4_weight_only_splitk
    # x [4, 128] bf16, wq [128, 64] bytes (pitch 64), wsb [128, 8] (pitch 16), y [4, 128]
    ok = (FAKE, 128, FAKE, 64, FAKE, 16, FAKE, FAKE, 128, 4, 128, 128)
    assert _status(g, *ok[:10], 100, 128, None) == 2                         # N % 128
    assert _status(g, *ok[:11], 96, None) == 2                               # K % 64
    assert _status(g, *ok[:3], 72, *ok[4:], None) == 3                       # code pitch not a multiple of 16
    assert _status(g, *ok[:6], None, *ok[7:], None) == 1                     # NULL tensor scale
    assert _status(g, *ok[:6], FAKE + 2, *ok[7:], None) == 3                 # tensor scale not 4-byte aligned
    assert _status(g, *ok[:9], 0, 128, 128, None) == 0                       # M = 0: nothing to do
    assert _status(gs, *ok, FAKE + 8, 1 << 20, None) == 3                    # workspace not 16-byte aligned
    assert _status(gs, *ok, FAKE, -1, None) == 1                             # negative workspace size
    assert _status(gs, *ok[:10], 100, 128, FAKE, 1 << 20, None) == 2         # N % 128, with a workspace
