"""Thin ctypes binding of librlq.so (include/rlq.h).

The functions named ``rlq_*`` mirror the C entry points one to one: plain
integers for device pointers, sizes and the stream, and an ``RlqError`` raised
for a non-OK status.  The lower-case helpers below them take torch tensors,
allocate outputs with torch (device memory is PyTorch's plumbing here) and call
the same entry points; every step of the computation runs in the library's
CUDA kernels.  There is no fallback: if the library is missing or cannot be
loaded, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

GRP = 128

_P = ctypes.c_void_p
_I = ctypes.c_int64

_SIGS = {
    "rlq_quant_act_1x128": [_P, _I, _I, _I, _P, _I, _P, _I, _P, _I, _P, _I, _P],
    "rlq_quant_weight_128x128": [_P, _I, _I, _I, _P, _I, _P, _I, _P, _I, _P],
    "rlq_rmsnorm_quant_act_1x128": [_P, _I, _I, _I, _P, ctypes.c_float, _P, _P, _I, _P, _I, _P, _I, _P, _I, _P],
    "rlq_gemm_fprop": [_P, _I, _P, _I, _P, _I, _P, _I, _P, _I, _I, _I, _I, _P],
    "rlq_gemm_dgrad": [_P, _I, _P, _I, _P, _I, ctypes.c_int, _P, _I, _P, _I, _I, _I, _I, _P],
    "rlq_gemm_wgrad": [_P, _I, _P, _I, _P, _I, _P, _I, _P, _I, _I, _I, _I, _P],
    "rlq_gemm_splitk_workspace_bytes": [ctypes.c_int, _I, _I, _I, ctypes.POINTER(_I)],
    "rlq_gemm_fprop_splitk": [_P, _I, _P, _I, _P, _I, _P, _I, _P, _I, _I, _I, _I, _P, _I, _P],
    "rlq_gemm_dgrad_splitk": [_P, _I, _P, _I, _P, _I, ctypes.c_int, _P, _I, _P, _I, _I, _I, _I, _P, _I, _P],
    "rlq_gemm_wgrad_splitk": [_P, _I, _P, _I, _P, _I, _P, _I, _P, _I, _I, _I, _I, _P, _I, _P],
    "rlq_gemm_fprop_splitk_static": [_P, _I, _P, _I, _P, _I, _P, _I, _P, _I, _I, _I, _I, _P],
    "rlq_quant_per_row": [_P, _I, _I, _I, _P, _I, _P, _P, _I, _P],
    "rlq_gemm_fprop_per_channel": [_P, _I, _P, _I, _P, _I, _P, _I, _P, _I, _I, _I, _I, _P],
    "rlq_gemm_fprop_per_channel_splitk": [_P, _I, _P, _I, _P, _I, _P, _I, _P, _I, _I, _I, _I, _P, _I, _P],
    "rlq_uaq_fold": [_P, _I, _I, _I, _P, _P, _I, _I, _P],
    "rlq_gemm_wgrad_accumulate": [_P, _I, _P, _I, _P, _I, _P, _I, _P, _I, _I, _I, _I, _P, _I, _P],
    "rlq_quant_nvfp4": [_P, _I, _I, _I, _P, _I, _P, _I, _P, _P],
    "rlq_gemm_nvfp4_weight_only": [_P, _I, _P, _I, _P, _I, _P, _P, _I, _I, _I, _I, _P],
    "rlq_gemm_nvfp4_weight_only_splitk": [_P, _I, _P, _I, _P, _I, _P, _P, _I, _I, _I, _I, _P, _I, _P],
    "rlq_aqn_sigma": [ctypes.c_float, ctypes.c_float, _I, _I, ctypes.POINTER(ctypes.c_float)],
    "rlq_aqn_perturb": [_P, _I, _P, ctypes.c_float, _P],
    "rlq_check": [_P],
    "rlq_diag_bounded_wait": [_I, _P],
    "rlq_diag_arm_gemm_stall": [],
}

STATUS = {0: "RLQ_OK", 1: "RLQ_ERR_INVALID_ARG", 2: "RLQ_ERR_UNSUPPORTED", 3: "RLQ_ERR_MISALIGNED",
          4: "RLQ_ERR_CUDA", 5: "RLQ_ERR_TIMEOUT"}


class RlqError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load librlq.so (building it first if its sources are newer)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path) or _build._stale():
                _build.build()
            L = ctypes.CDLL(path)
            for name, args in _SIGS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            L.rlq_status_string.argtypes = [ctypes.c_int]
            L.rlq_status_string.restype = ctypes.c_char_p
            L.rlq_last_error.argtypes = []
            L.rlq_last_error.restype = ctypes.c_char_p
            L.rlq_version.argtypes = []
            L.rlq_version.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _call(name: str, *args) -> int:
    L = lib()
    st = getattr(L, name)(*args)
    if st != 0:
        raise RlqError(st, L.rlq_last_error().decode(errors="replace"))
    return st


# ------------------------------------------------- raw C-ABI mirrors ---

def rlq_quant_act_1x128(x, M, K, ldx, q, ldq, s, lds, qT, ldqT, sc, ldsc, stream):
    return _call("rlq_quant_act_1x128", x, M, K, ldx, q, ldq, s, lds, qT, ldqT, sc, ldsc, stream)


def rlq_rmsnorm_quant_act_1x128(h, M, K, ldh, gamma, eps, rstd, q, ldq, s, lds, qT, ldqT, sc, ldsc, stream):
    return _call("rlq_rmsnorm_quant_act_1x128", h, M, K, ldh, gamma, eps, rstd, q, ldq, s, lds, qT, ldqT, sc, ldsc,
                 stream)


def rlq_quant_weight_128x128(w, N, K, ldw, q, ldq, s, lds, qT, ldqT, stream):
    return _call("rlq_quant_weight_128x128", w, N, K, ldw, q, ldq, s, lds, qT, ldqT, stream)


def rlq_gemm_fprop(xq, ldxq, xs, ldxs, wq, ldwq, ws, ldws, y, ldy, M, N, K, stream):
    return _call("rlq_gemm_fprop", xq, ldxq, xs, ldxs, wq, ldwq, ws, ldws, y, ldy, M, N, K, stream)


def rlq_gemm_dgrad(dyq, lddyq, dys, lddys, w, ldw, wq_is_transposed, ws, ldws, dx, lddx, M, N, K, stream):
    return _call("rlq_gemm_dgrad", dyq, lddyq, dys, lddys, w, ldw, wq_is_transposed, ws, ldws, dx, lddx,
                 M, N, K, stream)


def rlq_gemm_wgrad(dyqT, lddyqT, dysc, lddysc, xqT, ldxqT, xsc, ldxsc, dw, lddw, M, N, K, stream):
    return _call("rlq_gemm_wgrad", dyqT, lddyqT, dysc, lddysc, xqT, ldxqT, xsc, ldxsc, dw, lddw, M, N, K, stream)


GEMM_FPROP, GEMM_DGRAD, GEMM_WGRAD, GEMM_NVFP4_WEIGHT_ONLY = 0, 1, 2, 3


def rlq_gemm_splitk_workspace_bytes(kind, M, N, K) -> int:
    out = _I(0)
    _call("rlq_gemm_splitk_workspace_bytes", kind, M, N, K, ctypes.byref(out))
    return out.value


def rlq_gemm_fprop_splitk(xq, ldxq, xs, ldxs, wq, ldwq, ws, ldws, y, ldy, M, N, K, workspace, workspace_bytes,
                          stream):
    return _call("rlq_gemm_fprop_splitk", xq, ldxq, xs, ldxs, wq, ldwq, ws, ldws, y, ldy, M, N, K, workspace,
                 workspace_bytes, stream)


def rlq_gemm_dgrad_splitk(dyq, lddyq, dys, lddys, w, ldw, wq_is_transposed, ws, ldws, dx, lddx, M, N, K, workspace,
                          workspace_bytes, stream):
    return _call("rlq_gemm_dgrad_splitk", dyq, lddyq, dys, lddys, w, ldw, wq_is_transposed, ws, ldws, dx, lddx,
                 M, N, K, workspace, workspace_bytes, stream)


def rlq_gemm_wgrad_splitk(dyqT, lddyqT, dysc, lddysc, xqT, ldxqT, xsc, ldxsc, dw, lddw, M, N, K, workspace,
                          workspace_bytes, stream):
    return _call("rlq_gemm_wgrad_splitk", dyqT, lddyqT, dysc, lddysc, xqT, ldxqT, xsc, ldxsc, dw, lddw, M, N, K,
                 workspace, workspace_bytes, stream)


# Size of the library's static split-K scratch (RLQ_STATIC_SCRATCH_BYTES in rlq.h).
STATIC_SCRATCH_BYTES = 16 << 20


def rlq_gemm_fprop_splitk_static(xq, ldxq, xs, ldxs, wq, ldwq, ws, ldws, y, ldy, M, N, K, stream):
    """Split-K FProp on the library's static scratch, for callers that cannot
    allocate device memory (see rlq.h); the plan must fit STATIC_SCRATCH_BYTES."""
    return _call("rlq_gemm_fprop_splitk_static", xq, ldxq, xs, ldxs, wq, ldwq, ws, ldws, y, ldy, M, N, K, stream)


def rlq_quant_per_row(x, M, K, ldx, q, ldq, s, s_rep, ld_rep, stream):
    return _call("rlq_quant_per_row", x, M, K, ldx, q, ldq, s, s_rep, ld_rep, stream)


def rlq_gemm_fprop_per_channel(xq, ldxq, xs_rep, ldxs, wq, ldwq, ws_rep, ldws, y, ldy, M, N, K, stream):
    return _call("rlq_gemm_fprop_per_channel", xq, ldxq, xs_rep, ldxs, wq, ldwq, ws_rep, ldws, y, ldy, M, N, K,
                 stream)


def rlq_gemm_fprop_per_channel_splitk(xq, ldxq, xs_rep, ldxs, wq, ldwq, ws_rep, ldws, y, ldy, M, N, K, workspace,
                                      workspace_bytes, stream):
    return _call("rlq_gemm_fprop_per_channel_splitk", xq, ldxq, xs_rep, ldxs, wq, ldwq, ws_rep, ldws, y, ldy, M, N,
                 K, workspace, workspace_bytes, stream)


def rlq_gemm_wgrad_accumulate(dyqT, lddyqT, dysc, lddysc, xqT, ldxqT, xsc, ldxsc, dw_acc, ld_acc, M, N, K,
                              workspace, workspace_bytes, stream):
    return _call("rlq_gemm_wgrad_accumulate", dyqT, lddyqT, dysc, lddysc, xqT, ldxqT, xsc, ldxsc, dw_acc, ld_acc,
                 M, N, K, workspace, workspace_bytes, stream)


def rlq_quant_nvfp4(w, N, K, ldw, q, ldq, sb, ldsb, st, stream):
    return _call("rlq_quant_nvfp4", w, N, K, ldw, q, ldq, sb, ldsb, st, stream)


def rlq_gemm_nvfp4_weight_only(x, ldx, wq, ldwq, wsb, ldwsb, wst, y, ldy, M, N, K, stream):
    return _call("rlq_gemm_nvfp4_weight_only", x, ldx, wq, ldwq, wsb, ldwsb, wst, y, ldy, M, N, K, stream)


def rlq_gemm_nvfp4_weight_only_splitk(x, ldx, wq, ldwq, wsb, ldwsb, wst, y, ldy, M, N, K, workspace,
                                      workspace_bytes, stream):
    return _call("rlq_gemm_nvfp4_weight_only_splitk", x, ldx, wq, ldwq, wsb, ldwsb, wst, y, ldy, M, N, K, workspace,
                 workspace_bytes, stream)


def rlq_aqn_sigma(sigma_start, sigma_end, t, T) -> float:
    out = ctypes.c_float()
    _call("rlq_aqn_sigma", sigma_start, sigma_end, t, T, ctypes.byref(out))
    return out.value


def rlq_aqn_perturb(gamma, K, z, sigma, stream):
    return _call("rlq_aqn_perturb", gamma, K, z, sigma, stream)


def rlq_uaq_fold(w, N, K, ldw, s, prev, R, ldp, stream):
    return _call("rlq_uaq_fold", w, N, K, ldw, s, prev, R, ldp, stream)


def rlq_check(stream):
    return _call("rlq_check", stream)


def rlq_diag_bounded_wait(timeout_us, stream):
    return _call("rlq_diag_bounded_wait", timeout_us, stream)


def rlq_diag_arm_gemm_stall():
    return _call("rlq_diag_arm_gemm_stall")


def rlq_status_string(status: int) -> str:
    return lib().rlq_status_string(status).decode()


def rlq_last_error() -> str:
    return lib().rlq_last_error().decode(errors="replace")


def rlq_version() -> str:
    return lib().rlq_version().decode()


# ------------------------------------------------------ torch helpers ---

def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _ld(t) -> int:
    """Row pitch in elements of a 2-D tensor whose rows are contiguous."""
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with contiguous rows")
    return t.stride(0)


def _round_up(v: int, m: int) -> int:
    return (v + m - 1) // m * m


def empty_codes_T(K: int, M: int, device) -> torch.Tensor:
    """[K, M] uint8 view of a [K, round_up(M, 16)] buffer (TMA-ready pitch)."""
    return torch.empty((K, _round_up(max(M, 1), 16)), dtype=torch.uint8, device=device)[:, :M]


def quant_act_1x128(x: torch.Tensor, colwise: bool = False, stream=None):
    """1x128 quantization of bf16 x [M, K]; with ``colwise`` also the fused
    128x1 codes (transposed) and scales.

    Returns (q [M,K] u8, s [K/128, M] f32, qT [K, M] u8 or None, sc [ceil(M/128), K] f32 or None).
    """
    if x.dtype != torch.bfloat16:
        raise TypeError("x must be bfloat16")
    M, K = x.shape
    dev = x.device
    q = torch.empty((M, K), dtype=torch.uint8, device=dev)
    s = torch.empty((K // GRP, M), dtype=torch.float32, device=dev)
    qT = sc = None
    if colwise:
        qT = empty_codes_T(K, M, dev)
        sc = torch.empty(((M + GRP - 1) // GRP, K), dtype=torch.float32, device=dev)
    rlq_quant_act_1x128(x.data_ptr(), M, K, _ld(x), q.data_ptr(), K, s.data_ptr(), max(M, 1),
                        _ptr(qT), _ld(qT) if qT is not None else 0, _ptr(sc), K if sc is not None else 0,
                        _stream(stream))
    return q, s, qT, sc


def rmsnorm_quant_act_1x128(h: torch.Tensor, gamma: torch.Tensor, eps: float, colwise: bool = False, stream=None):
    """RMSNorm of the bf16 hidden state h [M, K] with the (UAQ-folded) bf16 norm
    weight gamma [K], quantized 1x128 (and with ``colwise`` 128x1) without
    writing the normalised activation.

    Returns (q, s, qT, sc) as ``quant_act_1x128`` and rstd [M] f32."""
    if h.dtype != torch.bfloat16 or gamma.dtype != torch.bfloat16:
        raise TypeError("h and gamma must be bfloat16")
    M, K = h.shape
    if gamma.shape != (K,) or not gamma.is_contiguous():
        raise ValueError("gamma must be a contiguous [K] tensor")
    dev = h.device
    q = torch.empty((M, K), dtype=torch.uint8, device=dev)
    s = torch.empty((K // GRP, M), dtype=torch.float32, device=dev)
    rstd = torch.empty((max(M, 1),), dtype=torch.float32, device=dev)[:M]
    qT = sc = None
    if colwise:
        qT = empty_codes_T(K, M, dev)
        sc = torch.empty(((M + GRP - 1) // GRP, K), dtype=torch.float32, device=dev)
    rlq_rmsnorm_quant_act_1x128(h.data_ptr(), M, K, _ld(h), gamma.data_ptr(), eps, rstd.data_ptr(), q.data_ptr(), K,
                                s.data_ptr(), max(M, 1), _ptr(qT), _ld(qT) if qT is not None else 0, _ptr(sc),
                                K if sc is not None else 0, _stream(stream))
    return q, s, qT, sc, rstd


def quant_weight_128x128(w: torch.Tensor, transposed: bool = False, stream=None):
    """128x128 block quantization of bf16 w [N, K].

    Returns (q [N,K] u8, s [N/128, K/128] f32, qT [K,N] u8 or None).
    """
    if w.dtype != torch.bfloat16:
        raise TypeError("w must be bfloat16")
    N, K = w.shape
    dev = w.device
    q = torch.empty((N, K), dtype=torch.uint8, device=dev)
    s = torch.empty((N // GRP, K // GRP), dtype=torch.float32, device=dev)
    qT = torch.empty((K, N), dtype=torch.uint8, device=dev) if transposed else None
    rlq_quant_weight_128x128(w.data_ptr(), N, K, _ld(w), q.data_ptr(), K, s.data_ptr(), max(K // GRP, 1),
                             _ptr(qT), N if qT is not None else 0, _stream(stream))
    return q, s, qT


def quant_per_row(x: torch.Tensor, replicate: bool = True, stream=None):
    """Per-row FP8 quantization of bf16 x [M, K] (per-token activations, or
    per-channel weights with x = W).

    Returns (q [M,K] u8, s [M] f32, s_rep [K/128, M] f32 or None): s_rep holds
    each row's scale once per K-block, the layout ``gemm_fprop_per_channel`` reads.
    """
    if x.dtype != torch.bfloat16:
        raise TypeError("x must be bfloat16")
    M, K = x.shape
    dev = x.device
    q = torch.empty((M, K), dtype=torch.uint8, device=dev)
    s = torch.empty((max(M, 1),), dtype=torch.float32, device=dev)[:M]
    Mp = _round_up(max(M, 1), 4)
    s_rep = torch.empty((K // GRP, Mp), dtype=torch.float32, device=dev)[:, :M] if replicate else None
    rlq_quant_per_row(x.data_ptr(), M, K, _ld(x), q.data_ptr(), K, s.data_ptr(), _ptr(s_rep),
                      Mp if replicate else 0, _stream(stream))
    return q, s, s_rep


def gemm_fprop_per_channel(xq, xs_rep, wq, ws_rep, out=None, stream=None, split_k: bool = False, workspace=None):
    """Y [M, N] bf16 = diag(sx) Qx Qw^T diag(sw) from per-token X codes and
    per-channel W codes, with the scales in the replicated [K/128, rows] layout.
    ``split_k`` as in ``gemm_fprop`` (the FProp plan)."""
    M, K = xq.shape
    N = wq.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    args = (xq.data_ptr(), _ld(xq), xs_rep.data_ptr(), _ld(xs_rep), wq.data_ptr(), _ld(wq), ws_rep.data_ptr(),
            _ld(ws_rep), y.data_ptr(), _ld(y), M, N, K)
    if split_k:
        rlq_gemm_fprop_per_channel_splitk(*args, *_workspace(GEMM_FPROP, M, N, K, workspace, xq.device),
                                          _stream(stream))
    else:
        rlq_gemm_fprop_per_channel(*args, _stream(stream))
    return y


def _workspace(kind: int, M: int, N: int, K: int, workspace, device):
    """(pointer, bytes) of the split-K workspace: the caller's uint8 tensor, or
    one allocated with torch for the library's plan (None when it is one pass)."""
    if workspace is None:
        nbytes = rlq_gemm_splitk_workspace_bytes(kind, M, N, K)
        if nbytes == 0:
            return None, 0
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def gemm_fprop(xq, xs, wq, ws, out=None, stream=None, split_k: bool = False, workspace=None):
    """Y [M, N] bf16 = X W^T from 1x128 X codes and 128x128 W codes.

    ``split_k`` runs the split-K form with ``workspace`` (a device tensor) or
    a workspace allocated here for the library's plan."""
    M, K = xq.shape
    N = wq.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    args = (xq.data_ptr(), _ld(xq), xs.data_ptr(), _ld(xs), wq.data_ptr(), _ld(wq), ws.data_ptr(), _ld(ws),
            y.data_ptr(), _ld(y), M, N, K)
    if split_k:
        rlq_gemm_fprop_splitk(*args, *_workspace(GEMM_FPROP, M, N, K, workspace, xq.device), _stream(stream))
    else:
        rlq_gemm_fprop(*args, _stream(stream))
    return y


def gemm_dgrad(dyq, dys, w, ws, transposed: bool = True, out=None, stream=None, split_k: bool = False,
               workspace=None):
    """dX [M, K] bf16 = dY W.  ``w`` is the transposed weight codes [K, N]
    (``transposed=True``) or the FProp codes [N, K]."""
    M, N = dyq.shape
    K = w.shape[0] if transposed else w.shape[1]
    dx = out if out is not None else torch.empty((M, K), dtype=torch.bfloat16, device=dyq.device)
    args = (dyq.data_ptr(), _ld(dyq), dys.data_ptr(), _ld(dys), w.data_ptr(), _ld(w), 1 if transposed else 0,
            ws.data_ptr(), _ld(ws), dx.data_ptr(), _ld(dx), M, N, K)
    if split_k:
        rlq_gemm_dgrad_splitk(*args, *_workspace(GEMM_DGRAD, M, N, K, workspace, dyq.device), _stream(stream))
    else:
        rlq_gemm_dgrad(*args, _stream(stream))
    return dx


def gemm_wgrad(dyqT, dysc, xqT, xsc, out=None, stream=None, split_k: bool = False, workspace=None):
    """dW [N, K] bf16 = dY^T X from the 128x1 (transposed) codes of dY and X."""
    N, M = dyqT.shape
    K = xqT.shape[0]
    dw = out if out is not None else torch.empty((N, K), dtype=torch.bfloat16, device=dyqT.device)
    args = (dyqT.data_ptr(), _ld(dyqT), dysc.data_ptr(), _ld(dysc), xqT.data_ptr(), _ld(xqT),
            xsc.data_ptr(), _ld(xsc), dw.data_ptr(), _ld(dw), M, N, K)
    if split_k:
        rlq_gemm_wgrad_splitk(*args, *_workspace(GEMM_WGRAD, M, N, K, workspace, dyqT.device), _stream(stream))
    else:
        rlq_gemm_wgrad(*args, _stream(stream))
    return dw


def gemm_wgrad_accumulate_(dw_acc: torch.Tensor, dyqT, dysc, xqT, xsc, workspace=None, stream=None):
    """dw_acc [N, K] fp32 += dY^T X (the WGrad product, kept in fp32).  The
    workspace (uint8 device tensor) defaults to the library's split-K plan (none
    when the plan is one pass: the GEMM's epilogue then adds into dw_acc)."""
    if dw_acc.dtype != torch.float32:
        raise TypeError("dw_acc must be float32")
    N, M = dyqT.shape
    K = xqT.shape[0]
    ptr, nbytes = _workspace(GEMM_WGRAD, M, N, K, workspace, dw_acc.device)
    rlq_gemm_wgrad_accumulate(dyqT.data_ptr(), _ld(dyqT), dysc.data_ptr(), _ld(dysc), xqT.data_ptr(), _ld(xqT),
                              xsc.data_ptr(), _ld(xsc), dw_acc.data_ptr(), _ld(dw_acc), M, N, K, ptr, nbytes,
                              _stream(stream))
    return dw_acc


def uaq_fold_(w: torch.Tensor, s: torch.Tensor, prev: torch.Tensor | None = None, stream=None):
    """In-place UAQ fold: w[:, k] /= s[k], prev[:, k] *= s[k] (bf16, fp32 math)."""
    N, K = w.shape
    R = prev.shape[0] if prev is not None else 0
    rlq_uaq_fold(w.data_ptr(), N, K, _ld(w), s.data_ptr(), _ptr(prev), R, _ld(prev) if prev is not None else 0,
                 _stream(stream))
    return w, prev


def quant_nvfp4(w: torch.Tensor, stream=None):
    """NVFP4 quantization of bf16 w [N, K] (K % 16 == 0).

    Returns (q [N, K/2] u8 packed E2M1 codes, low nibble first; sb [N, K/16] u8
    E4M3 block-scale codes; st [1] f32 tensor scale)."""
    if w.dtype != torch.bfloat16:
        raise TypeError("w must be bfloat16")
    N, K = w.shape
    dev = w.device
    # pitches rounded to 16 bytes: the layout gemm_nvfp4_weight_only reads by TMA
    kq = _round_up(max(K // 2, 1), 16)
    ks = _round_up(max(K // 16, 1), 16)
    q = torch.empty((N, kq), dtype=torch.uint8, device=dev)[:, :K // 2]
    sb = torch.empty((N, ks), dtype=torch.uint8, device=dev)[:, :K // 16]
    st = torch.empty((1,), dtype=torch.float32, device=dev)
    rlq_quant_nvfp4(w.data_ptr(), N, K, _ld(w), q.data_ptr(), kq, sb.data_ptr(), ks, st.data_ptr(), _stream(stream))
    return q, sb, st


def gemm_nvfp4_weight_only(x: torch.Tensor, q, sb, st, out=None, stream=None, split_k: bool = False,
                           workspace=None):
    """Y [M, N] bf16 = X W^T with bf16 X [M, K] and NVFP4 weights (the outputs of
    ``quant_nvfp4``: q [N, K/2] packed E2M1, sb [N, K/16] E4M3, st [1] f32).

    ``split_k`` runs the split-K form with ``workspace`` (a uint8 device tensor)
    or a workspace allocated here for the library's plan."""
    if x.dtype != torch.bfloat16:
        raise TypeError("x must be bfloat16")
    M, K = x.shape
    N = q.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    args = (x.data_ptr(), _ld(x), q.data_ptr(), q.stride(0), sb.data_ptr(), sb.stride(0), st.data_ptr(),
            y.data_ptr(), _ld(y), M, N, K)
    if split_k:
        rlq_gemm_nvfp4_weight_only_splitk(*args, *_workspace(GEMM_NVFP4_WEIGHT_ONLY, M, N, K, workspace, x.device),
                                          _stream(stream))
    else:
        rlq_gemm_nvfp4_weight_only(*args, _stream(stream))
    return y


def aqn_perturb_(gamma: torch.Tensor, z: torch.Tensor, sigma: float, stream=None):
    """In-place AQN: gamma[k] = bf16(gamma[k] + sigma * z[k]) for a bf16 norm scale
    gamma [K] and one standard-normal draw per channel z [K] (f32)."""
    if gamma.dtype != torch.bfloat16 or z.dtype != torch.float32 or gamma.dim() != 1 or z.shape != gamma.shape:
        raise TypeError("gamma must be 1-D bfloat16 and z float32 of the same length")
    if not (gamma.is_contiguous() and z.is_contiguous()):
        raise ValueError("gamma and z must be contiguous")
    rlq_aqn_perturb(gamma.data_ptr(), gamma.numel(), z.data_ptr(), sigma, _stream(stream))
    return gamma


def check(stream=None):
    """Synchronise the stream and raise RlqError on a recorded device-side timeout."""
    return rlq_check(_stream(stream))
