"""Oracle for the quantized actor linear layer — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
path (``fp8_block_scaled_quantize_gb300``) never imports it, shares no code,
header, table or helper with it, and fails loudly when its CUDA library is
missing instead of falling back here.

Contents
--------
* ``rlq_oracle.c`` (plain C, built on first use with gcc): E4M3 encode/decode,
  the 1x128 / 128x1 / 128x128 group quantizers, the per-row (per-token /
  per-channel) quantizer, the UAQ fold, the RMSNorm whose weight carries the
  folded UAQ scale, the AQN perturbation and the NVFP4
  weight quantizer (E2M1 codes, E4M3 block scales, fp32 tensor scale).  These are bit-level definitions;
  the GPU must reproduce their bytes exactly.
* This module: a ctypes binding for the C part and the fp64 GEMMs over
  dequantized operands (NumPy): the block-scaled FProp, DGrad and WGrad, and
  the per-token x per-channel FProp.

Sources (the web pages on quantized RL rollout):
* Jet-RL notes, section "细粒度 GEMM 量化方案" (Fig. 6): 128x128 per-block
  weight quantization; 1x128 per-group activation / gradient quantization;
  FProp takes 1x128 activations and 128x128 weights; DGrad takes FProp's
  configuration; WGrad takes a 1x128 first operand and a 128x1 second operand.
* QuRL notes, section 关键设计 §1 (UAQ): WX = (W/s)(sX), s applied per column
  of W and per row of the previous activation.
* QeRL news article: adaptive quantization noise (AQN), channel-wise Gaussian
  noise mapped into the LayerNorm scale, decaying on an exponential schedule.
* QuRL notes, section "损失函数 / 训练策略": channel-wise weight and token-wise
  activation quantization (INT8 or FP8; the FP8 form here): one group per row
  over all K columns, the scales factored out of the GEMM's sum.
* The FP8 sub-format (E4M3, max 448), the scale rule (amax/448, 1.0 for an
  all-zero group), RN-satfinite rounding and fp32 IEEE division are the
  plainest readings of what the pages leave open.

Pins: ``tests/test_oracle_*.py`` check every function here against the OCP
E4M3 definition, an independent library (torch / ml_dtypes float8), exact
rational arithmetic, exhaustive enumeration and closed-form bounds.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rlq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

GRP = 128

_lib = None
_lock = threading.Lock()

_P = ctypes.c_void_p
_I = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile ``rlq_oracle.c`` into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_encode.argtypes = [ctypes.c_float]
            L.orc_group_scale.restype = ctypes.c_float
            L.orc_group_scale.argtypes = [ctypes.c_float]
            L.orc_quant_element.restype = ctypes.c_uint8
            L.orc_quant_element.argtypes = [ctypes.c_float, ctypes.c_float]
            L.orc_f32_to_bf16_rn.restype = ctypes.c_uint16
            L.orc_f32_to_bf16_rn.argtypes = [ctypes.c_float]
            L.orc_quant_rows_1x128.argtypes = [_P, _I, _I, _I, _P, _I, _P, _I]
            L.orc_quant_cols_128x1.argtypes = [_P, _I, _I, _I, _P, _I, _P, _I]
            L.orc_quant_weight_128x128.argtypes = [_P, _I, _I, _I, _P, _I, _P, _I, _P, _I]
            L.orc_quant_per_row.argtypes = [_P, _I, _I, _I, _P, _I, _P]
            L.orc_e2m1_decode.restype = ctypes.c_double
            L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
            L.orc_e2m1_encode.restype = ctypes.c_uint8
            L.orc_e2m1_encode.argtypes = [ctypes.c_float]
            L.orc_quant_nvfp4.argtypes = [_P, _I, _I, _I, _P, _I, _P, _I, _P]
            L.orc_aqn_sigma.restype = ctypes.c_float
            L.orc_aqn_sigma.argtypes = [ctypes.c_float, ctypes.c_float, _I, _I]
            L.orc_aqn_perturb.argtypes = [_P, _I, _P, ctypes.c_float]
            L.orc_uaq_fold.argtypes = [_P, _I, _I, _I, _P, _P, _I, _I]
            L.orc_rmsnorm.argtypes = [_P, _I, _I, _I, _P, ctypes.c_float, _P, _I, _P]
            L.orc_e4m3_encode_array.argtypes = [_P, _I, _P]
            L.orc_e4m3_decode_array.argtypes = [_P, _I, _P]
            L.orc_f32_to_bf16_array.argtypes = [_P, _I, _P]
            L.orc_quant_element_array.argtypes = [_P, _P, _I, _P]
            L.orc_num_threads.restype = ctypes.c_int
            L.orc_set_num_threads.argtypes = [ctypes.c_int]
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def num_threads() -> int:
    """OpenMP threads the C oracle runs on."""
    return int(lib().orc_num_threads())


def set_num_threads(n: int) -> None:
    """OpenMP threads for the C oracle's later calls (for timing it on fewer cores)."""
    lib().orc_set_num_threads(int(n))


# ------------------------------------------------------------------ E4M3 ---

def e4m3_decode(codes) -> np.ndarray:
    """fp64 value of each E4M3 code (NaN for 0x7F / 0xFF)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().orc_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_encode(values) -> np.ndarray:
    """RN-even, satfinite fp32 -> E4M3 code of each value."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def f32_to_bf16(values) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16_array(_ptr(v), v.size, _ptr(out))
    return out


def bf16_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 values (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def group_scale(amax: float) -> float:
    return float(lib().orc_group_scale(amax))


def quant_element(x, s) -> np.ndarray:
    """encode(fl32(x / s)) element-wise for arrays x, s (fp32)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    s = np.ascontiguousarray(np.broadcast_to(np.asarray(s, np.float32), x.shape))
    out = np.empty(x.shape, dtype=np.uint8)
    lib().orc_quant_element_array(_ptr(x), _ptr(s), x.size, _ptr(out))
    return out


_LUT = None


def e4m3_lut() -> np.ndarray:
    """fp64 value of all 256 codes (index = code)."""
    global _LUT
    if _LUT is None:
        _LUT = e4m3_decode(np.arange(256, dtype=np.uint8))
    return _LUT


def dequant_codes(codes) -> np.ndarray:
    return e4m3_lut()[np.asarray(codes, dtype=np.uint8)]


# ------------------------------------------------------------ quantizers ---

def _bf16_2d(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype != np.uint16 or x.ndim != 2:
        raise TypeError("expected a 2-D uint16 array of bf16 bit patterns")
    return np.ascontiguousarray(x)


def quant_rows_1x128(x):
    """1x128 groups along K.  x: bf16 bits [M,K], K % 128 == 0.

    Returns (q u8 [M,K], s f32 [K/128, M]); s[kb, m] is the dequant multiplier
    of row m's K-block kb.
    """
    x = _bf16_2d(x)
    M, K = x.shape
    if K % GRP:
        raise ValueError("K must be a multiple of 128")
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // GRP, M), np.float32)
    lib().orc_quant_rows_1x128(_ptr(x), M, K, K, _ptr(q), K, _ptr(s), M)
    return q, s


def quant_cols_128x1(x):
    """128x1 groups along M (tokens), codes transposed.  x: bf16 bits [M,K].

    Returns (qT u8 [K, M], sc f32 [ceil(M/128), K]).
    """
    x = _bf16_2d(x)
    M, K = x.shape
    MB = (M + GRP - 1) // GRP
    qT = np.empty((K, M), np.uint8)
    sc = np.empty((MB, K), np.float32)
    lib().orc_quant_cols_128x1(_ptr(x), M, K, K, _ptr(qT), M, _ptr(sc), K)
    return qT, sc


def quant_weight_128x128(w, transposed: bool = False):
    """128x128 blocks.  w: bf16 bits [N,K], N, K % 128 == 0.

    Returns (q u8 [N,K], s f32 [N/128, K/128], qT u8 [K,N] or None).
    """
    w = _bf16_2d(w)
    N, K = w.shape
    if N % GRP or K % GRP:
        raise ValueError("N and K must be multiples of 128")
    q = np.empty((N, K), np.uint8)
    s = np.empty((N // GRP, K // GRP), np.float32)
    qT = np.empty((K, N), np.uint8) if transposed else None
    lib().orc_quant_weight_128x128(_ptr(w), N, K, K, _ptr(q), K, _ptr(s), K // GRP,
                                   _ptr(qT) if qT is not None else None, N)
    return q, s, qT


def quant_per_row(x):
    """One group per row over all K columns: per-token activations (rows of X)
    or per-channel weights (rows of W, one per output channel).  QuRL notes,
    "损失函数 / 训练策略" (channel-wise weights, token-wise activations).

    x: bf16 bits [M,K] (any K >= 1).  Returns (q u8 [M,K], s f32 [M]).
    """
    x = _bf16_2d(x)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty((M,), np.float32)
    lib().orc_quant_per_row(_ptr(x), M, K, K, _ptr(q), K, _ptr(s))
    return q, s


def uaq_fold(w, s, prev=None):
    """UAQ fold on copies: returns (W / s per column, prev * s per column).

    w: bf16 bits [N,K]; s: f32 [K] (> 0, finite); prev: bf16 bits [R,K] or None.
    """
    w = _bf16_2d(w).copy()
    N, K = w.shape
    s = np.ascontiguousarray(s, dtype=np.float32)
    if s.shape != (K,):
        raise ValueError("s must have K entries")
    if prev is not None:
        prev = _bf16_2d(prev).copy()
        if prev.shape[1] != K:
            raise ValueError("prev must have K columns")
        R = prev.shape[0]
    else:
        R = 0
    lib().orc_uaq_fold(_ptr(w), N, K, K, _ptr(s),
                       _ptr(prev) if prev is not None else None, R, K)
    return w, prev


def rmsnorm(h, gamma, eps: float):
    """RMSNorm of a bf16 hidden state with the (UAQ-folded) weight gamma, the
    activation the linear layer quantizes.  QuRL notes, 关键设计 §1: the UAQ
    scale s can be folded straight into the norm's scale (gamma' = gamma * s,
    e.g. with ``uaq_fold``).  Reading of the norm (the pages give no formula):
    x = h / sqrt(mean(h^2) + eps) * gamma in fp32 steps, the sum of squares
    accumulated by fused multiply-adds in index order, one rounding to bf16:

      acc = fma-sum of h[m,k]^2 over k in order;  ms = fl32(acc / K)
      r   = fl32(1 / fl32(sqrt(fl32(ms + eps))))
      x   = bf16_RN(fl32(fl32(h * r) * gamma[k]))

    h: bf16 bits [M,K]; gamma: bf16 bits [K]; eps fp32 (>= 0).
    Returns (x bf16 bits [M,K], rstd f32 [M] = r per row).
    """
    h = _bf16_2d(h)
    M, K = h.shape
    g = np.ascontiguousarray(np.asarray(gamma, dtype=np.uint16).reshape(-1))
    if g.shape != (K,):
        raise ValueError("gamma must have K entries")
    x = np.empty((M, K), np.uint16)
    rstd = np.empty((M,), np.float32)
    lib().orc_rmsnorm(_ptr(h), M, K, K, _ptr(g), float(eps), _ptr(x), K, _ptr(rstd))
    return x, rstd


NVFP4_BLOCK = 16


def e2m1_decode(code: int) -> float:
    """Value of a 4-bit E2M1 code (the NVFP4 element format)."""
    return float(lib().orc_e2m1_decode(int(code) & 0xF))


def e2m1_encode(v: float) -> int:
    """RN-even, saturating (+-6) fp32 -> E2M1 code; the sign of zero is kept."""
    return int(lib().orc_e2m1_encode(float(v)))


def quant_nvfp4(w):
    """NVFP4 weight quantization (QeRL news article: 4-bit floats with two-level
    scaling, FP8 E4M3 block scales and an FP32 tensor scale).  w: bf16 bits [N,K],
    K % 16 == 0.  Returns (q u8 [N,K] one E2M1 code per byte, sb u8 [N, K/16]
    E4M3 block-scale codes, st fp32 tensor scale); x ~= e2m1(q) * e4m3(sb) * st.
    """
    w = _bf16_2d(w)
    N, K = w.shape
    if K % NVFP4_BLOCK:
        raise ValueError("K must be a multiple of 16")
    q = np.empty((N, K), np.uint8)
    sb = np.empty((N, K // NVFP4_BLOCK), np.uint8)
    st = np.empty((1,), np.float32)
    lib().orc_quant_nvfp4(_ptr(w), N, K, K, _ptr(q), K, _ptr(sb), K // NVFP4_BLOCK, _ptr(st))
    return q, sb, float(st[0])


def dequant_nvfp4(q, sb, st) -> np.ndarray:
    """fp64 values of NVFP4 codes: e2m1(q) * e4m3(sb) (per 16-block) * st."""
    lut4 = np.array([e2m1_decode(c) for c in range(16)])
    v = lut4[np.asarray(q) & 0xF]
    s = dequant_codes(np.asarray(sb)).repeat(NVFP4_BLOCK, axis=1)
    return v * s * float(st)


def gemm_nvfp4_weight_only(x, q, sb, st, rows=None, cols=None) -> np.ndarray:
    """Y = X W^T with bf16 activations and NVFP4 weights (QeRL news article: the
    rollout runs FP4 x BF16 kernels): W[n, k] = e2m1(q[n, k]) * e4m3(sb[n, k/16]) * st.
    x: bf16 bits [M, K]; q: one E2M1 code per byte [N, K] (as ``quant_nvfp4``
    returns); sb [N, K/16]; st fp32.  fp64: the bf16 values, the E2M1 x E4M3
    products and their K-term sums are exact for moderate K, then one scaling by st.
    """
    xr = bf16_to_f32(np.asarray(x))
    rows = np.arange(xr.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(np.asarray(q).shape[0]) if cols is None else np.asarray(cols)
    lut4 = np.array([e2m1_decode(c) for c in range(16)])
    wq = lut4[np.asarray(q)[cols] & 0xF] * dequant_codes(np.asarray(sb)[cols]).repeat(NVFP4_BLOCK, axis=1)
    return (xr[rows].astype(np.float64) @ wq.T) * float(st)


def aqn_sigma(sigma_start: float, sigma_end: float, t: int, T: int) -> float:
    """Noise level of AQN step t of T: geometric from sigma_start (t = 0) to
    sigma_end (t = T - 1), as an fp32 value.  QeRL news article: adaptive
    quantization noise decays on an exponential schedule."""
    return float(lib().orc_aqn_sigma(sigma_start, sigma_end, t, T))


def aqn_perturb(gamma, z, sigma: float):
    """AQN on a copy of a norm scale: gamma'[k] = bf16_RN(fl32(gamma[k] + fl32(sigma * z[k]))).

    gamma: bf16 bits [K]; z: f32 [K] (one standard-normal draw per channel, made
    by the caller).  QeRL news article: channel-wise Gaussian perturbations
    mapped into the LayerNorm scale parameters."""
    g = np.ascontiguousarray(np.asarray(gamma, dtype=np.uint16)).copy()
    z = np.ascontiguousarray(z, dtype=np.float32)
    if g.ndim != 1 or z.shape != g.shape:
        raise ValueError("gamma and z must be 1-D of the same length")
    lib().orc_aqn_perturb(_ptr(g), g.size, _ptr(z), sigma)
    return g


# ------------------------------------------------------------ fp64 GEMMs ---

def block_scaled_gemm(a_codes, sa, b_codes, sb) -> np.ndarray:
    """Y[r, c] = sum_cb sa[cb, r] * sb[cb, c] * sum_{j in cb} a[r, j] * b[c, j].

    a_codes u8 [R, L], b_codes u8 [C, L] (L = contraction length, blocks of 128
    along it, the last one possibly partial); sa [ceil(L/128), R],
    sb [ceil(L/128), C].  Every code product and 128-term sum is exact in fp64,
    and so is sa * sb; only the per-block scaling and the sum over blocks round.
    """
    a = dequant_codes(a_codes)
    b = dequant_codes(b_codes)
    R, L = a.shape
    C = b.shape[0]
    LB = (L + GRP - 1) // GRP
    sa = np.asarray(sa, np.float64)
    sb = np.asarray(sb, np.float64)
    assert b.shape[1] == L and sa.shape == (LB, R) and sb.shape == (LB, C)
    y = np.zeros((R, C), np.float64)
    for cb in range(LB):
        j0, j1 = cb * GRP, min(L, (cb + 1) * GRP)
        partial = a[:, j0:j1] @ b[:, j0:j1].T
        y += (sa[cb][:, None] * sb[cb][None, :]) * partial
    return y


def gemm_fprop(qx, sx, qw, sw, rows=None, cols=None) -> np.ndarray:
    """FProp Y = X W^T from 1x128 X codes and 128x128 W codes.

    qx [M,K], sx [K/128, M], qw [N,K], sw [N/128, K/128].  Optional row / column
    index arrays restrict the output to Y[rows][:, cols].
    """
    qx, sx = np.asarray(qx), np.asarray(sx)
    qw, sw = np.asarray(qw), np.asarray(sw)
    rows = np.arange(qx.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(qw.shape[0]) if cols is None else np.asarray(cols)
    sb = sw[cols // GRP, :].T  # [K/128, len(cols)]
    return block_scaled_gemm(qx[rows], sx[:, rows], qw[cols], sb)


def gemm_dgrad(qdy, sdy, qw, sw, rows=None, cols=None) -> np.ndarray:
    """DGrad dX = dY W from 1x128 dY codes (along N) and 128x128 W codes.

    qdy [M,N], sdy [N/128, M], qw [N,K], sw [N/128, K/128].  The weight blocks
    are the FProp ones read transposed: the scale of contraction block nb and
    output column k is sw[nb, k // 128].
    """
    qdy, sdy = np.asarray(qdy), np.asarray(sdy)
    qw, sw = np.asarray(qw), np.asarray(sw)
    rows = np.arange(qdy.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(qw.shape[1]) if cols is None else np.asarray(cols)
    b = np.ascontiguousarray(qw[:, cols].T)  # [len(cols), N]
    sb = sw[:, cols // GRP]                  # [N/128, len(cols)]
    return block_scaled_gemm(qdy[rows], sdy[:, rows], b, sb)


def gemm_wgrad(qdyT, sdyc, qxT, sxc, rows=None, cols=None) -> np.ndarray:
    """WGrad dW = dY^T X from 128x1 codes of dY and X (both transposed).

    qdyT [N, M], sdyc [ceil(M/128), N], qxT [K, M], sxc [ceil(M/128), K].
    The contraction runs over the M tokens in blocks of 128 (last one partial).
    """
    qdyT, sdyc = np.asarray(qdyT), np.asarray(sdyc)
    qxT, sxc = np.asarray(qxT), np.asarray(sxc)
    rows = np.arange(qdyT.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(qxT.shape[0]) if cols is None else np.asarray(cols)
    return block_scaled_gemm(qdyT[rows], sdyc[:, rows], qxT[cols], sxc[:, cols])


def gemm_per_channel(qx, sx, qw, sw, rows=None, cols=None) -> np.ndarray:
    """Y = diag(sx) (Qx Qw^T) diag(sw): per-token X codes qx [M,K] with sx [M],
    per-channel W codes qw [N,K] with sw [N].  The scales are constant along K,
    so they factor out of the sum: the code products and the K-term sum are exact
    in fp64 (K <= 2^20), and only the two scalings round.
    """
    qx, qw = np.asarray(qx), np.asarray(qw)
    sx, sw = np.asarray(sx, np.float64), np.asarray(sw, np.float64)
    rows = np.arange(qx.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(qw.shape[0]) if cols is None else np.asarray(cols)
    p = dequant_codes(qx[rows]) @ dequant_codes(qw[cols]).T
    return sx[rows][:, None] * p * sw[cols][None, :]


def dequant_rows(q, s) -> np.ndarray:
    """fp64 values of 1x128 codes: x[m, k] = decode(q[m, k]) * s[k // 128, m]."""
    v = dequant_codes(q)
    M, K = v.shape
    return v * np.repeat(np.asarray(s, np.float64).T, GRP, axis=1)[:, :K]


def dequant_weight(q, s) -> np.ndarray:
    """fp64 values of 128x128 codes."""
    v = dequant_codes(q)
    s = np.asarray(s, np.float64)
    return v * np.repeat(np.repeat(s, GRP, axis=0), GRP, axis=1)


def bf16_round(values) -> np.ndarray:
    """fp32 values rounded to bf16 (returned as fp32)."""
    return bf16_to_f32(f32_to_bf16(values))
