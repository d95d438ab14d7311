"""GPU parity of the quantizers (through the C ABI) against the oracle: codes
and scales bit-exact, on ragged and multi-tile shapes, crafted edge values,
pitched buffers with guard bands, the full-size workloads, and the exhaustive
(x, amax) bf16 element map."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_quantize_gb300 import inputs as I
from fp8_block_scaled_quantize_gb300 import rlq
from gpu_util import normal_bits, np_, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [(1, 128), (7, 256), (128, 128), (129, 384), (200, 512), (1000, 1024), (4096, 4096)]


def _check_rows(x_bits, q, s):
    oq, os_ = oracle.quant_rows_1x128(x_bits)
    assert np.array_equal(np_(q), oq), "row-wise codes differ"
    assert np.array_equal(np_(s), os_), "row-wise scales differ"


def _check_cols(x_bits, qT, sc):
    oqT, osc = oracle.quant_cols_128x1(x_bits)
    assert np.array_equal(np_(qT), oqT), "column-wise codes differ"
    assert np.array_equal(np_(sc), osc), "column-wise scales differ"


@pytest.mark.parametrize("M,K", SHAPES)
def test_rowwise_parity(M, K):
    x = normal_bits(10, (M, K))
    q, s, qT, sc = rlq.quant_act_1x128(to_dev(x))
    assert qT is None and sc is None
    _check_rows(x, q, s)


@pytest.mark.parametrize("K", [640, 1152, 1920, 2176, 2304, 4224, 6272])
def test_rowwise_segment_boundaries(K):
    """Row lengths whose segments (up to 16 groups per warp) end inside the last
    load or leave whole loads unused: 3, 5, 8 loads of one segment; 2, 3 and 4
    segments per row with 5 to 7 loads each."""
    x = normal_bits(11, (37, K))
    q, s, _, _ = rlq.quant_act_1x128(to_dev(x))
    _check_rows(x, q, s)


@pytest.mark.parametrize("M,K", SHAPES)
def test_dual_parity(M, K):
    x = normal_bits(11, (M, K), std=1e-3)
    q, s, qT, sc = rlq.quant_act_1x128(to_dev(x), colwise=True)
    _check_rows(x, q, s)
    _check_cols(x, qT, sc)


@pytest.mark.parametrize("N,K", [(128, 128), (256, 384), (1024, 512), (384, 1280)])
@pytest.mark.parametrize("transposed", [False, True])
def test_weight_parity(N, K, transposed):
    w = normal_bits(12, (N, K), std=0.02)
    q, s, qT = rlq.quant_weight_128x128(to_dev(w), transposed=transposed)
    oq, os_, oqT = oracle.quant_weight_128x128(w, transposed=transposed)
    assert np.array_equal(np_(q), oq) and np.array_equal(np_(s), os_)
    if transposed:
        assert np.array_equal(np_(qT), oqT)



def _group_scaled(seed, M, K, span=30):
    """N(0,1) values times 2^e with e drawn per 1x128 group, times a per-column
    factor in [1, 2): every row group, column group and 128x128 block of a tile
    has its own magnitude."""
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((M, K)).astype(np.float32)
    e = rng.integers(-span, span + 1, size=(M, K // 128))
    v *= np.exp2(e).repeat(128, axis=1).astype(np.float32)
    v *= (1.0 + rng.random((1, K))).astype(np.float32)
    return I.to_bf16_bits(v)


@pytest.mark.parametrize("M,K", [(128, 256), (300, 512), (1000, 384)])
def test_group_scales_differ_within_a_tile(M, K):
    """A scale handed to the wrong group (row or column) or computed from the wrong
    lanes changes codes here, since no two neighbouring groups share a magnitude."""
    x = _group_scaled(31, M, K)
    q, s, qT, sc = rlq.quant_act_1x128(to_dev(x), colwise=True)
    _check_rows(x, q, s)
    _check_cols(x, qT, sc)
    q2, s2, _, _ = rlq.quant_act_1x128(to_dev(x))
    _check_rows(x, q2, s2)


def test_weight_block_scales_differ():
    """Weight blocks with magnitudes 2^-30 .. 2^30 apart, with the transposed copy."""
    w = _group_scaled(32, 640, 768)
    q, s, qT = rlq.quant_weight_128x128(to_dev(w), transposed=True)
    oq, os_, oqT = oracle.quant_weight_128x128(w, transposed=True)
    assert np.array_equal(np_(s), os_), "block scales differ"
    assert np.array_equal(np_(q), oq), "block codes differ"
    assert np.array_equal(np_(qT), oqT), "transposed codes differ"

def _edge_matrix(M=256, K=1024):
    """Groups that stress the corner cases: all-zero and signed-zero groups,
    subnormal bf16 (subnormal scales), the largest bf16, exact E4M3
    midpoints at scale 1, alternating signs, single outliers."""
    rng = np.random.default_rng(77)
    v = rng.standard_normal((M, K)).astype(np.float32)
    v[0, :128] = 0.0
    v[1, :128] = -0.0
    v[1, 128:256] = np.where(np.arange(128) % 2, 0.0, -0.0)
    sub = (np.arange(1, 129, dtype=np.uint32) << 16).view(np.float32)  # bf16 subnormals 2^-133 ..
    v[2, :128] = sub
    v[3, :128] = -sub[::-1]
    v[4, :128] = np.float32(3.3895314e38)  # largest finite bf16
    v[4, 5] = -3.3895314e38
    grid = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)  # 126 midpoints, exact in bf16
    v[5, :126] = mids
    v[5, 126] = 0.0
    v[5, 127] = 448.0  # amax 448: scale exactly 1, so the midpoints are ties
    v[6, :128] = np.where(np.arange(128) % 2, 1.0, -1.0) * np.float32(1e-30)
    v[7, 300] = 1e4
    v[8:12] = v[8:12] * np.float32(2.0 ** -120)  # tiny scales (below 2^-100 after /448)
    v[12:16] = v[12:16] * np.float32(2.0 ** 100)
    bits = I.to_bf16_bits(v)
    return bits


def test_edge_values_all_quantizers():
    x = _edge_matrix()
    q, s, qT, sc = rlq.quant_act_1x128(to_dev(x), colwise=True)
    _check_rows(x, q, s)
    _check_cols(x, qT, sc)
    q2, s2, _, _ = rlq.quant_act_1x128(to_dev(x))
    _check_rows(x, q2, s2)
    wq, ws, wqT = rlq.quant_weight_128x128(to_dev(x), transposed=True)
    oq, os_, oqT = oracle.quant_weight_128x128(x, transposed=True)
    assert np.array_equal(np_(wq), oq) and np.array_equal(np_(ws), os_) and np.array_equal(np_(wqT), oqT)
    # the tie row: codes of the midpoints are the even neighbours
    assert np.all(np_(q)[5, :127] % 2 == 0)


SENT = 0xA5


def test_pitched_buffers_and_guard_bands():
    """ld > row length everywhere; nothing outside the described regions is written."""
    M, K = 300, 384
    x = normal_bits(13, (M, K))
    dev = "cuda"
    xb = torch.zeros((M, K + 64), dtype=torch.bfloat16, device=dev)
    xb[:, :K] = to_dev(x)
    qb = torch.full((M + 3, K + 48), SENT, dtype=torch.uint8, device=dev)
    sb = torch.full((K // 128 + 1, M + 17), -7.0, dtype=torch.float32, device=dev)
    ldqT = 320
    qTb = torch.full((K + 2, ldqT), SENT, dtype=torch.uint8, device=dev)
    MB = (M + 127) // 128
    scb = torch.full((MB + 1, K + 20), -7.0, dtype=torch.float32, device=dev)
    s_ = torch.cuda.current_stream().cuda_stream
    rlq.rlq_quant_act_1x128(xb.data_ptr(), M, K, K + 64, qb.data_ptr(), K + 48, sb.data_ptr(), M + 17,
                            qTb.data_ptr(), ldqT, scb.data_ptr(), K + 20, s_)
    rlq.check()
    oq, os_ = oracle.quant_rows_1x128(x)
    oqT, osc = oracle.quant_cols_128x1(x)
    qh, sh, qTh, sch = np_(qb), np_(sb), np_(qTb), np_(scb)
    assert np.array_equal(qh[:M, :K], oq) and np.all(qh[:M, K:] == SENT) and np.all(qh[M:] == SENT)
    assert np.array_equal(sh[:K // 128, :M], os_) and np.all(sh[:K // 128, M:] == -7) and np.all(sh[K // 128:] == -7)
    assert np.array_equal(qTh[:K, :M], oqT) and np.all(qTh[:K, M:] == SENT) and np.all(qTh[K:] == SENT)
    assert np.array_equal(sch[:MB, :K], osc) and np.all(sch[:MB, K:] == -7) and np.all(sch[MB:] == -7)

    # weights with pitches and the transposed copy
    N = 256
    w = normal_bits(14, (N, K), std=0.02)
    wb = torch.zeros((N, K + 8), dtype=torch.bfloat16, device=dev)
    wb[:, :K] = to_dev(w)
    wq = torch.full((N + 1, K + 16), SENT, dtype=torch.uint8, device=dev)
    ws = torch.full((N // 128 + 1, K // 128 + 5), -7.0, dtype=torch.float32, device=dev)
    wqT = torch.full((K + 1, N + 32), SENT, dtype=torch.uint8, device=dev)
    rlq.rlq_quant_weight_128x128(wb.data_ptr(), N, K, K + 8, wq.data_ptr(), K + 16, ws.data_ptr(), K // 128 + 5,
                                 wqT.data_ptr(), N + 32, s_)
    rlq.check()
    oq, os_, oqT = oracle.quant_weight_128x128(w, transposed=True)
    wqh, wsh, wqTh = np_(wq), np_(ws), np_(wqT)
    assert np.array_equal(wqh[:N, :K], oq) and np.all(wqh[:N, K:] == SENT) and np.all(wqh[N:] == SENT)
    assert np.array_equal(wsh[:N // 128, :K // 128], os_) and np.all(wsh[:N // 128, K // 128:] == -7)
    assert np.array_equal(wqTh[:K, :N], oqT) and np.all(wqTh[:K, N:] == SENT) and np.all(wqTh[K:] == SENT)


def test_empty_inputs_are_noops():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    q, s, qT, sc = rlq.quant_act_1x128(x, colwise=True)
    assert q.shape == (0, 256) and qT.shape == (256, 0) and sc.shape == (0, 256)
    w = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    rlq.quant_weight_128x128(w)
    rlq.check()


# ------------------------------------------------------- full-size workloads ---

def test_full_size_decode_upproj_8b():
    d = I.decode_upproj_8b()
    q, s, _, _ = rlq.quant_act_1x128(to_dev(d["x"]))
    _check_rows(d["x"], q, s)
    wq, ws, wqT = rlq.quant_weight_128x128(to_dev(d["w"]), transposed=True)
    oq, os_, oqT = oracle.quant_weight_128x128(d["w"], transposed=True)
    assert np.array_equal(np_(wq), oq) and np.array_equal(np_(ws), os_) and np.array_equal(np_(wqT), oqT)


def test_full_size_train_step_8b():
    d = I.train_step_8b()
    for name in ("x", "dy"):
        q, s, qT, sc = rlq.quant_act_1x128(to_dev(d[name]), colwise=True)
        _check_rows(d[name], q, s)
        _check_cols(d[name], qT, sc)
        del q, s, qT, sc


@pytest.mark.parametrize("which", ["gate_up", "down"])
def test_full_size_qwen7b(which):
    d = I.qwen7b_layer(4096, which)
    q, s, _, _ = rlq.quant_act_1x128(to_dev(d["x"]))
    _check_rows(d["x"], q, s)
    wq, ws, _ = rlq.quant_weight_128x128(to_dev(d["w"]))
    oq, os_, _ = oracle.quant_weight_128x128(d["w"])
    assert np.array_equal(np_(wq), oq) and np.array_equal(np_(ws), os_)


@pytest.mark.parametrize("orient", ["up", "down"])
@pytest.mark.parametrize("M", [1, 16, 1024, 16384])
def test_full_size_sweep_32b(orient, M):
    d = I.sweep_32b(M, orient, with_w=(M == 1))
    q, s, qT, sc = rlq.quant_act_1x128(to_dev(d["x"]), colwise=True)
    _check_rows(d["x"], q, s)
    _check_cols(d["x"], qT, sc)
    if M <= 1024:
        q, s, qT, sc = rlq.quant_act_1x128(to_dev(d["dy"]), colwise=True)
        _check_rows(d["dy"], q, s)
        _check_cols(d["dy"], qT, sc)
    if "w" in d:
        wq, ws, _ = rlq.quant_weight_128x128(to_dev(d["w"]))
        oq, os_, _ = oracle.quant_weight_128x128(d["w"])
        assert np.array_equal(np_(wq), oq) and np.array_equal(np_(ws), os_)


# ----------------------------------------------------- exhaustive element map ---

def _pair_groups(a_lo, a_hi, width=127):
    """Groups [amax, x_1 .. x_width] covering every bf16 x with |x| <= amax, both
    signs, for amax bit patterns a_lo .. a_hi-1 (positive finite)."""
    a = np.arange(a_lo, a_hi, dtype=np.int64)
    lens = 2 * (a + 1)
    ng = (lens + width - 1) // width
    padded = ng * width
    starts = np.concatenate([[0], np.cumsum(padded)[:-1]])
    j = np.arange(int(padded.sum()), dtype=np.int64) - np.repeat(starts, padded)
    ar = np.repeat(a, padded)
    v = np.where(j <= ar, j, np.where(j < 2 * (ar + 1), (j - (ar + 1)) | 0x8000, ar))
    body = v.reshape(-1, width)
    head = np.repeat(a, ng)[:, None]
    return np.concatenate([head, body], axis=1).astype(np.uint16)


@pytest.mark.slow
def test_exhaustive_element_map_rowwise_and_colwise():
    """Every (x, amax) bf16 pair with |x| <= amax, as 1x128 groups (row-wise
    kernel) and, transposed, as 128x1 groups (fused kernel)."""
    total = 0
    # chunk boundaries equalising the pair count (it grows as amax^2)
    edges = np.unique(np.sqrt(np.linspace(1, 0x7F80 ** 2, 33)).astype(np.int64))
    edges[0], edges[-1] = 1, 0x7F80
    for lo, hi in zip(edges[:-1], edges[1:]):
        g = _pair_groups(int(lo), int(hi))
        G = g.shape[0]
        per_row = 64
        pad = (-G) % per_row
        x = np.concatenate([g, np.zeros((pad, 128), np.uint16)]) if pad else g
        x = x.reshape(-1, per_row * 128)
        q, s, _, _ = rlq.quant_act_1x128(to_dev(x))
        _check_rows(x, q, s)
        del q, s
        # the same groups as 128x1 column groups: column j of xt is group j
        Gc = (G // 128) * 128
        xt = np.ascontiguousarray(g[:Gc].T)
        _, _, qT, sc = rlq.quant_act_1x128(to_dev(xt), colwise=True)
        _check_cols(xt, qT, sc)
        del qT, sc
        total += G * 127
    assert total >= 1_065_000_000
