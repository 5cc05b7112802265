"""Pins for the oracle's W8A8 GEMV (w8a8_decode.rs: w8a8_gemv,
W8a8Weight::new, W8a8Weight::boundaries).

Checked against a library computation (torch float8 decode -> float64
matmul), hand-computed segment routing, and the identities the definition
implies (segments = concatenation, M rows = M single-row calls, one K block of
Block128 = PerRow with the block's scale, zero rows give zero).
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_decode_linear_gb300 import synthetic as syn


def _lib_dequant_w(codes, scale, fmt, k):
    w = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64)
    s = torch.from_numpy(scale).to(torch.float64)
    if fmt == oracle.PER_ROW:
        return w * s[:, None]
    n = codes.shape[0]
    full = s.repeat_interleave(128, 0)[:n].repeat_interleave(128, 1)
    return w * full


def _lib_dequant_x(q, s, fmt):
    x = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64)
    st = torch.from_numpy(s).to(torch.float64)
    if fmt == oracle.PER_ROW:
        return x * st[:, None]
    return x * st.repeat_interleave(128, 1)


def _case(fmt, rows, k, segs, seed=0):
    x = syn.bf16_normal((rows, k), seed)
    q, s = oracle.act_quant(fmt, x, k)
    ws = [syn.fp8_weight(n, k, fmt, 0.02, seed + 1 + i) for i, n in enumerate(segs)]
    return q, s, ws


@pytest.mark.parametrize("fmt", [oracle.PER_ROW, oracle.BLOCK128])
@pytest.mark.parametrize("rows,k,segs", [(1, 128, [16]), (3, 256, [48, 32]),
                                          (5, 384, [128, 256, 100]), (2, 512, [256, 256, 256])])
def test_gemv_matches_library_matmul(fmt, rows, k, segs):
    if fmt == oracle.PER_ROW:
        segs = [n if i == len(segs) - 1 else (n + 15) // 16 * 16 for i, n in enumerate(segs)]
    else:
        segs = [n if i == len(segs) - 1 else (n + 127) // 128 * 128 for i, n in enumerate(segs)]
    q, s, ws = _case(fmt, rows, k, segs)
    y, b = oracle.w8a8_gemv(fmt, q, s, ws)
    W = torch.cat([_lib_dequant_w(c, sc, fmt, k) for c, sc in ws], 0)
    X = _lib_dequant_x(q, s, fmt)
    ref = (X @ W.T).numpy()
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    absref = (X.abs() @ W.abs().T).numpy()
    assert np.allclose(b, absref, rtol=1e-12)
    assert np.all(b >= np.abs(y) - 1e-12)


def test_segment_routing_hand_computed():
    # three segments whose codes decode to 1, 2 and 4 (0x38, 0x40, 0x48), unit
    # scales, x all ones (act scale 1/448 with code 0x7E = 448): y[j] = K * v_seg
    k = 128
    n = [32, 16, 8]
    ws = [(np.full((nn, k), code, np.uint8), np.ones(nn, np.float32))
          for nn, code in zip(n, (0x38, 0x40, 0x48))]
    q = np.full((1, k), 0x7E, np.uint8)
    s = np.array([1.0 / 448], np.float32)
    y, _ = oracle.w8a8_gemv(oracle.PER_ROW, q, s, ws)
    a = 448.0 * np.float64(np.float32(1.0 / 448))  # act value after dequant
    want = np.concatenate([np.full(32, 128 * a), np.full(16, 256 * a), np.full(8, 512 * a)])
    assert np.allclose(y[0], want, rtol=1e-15)


@pytest.mark.parametrize("fmt", [oracle.PER_ROW, oracle.BLOCK128])
def test_segments_equal_concatenation(fmt):
    q, s, ws = _case(fmt, 4, 256, [128, 128, 96], seed=3)
    y, _ = oracle.w8a8_gemv(fmt, q, s, ws)
    parts = [oracle.w8a8_gemv(fmt, q, s, [w])[0] for w in ws]
    assert np.array_equal(y, np.concatenate(parts, axis=1))


@pytest.mark.parametrize("fmt", [oracle.PER_ROW, oracle.BLOCK128])
def test_rows_equal_single_row_calls(fmt):
    q, s, ws = _case(fmt, 6, 256, [128, 64], seed=4)
    y, _ = oracle.w8a8_gemv(fmt, q, s, ws)
    for m in range(6):
        ym, _ = oracle.w8a8_gemv(fmt, q[m:m + 1], s[m:m + 1], ws)
        assert np.array_equal(ym[0], y[m])


def test_single_block_block128_equals_perrow():
    k = 128
    q, s, ws = _case(oracle.BLOCK128, 3, k, [256], seed=5)
    codes, bscale = ws[0]  # bscale [2, 1]
    y_b, _ = oracle.w8a8_gemv(oracle.BLOCK128, q, s, ws)
    rscale = np.repeat(bscale[:, 0], 128).astype(np.float32)
    y_r, _ = oracle.w8a8_gemv(oracle.PER_ROW, q, s[:, 0].copy(), [(codes, rscale)])
    assert np.allclose(y_b, y_r, rtol=1e-15, atol=0)


def test_zero_weight_row_gives_zero():
    q, s, ws = _case(oracle.PER_ROW, 2, 256, [32], seed=6)
    codes, sc = ws[0]
    codes = codes.copy()
    codes[7] = 0
    y, b = oracle.w8a8_gemv(oracle.PER_ROW, q, s, [(codes, sc)])
    assert np.all(y[:, 7] == 0) and np.all(b[:, 7] == 0)


def test_sampled_equals_full():
    q, s, ws = _case(oracle.BLOCK128, 4, 256, [128, 128, 40], seed=8)
    y, b = oracle.w8a8_gemv(oracle.BLOCK128, q, s, ws)
    rng = np.random.default_rng(0)
    r = rng.integers(0, 4, 50)
    c = rng.integers(0, 296, 50)
    ys, bs = oracle.w8a8_gemv_sampled(oracle.BLOCK128, q, s, ws, r, c)
    assert np.array_equal(ys, y[r, c]) and np.array_equal(bs, b[r, c])


def test_result_does_not_depend_on_thread_count():
    """the oracle's parallel loops split output columns only, so one thread
    and all threads give the same bits (the CPU baseline times both)"""
    q, s, ws = _case(oracle.BLOCK128, 3, 512, [256, 128, 72], seed=11)
    cores = oracle.num_threads()
    y, b = oracle.w8a8_gemv(oracle.BLOCK128, q, s, ws)
    oracle.set_num_threads(1)
    try:
        assert oracle.num_threads() == 1 or cores == 1
        y1, b1 = oracle.w8a8_gemv(oracle.BLOCK128, q, s, ws)
    finally:
        oracle.set_num_threads(cores)
    assert oracle.num_threads() == cores
    assert np.array_equal(y, y1) and np.array_equal(b, b1)
