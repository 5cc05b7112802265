"""Pins for the oracle's weight preparation: FP8 weight quantisation per
output row or per 128x128 block (scale = absmax / 448, the weight recipe of
the workloads, in the scale layouts of w8a8_decode.rs enum W8a8Scale) and
AWQ packing in the shift order of fused_int4_qkv.rs (QKV_AWQ_SHIFTS).

The FP8 quantiser is checked against a library-built implementation (numpy
absmax in binary32, torch float8_e4m3fn cast) on rows and blocks with special
values, and against invariants at larger sizes.  The packer is checked
against the hand-computed words of tests/golden/awq_nibble_cases.txt and
through the oracle's own (separately pinned) AWQ GEMV, which unpacks it.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from quantized_decode_linear_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_e4m3(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def _special_rows(n: int, k: int, seed: int) -> np.ndarray:
    w = syn.normal_f32((n, k), seed=seed, std=0.02)
    w[0] = 0.0                      # all-zero row: scale 0, codes 0x00
    w[1] = -0.0                     # negative zeros keep their sign: 0x80
    w[2] = 1e-6
    w[2, 5] = 3.0                   # one large value, the rest in FP8's subnormal range
    w[3, :] = np.float32(-7.25)     # constant row: every code is -448
    return w


def _reference(fmt: int, w: np.ndarray):
    """numpy absmax / 448 in binary32, torch cast of w / s"""
    n, k = w.shape
    if fmt == oracle.PER_ROW:
        s = (np.abs(w).max(axis=1) / np.float32(448.0)).astype(np.float32)
        div = np.where(s == 0, np.float32(1.0), s)[:, None]
    else:
        pad = (-n) % 128
        a = np.pad(np.abs(w), ((0, pad), (0, 0)))
        nb = a.shape[0] // 128
        s = (a.reshape(nb, 128, k // 128, 128).max(axis=(1, 3)) / np.float32(448.0)).astype(np.float32)
        safe = np.where(s == 0, np.float32(1.0), s)
        div = np.repeat(np.repeat(safe, 128, axis=0)[:n], 128, axis=1)
    return _torch_e4m3((w / div).astype(np.float32)), s


@pytest.mark.parametrize("fmt", [oracle.PER_ROW, oracle.BLOCK128])
@pytest.mark.parametrize("n,k", [(4, 128), (37, 384), (200, 256), (300, 1024)])
def test_fp8_weight_quant_matches_library_cast(fmt, n, k):
    w = _special_rows(n, k, seed=n + k)
    if fmt == oracle.BLOCK128 and n > 128:
        w[128:256, 128:256] = 0.0   # one all-zero block
    codes, s = oracle.fp8_weight_quant(fmt, w)
    ref_codes, ref_s = _reference(fmt, w)
    assert np.array_equal(s.view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(codes, ref_codes)


def test_fp8_weight_quant_special_rows():
    w = _special_rows(8, 256, seed=3)
    codes, s = oracle.fp8_weight_quant(oracle.PER_ROW, w)
    assert s[0] == 0 and s[1] == 0
    assert np.all(codes[0] == 0x00) and np.all(codes[1] == 0x80)
    assert codes[2, 5] == 0x7E                      # the absmax element: 448
    assert np.all(codes[3] == 0xFE)                 # -448 everywhere
    assert np.any((codes[2] & 0x78) == 0) and np.any(codes[2] != 0)  # subnormal codes appear


@pytest.mark.parametrize("fmt", [oracle.PER_ROW, oracle.BLOCK128])
def test_fp8_weight_quant_invariants(fmt):
    n, k = 1000, 2048
    w = syn.normal_f32((n, k), seed=11, std=0.015)
    codes, s = oracle.fp8_weight_quant(fmt, w)
    dec = oracle.e4m3_decode(codes)
    if fmt == oracle.PER_ROW:
        sf = np.repeat(s[:, None], k, axis=1)
        blocks = w.reshape(n, 1, k)
        cb = codes.reshape(n, 1, k)
    else:
        sf = np.repeat(np.repeat(s, 128, axis=0)[:n], 128, axis=1)
        pad = (-n) % 128
        blocks = np.pad(w, ((0, pad), (0, 0))).reshape(-1, 128, k // 128, 128).transpose(0, 2, 1, 3)
        blocks = blocks.reshape(-1, 128 * 128)
        cb = np.pad(codes, ((0, pad), (0, 0))).reshape(-1, 128, k // 128, 128).transpose(0, 2, 1, 3)
        cb = cb.reshape(-1, 128 * 128)
        blocks = blocks.reshape(blocks.shape[0], 1, -1)
        cb = cb.reshape(cb.shape[0], 1, -1)
    # the absmax element of every row / block codes to +-448
    flat_w = blocks.reshape(blocks.shape[0], -1)
    flat_c = cb.reshape(cb.shape[0], -1)
    arg = np.abs(flat_w).argmax(axis=1)
    assert np.all((flat_c[np.arange(flat_c.shape[0]), arg] & 0x7F) == 0x7E)
    # every code is within half an FP8 step (3 mantissa bits) of w / s
    q = w / sf
    assert np.all(np.abs(dec - q) <= np.maximum(np.abs(q) * 2.0**-4, 2.0**-10) + 1e-6)


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(line.split())
    return rows


def test_awq_pack_hand_cases():
    """column codes -> the hand-computed packed word (QKV_AWQ_SHIFTS)"""
    for row in _read_golden("awq_nibble_cases.txt"):
        word = int(row[0], 16)
        cols = np.array([[int(v) for v in row[1:9]]], np.uint8)
        assert int(oracle.awq_pack(cols)[0, 0]) == word, (row, hex(int(oracle.awq_pack(cols)[0, 0])))


@pytest.mark.parametrize("k,n", [(1, 8), (16, 64), (128, 256)])
def test_awq_pack_unpacked_by_the_gemv(k, n):
    """packing random codes, then the oracle's AWQ GEMV with one-hot x,
    unit scales and zero zeros returns the codes (the GEMV's unpacking is
    pinned separately)"""
    rng = np.random.default_rng(k + n)
    nib = rng.integers(0, 16, size=(k, n), dtype=np.uint8)
    qw = oracle.awq_pack(nib)
    x = np.eye(k, dtype=np.float32)
    tiny_qw = np.zeros((k, 1), np.uint32)
    ones = np.ones((1, n), np.float32)
    zeros = np.zeros((1, n), np.float32)
    outs, _ = oracle.int4_qkv(x, n, 8, k, [qw, tiny_qw, tiny_qw], [ones, ones[:, :8], ones[:, :8]],
                              [zeros, zeros[:, :8], zeros[:, :8]])
    assert np.array_equal(outs[0], nib.astype(np.float64))


def test_awq_pack_uses_low_nibble_only():
    nib = np.array([[0x10, 0xF1, 0x22, 0x03, 0x04, 0x05, 0x06, 0x07]], np.uint8)
    assert int(oracle.awq_pack(nib)[0, 0]) == int(oracle.awq_pack(nib & 0xF)[0, 0])
