"""Pins for the oracle's AWQ INT4 fused-QKV GEMV (fused_int4_qkv.rs:
QKV_AWQ_SHIFTS, unpack_awq_qkv, fused_int4_qkv_q/_k/_v).

Checked against hand-computed nibble and dequantisation cases from the
page's shift table, and against a brute force that builds the dense weight
from the inverse statement of the packing (physical nibble p of a word holds
column [0, 2, 4, 6, 1, 3, 5, 7][p]) followed by a library float64 matmul.
"""
import os

import numpy as np
import pytest

import oracle
from quantized_decode_linear_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(line.split())
    return rows


def _dense_by_physical_nibbles(qw: np.ndarray) -> np.ndarray:
    k, npk = qw.shape
    col_of_nibble = [0, 2, 4, 6, 1, 3, 5, 7]
    w = np.zeros((k, npk * 8), np.float64)
    for p in range(8):
        nib = (qw >> np.uint32(4 * p)) & np.uint32(0xF)
        w[:, col_of_nibble[p]::8] = nib
    return w


def _run_single(words: np.ndarray, x: np.ndarray, sc=None, zr=None, group=None):
    """one projection in the q slot, tiny k/v slots"""
    k, npk = words.shape
    n = npk * 8
    group = group or k
    sc = np.ones((k // group, n), np.float32) if sc is None else sc
    zr = np.zeros((k // group, n), np.float32) if zr is None else zr
    tiny_qw = np.zeros((k, 1), np.uint32)
    tiny_s = np.ones((k // group, 8), np.float32)
    tiny_z = np.zeros((k // group, 8), np.float32)
    outs, bounds = oracle.int4_qkv(x, n, 8, group, [words, tiny_qw, tiny_qw],
                                   [sc, tiny_s, tiny_s], [zr, tiny_z, tiny_z])
    return outs[0], bounds[0]


def test_nibble_cases_hand_computed():
    for row in _read("awq_nibble_cases.txt"):
        word = int(row[0], 16)
        want = [int(v) for v in row[1:9]]
        out, _ = _run_single(np.array([[word]], np.uint32), np.ones((1, 1), np.float32), group=1)
        assert list(out[0].astype(int)) == want, (hex(word), out[0], want)


def test_dequant_cases_hand_computed():
    for nib, zero, scale, want in (map(float, r) for r in _read("int4_dequant_cases.txt")):
        word = np.array([[int(nib)]], np.uint32)  # column 0 holds nib
        out, _ = _run_single(word, np.ones((1, 1), np.float32),
                             sc=np.full((1, 8), scale, np.float32),
                             zr=np.full((1, 8), zero, np.float32), group=1)
        assert abs(out[0, 0] - want) <= np.spacing(np.float32(max(abs(want), 1e-30))), (
            nib, zero, scale, out[0, 0], want)


def test_one_hot_rows_select_k_and_group():
    k, n, group = 64, 16, 16
    qw, sc, zr = syn.int4_awq(k, n, group, seed=2)
    dense = _dense_by_physical_nibbles(qw)
    for kk in (0, 15, 16, 37, 63):
        x = np.zeros((1, k), np.float32)
        x[0, kk] = 1.0
        out, _ = _run_single(qw, x, sc, zr, group)
        g = kk // group
        want = ((dense[kk].astype(np.float32) - zr[g]) * sc[g]).astype(np.float64)
        assert np.array_equal(out[0], want)


@pytest.mark.parametrize("m,k,nq,nkv,group", [(1, 128, 64, 32, 128), (4, 256, 128, 64, 32),
                                               (3, 512, 256, 128, 128)])
@pytest.mark.parametrize("integer_zeros", [True, False])
def test_brute_force_dense_matmul(m, k, nq, nkv, group, integer_zeros):
    x = syn.normal_f32((m, k), seed=m + k)
    ws = [syn.int4_awq(k, n, group, seed=p, integer_zeros=integer_zeros)
          for p, n in enumerate((nq, nkv, nkv))]
    outs, bounds = oracle.int4_qkv(x, nq, nkv, group, [w[0] for w in ws], [w[1] for w in ws],
                                   [w[2] for w in ws])
    for p, (qw, sc, zr) in enumerate(ws):
        nib = _dense_by_physical_nibbles(qw)
        scf = np.repeat(sc, group, axis=0)
        zrf = np.repeat(zr, group, axis=0)
        w = ((nib.astype(np.float32) - zrf) * scf).astype(np.float64)  # page: f32 dequant
        ref = x.astype(np.float64) @ w
        absref = np.abs(x.astype(np.float64)) @ np.abs(w)
        assert np.allclose(outs[p], ref, rtol=1e-12, atol=1e-12 * absref.max())
        assert np.allclose(bounds[p], absref, rtol=1e-12)
