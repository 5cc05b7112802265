"""Pins for the oracle's KV-cache quantisers (kv_cache_quant.wgsl:
quantize_kv_fp8_per_token_f32, quantize_kv_int8_f32, quantize_kv_int4_f32 and
their dequantisers).

Checked against hand-computed cases (exact binary32 ties, packing order,
all-zero and constant inputs) and against properties the definitions fix at
any size: the absmax element maps to +-127, the round trip is within half a
step, the INT4 extremes map to codes 0 and 15, and each code is the nearest
integer on its grid."""
import os

import numpy as np
import pytest

import oracle
from quantized_decode_linear_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                out.append([part.split() for part in line.split("|")])
    return out


def test_int8_hand_cases():
    for vals, scale, codes in _rows("kv_quant_int8_cases.txt"):
        x = np.array([vals], np.float32)
        q, s = oracle.kv_quant_int8(x)
        assert s[0] == np.float32(scale[0]), (vals, s)
        assert q[0].tolist() == [int(c) for c in codes], (vals, q)
        # dequantised value: code * scale in binary32
        assert np.array_equal(oracle.kv_dequant_int8(q, s)[0],
                              (q[0].astype(np.float64) * float(s[0])).astype(np.float32))


def test_int4_hand_cases():
    for vals, sz, packed, deq in _rows("kv_quant_int4_cases.txt"):
        x = np.array(vals, np.float32)
        p, sc, zr = oracle.kv_quant_int4(x, len(vals))
        assert sc[0] == np.float32(sz[0])
        assert zr[0] == pytest.approx(float(sz[1]), rel=1e-6, abs=0)
        assert [f"{b:02x}" for b in p] == packed, (vals, p)
        out = oracle.kv_dequant_int4(p, sc, zr, len(vals), len(vals))
        assert out.tolist() == [float(d) for d in deq], (vals, out)


@pytest.mark.parametrize("tokens,dim", [(1, 128), (37, 64), (300, 128), (5, 96)])
def test_int8_properties(tokens, dim):
    x = syn.normal_f32((tokens, dim), seed=tokens + dim) * np.float32(3.0)
    x[0, :] = 0.0  # an all-zero token
    q, s = oracle.kv_quant_int8(x)
    amax = np.abs(x).max(axis=1)
    nz = amax > 0
    assert np.all(s[~nz] == np.float32(1e-8))
    # the absmax element sits on the end of the code range
    idx = np.abs(x).argmax(axis=1)
    assert np.all(np.abs(q[np.arange(tokens), idx])[nz] == 127)
    # the round trip is within half a step (plus the rounding of q * s)
    y = oracle.kv_dequant_int8(q, s)
    err = np.abs(y.astype(np.float64) - x)
    assert np.all(err <= 0.5 * s[:, None] * (1 + 2 ** -20) + np.abs(y) * 2 ** -23)
    # each code is a nearest integer to v / s (ties either way are allowed here)
    r = x.astype(np.float64) / s[:, None].astype(np.float64)
    assert np.all(np.abs(q - r) <= 0.5 + 1e-6)


@pytest.mark.parametrize("n,group", [(256, 32), (4096, 128), (96, 16), (1024, 64), (40, 2)])
def test_int4_properties(n, group):
    x = syn.normal_f32((n,), seed=n + group)
    p, sc, zr = oracle.kv_quant_int4(x, group)
    codes = np.empty(n, np.int64)
    codes[0::2] = p & 0xF
    codes[1::2] = p >> 4
    g = x.reshape(-1, group)
    cg = codes.reshape(-1, group)
    # the group minimum maps to 0 and the maximum to 15
    assert np.all(cg[np.arange(g.shape[0]), g.argmin(axis=1)] == 0)
    assert np.all(cg[np.arange(g.shape[0]), g.argmax(axis=1)] == 15)
    assert np.all((codes >= 0) & (codes <= 15))
    # the round trip is within half a step, up to the roundings of the
    # scale, the zero and the two products
    y = oracle.kv_dequant_int4(p, sc, zr, n, group).reshape(-1, group).astype(np.float64)
    step = sc.astype(np.float64)[:, None]
    span = np.abs(g).max(axis=1, keepdims=True)
    assert np.all(np.abs(y - g) <= 0.5 * step + 8 * 2 ** -23 * (span + step * 15))
