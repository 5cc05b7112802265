"""Pins for the oracle's activation quantisation (w8a8_decode.rs:
w8a8_act_quant, w8a8_act_quant_silu, W8a8Scale::act_scales_per_row).

Checked against invariants the definition fixes (the absmax element codes to
+-448, every code is the nearest grid value of x / s, scales are absmax/448
in binary32), special cases (PerRow on one 128-group equals Block128, SiLU
with large gate and unit up reduces to the plain quantiser, all-zero groups),
and a library-built implementation (torch float8 cast) on random data.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_decode_linear_gb300 import synthetic as syn


def _f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _groups(fmt, k):
    return k if fmt == oracle.PER_ROW else 128


@pytest.mark.parametrize("fmt", [oracle.PER_ROW, oracle.BLOCK128])
@pytest.mark.parametrize("rows,k,ldx", [(1, 128, 128), (3, 1024, 1032), (8, 4096, 4096)])
def test_act_quant_invariants(fmt, rows, k, ldx):
    x = syn.bf16_normal((rows, ldx), seed=rows * 7 + k)
    q, s = oracle.act_quant(fmt, x, k)
    xf = _f32(x[:, :k])
    g = _groups(fmt, k)
    xg = xf.reshape(rows, k // g, g)
    sg = s.reshape(rows, k // g)
    amax = np.abs(xg).max(axis=2)
    # scale is the binary32 quotient absmax / 448
    assert np.array_equal(sg, (amax / np.float32(448.0)).astype(np.float32))
    # the absmax element of each group codes to +-448
    arg = np.abs(xg).argmax(axis=2)
    qg = q.reshape(rows, k // g, g)
    top = np.take_along_axis(qg, arg[..., None], axis=2)[..., 0]
    assert np.all((top & 0x7F) == 0x7E)
    # library-built reference: torch's RNE cast of the binary32 quotient
    quot = (xg / sg[..., None]).astype(np.float32)
    lib = torch.from_numpy(np.clip(quot, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(qg, lib.numpy())


def test_perrow_on_one_group_equals_block128():
    x = syn.bf16_normal((5, 128), seed=3)
    q1, s1 = oracle.act_quant(oracle.PER_ROW, x, 128)
    q2, s2 = oracle.act_quant(oracle.BLOCK128, x, 128)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2[:, 0])


def test_zero_groups_and_signed_zero():
    x = np.zeros((2, 256), np.uint16)
    x[1, :128] = 0x8000  # -0 in the first group of row 1
    x[1, 200] = 0x3F80  # 1.0 in the second group
    q, s = oracle.act_quant(oracle.BLOCK128, x, 256)
    assert np.all(s[0] == 0) and s[1, 0] == 0 and s[1, 1] == np.float32(1.0) / np.float32(448)
    assert np.all(q[0] == 0) and np.all(q[1, :128] == 0x80)
    assert q[1, 200] == 0x7E and np.all(np.delete(q[1, 128:], 72) == 0)
    qr, sr = oracle.act_quant(oracle.PER_ROW, x, 256)
    assert sr[0] == 0 and np.all(qr[0] == 0)


def test_row_stride_is_honoured():
    x = syn.bf16_normal((4, 640), seed=11)
    q1, s1 = oracle.act_quant(oracle.BLOCK128, x, 512)
    q2, s2 = oracle.act_quant(oracle.BLOCK128, np.ascontiguousarray(x[:, :512]), 512)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


@pytest.mark.parametrize("fmt", [oracle.PER_ROW, oracle.BLOCK128])
def test_silu_with_large_gate_and_unit_up_is_plain_quant(fmt):
    # silu(g) = g / (1 + e^-g) = g exactly in binary32 once e^-g < 2^-25
    g = np.abs(syn.normal_f32((3, 256), seed=5)) * 10 + 20
    gate = syn.to_bf16_bits(g)
    up = syn.to_bf16_bits(np.ones_like(g))
    q1, s1 = oracle.act_quant_silu(fmt, gate, up, 256)
    q2, s2 = oracle.act_quant(fmt, gate, 256)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


@pytest.mark.parametrize("fmt", [oracle.PER_ROW, oracle.BLOCK128])
def test_silu_quant_matches_double_silu_up_to_ties(fmt):
    rows, k = 4, 512
    buf = syn.bf16_normal((rows, 2 * k), seed=9)
    gate, up = buf[:, :k], buf[:, k:]
    q, s = oracle.act_quant_silu(fmt, gate, up, k)
    g64 = _f32(gate).astype(np.float64)
    u64 = _f32(up).astype(np.float64)
    act = g64 / (1 + np.exp(-g64)) * u64
    grp = _groups(fmt, k)
    ag = act.reshape(rows, k // grp, grp)
    amax = np.abs(ag).max(axis=2)
    sg = s.reshape(rows, k // grp)
    assert np.allclose(sg, amax / 448, rtol=1e-6)
    # dequantised codes are within half an FP8 step (plus a hair for the
    # binary32 rounding of the activation) of act / s
    dec = oracle.e4m3_decode(q).reshape(ag.shape).astype(np.float64)
    ratio = ag / sg[..., None]
    step = np.where(np.abs(ratio) < 2.0**-6, 2.0**-9,
                    2.0**(np.floor(np.log2(np.maximum(np.abs(ratio), 2.0**-6))) - 3))
    assert np.all(np.abs(dec - ratio) <= step / 2 * (1 + 1e-5) + 1e-12)


def test_silu_separate_strides():
    rows, k = 3, 256
    g = syn.bf16_normal((rows, 300), seed=1)
    u = syn.bf16_normal((rows, 400), seed=2)
    q1, s1 = oracle.act_quant_silu(oracle.BLOCK128, g[:, :k], u[:, :k], k)
    q2, s2 = oracle.act_quant_silu(oracle.BLOCK128, np.ascontiguousarray(g[:, :k]),
                                   np.ascontiguousarray(u[:, :k]), k)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)
