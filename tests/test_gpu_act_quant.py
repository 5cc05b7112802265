"""GPU parity: activation quantisation codes and scales bit-exact against the
oracle (w8a8_decode.rs: w8a8_act_quant, w8a8_act_quant_silu)."""
import numpy as np
import pytest
import torch

import oracle
import quantized_decode_linear_gb300 as qdl
from quantized_decode_linear_gb300 import synthetic as syn
from _gpu import bf16_dev, f32_bits_equal, host, scratch

pytestmark = pytest.mark.gpu

SHAPES = [(1, 128, 128), (1, 1024, 1024), (3, 384, 392), (8, 4096, 4096), (17, 8192, 8200),
          (64, 14336, 14336), (256, 8192, 8192), (2, 65536, 65536), (256, 128, 136)]


def _run(fmt, x_bits, rows, k, silu=False, up_bits=None):
    q, s = scratch(rows, k, fmt)
    if silu:
        g, u = bf16_dev(x_bits), bf16_dev(up_bits)
        qdl.act_quant_silu(fmt, g, u, rows, k, q, s)
    else:
        x = bf16_dev(x_bits)
        qdl.act_quant(fmt, x, rows, k, q, s)
    torch.cuda.synchronize()
    sh = host(s)
    return host(q), (sh[:, 0] if fmt == qdl.PER_ROW else sh)


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
@pytest.mark.parametrize("rows,k,ldx", SHAPES)
def test_act_quant_bit_exact(fmt, rows, k, ldx):
    x = syn.bf16_normal((rows, ldx), seed=rows + k)
    q, s = _run(fmt, x, rows, k)
    qo, so = oracle.act_quant(fmt, x, k)
    assert np.array_equal(q, qo)
    assert f32_bits_equal(s, so)


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
def test_act_quant_special_values(fmt):
    rows, k = 12, 512
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 16, size=(rows, k), dtype=np.uint32).astype(np.uint16)
    bits[(bits & 0x7F80) == 0x7F80] = 0x3F80          # no inf/NaN (outside the contract)
    bits[0] = 0                                        # all +0
    bits[1] = 0x8000                                   # all -0
    bits[2, :] = 0x0001                                # bf16 subnormals: subnormal scale
    bits[2, 7] = 0x8003
    bits[3, :] = 0x7F7F                                # largest finite bf16
    bits[4, 130] = 0x7F7F                              # one huge value in a row of random ones
    bits[5, :128] = 0x0000
    x = bits
    q, s = _run(fmt, x, rows, k)
    qo, so = oracle.act_quant(fmt, x, k)
    assert np.array_equal(q, qo)
    assert f32_bits_equal(s, so)


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
@pytest.mark.parametrize("rows,k", [(1, 128), (5, 640), (64, 14336), (256, 4096)])
def test_act_quant_silu_bit_exact_one_buffer(fmt, rows, k):
    # gate = columns [0, k), up = columns [k, 2k) of one [rows, 2k] buffer
    buf = syn.bf16_normal((rows, 2 * k), seed=3 * rows + k)
    q, s = scratch(rows, k, fmt)
    d = bf16_dev(buf)
    qdl.act_quant_silu(fmt, d[:, :k], d[:, k:], rows, k, q, s, ld_gate=2 * k, ld_up=2 * k)
    torch.cuda.synchronize()
    qo, so = oracle.act_quant_silu(fmt, buf[:, :k], buf[:, k:], k)
    sh = host(s)
    assert np.array_equal(host(q), qo)
    assert f32_bits_equal(sh[:, 0] if fmt == qdl.PER_ROW else sh, so)


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
def test_act_quant_silu_wide_gate_range_separate_strides(fmt):
    rows, k = 9, 1024
    g = syn.to_bf16_bits(syn.normal_f32((rows, 1032), seed=1) * 30)  # saturating and tiny SiLU
    u = syn.bf16_normal((rows, 1040), seed=2)
    q, s = _run(fmt, g[:, :k].copy(), rows, k, silu=True, up_bits=u[:, :k].copy())
    qo, so = oracle.act_quant_silu(fmt, g[:, :k], u[:, :k], k)
    assert np.array_equal(q, qo)
    assert f32_bits_equal(s, so)
