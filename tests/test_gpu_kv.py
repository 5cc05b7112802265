"""GPU parity: KV-cache quantisers and dequantisers (kv_cache_quant.wgsl:
quantize_kv_fp8_per_token_f32 / quantize_kv_int8_f32, quantize_kv_int4_f32 and
the dequantize_* kernels) against the oracle.  Every step is one binary32
operation on both sides, so codes, scales, zeros and dequantised values must
agree bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import quantized_decode_linear_gb300 as qdl
from quantized_decode_linear_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _bits_equal(a, b):
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))


def _values(tokens, dim, seed):
    """normal values with a spread of magnitudes, an all-zero token, a tiny
    token, a constant token and exact halfway cases"""
    x = syn.normal_f32((tokens, dim), seed=seed)
    x *= np.float32(4.0) ** syn.normal_f32((tokens, 1), seed=seed + 1).round()
    if tokens > 3:
        x[1] = 0.0
        x[2] = np.float32(3e-9) * syn.normal_f32((dim,), seed=seed + 2)
        x[3] = np.float32(-1.25)
    if tokens > 4 and dim >= 8:
        x[4, :8] = [127, -63.5, 0.5, 1.5, 2.5, -2.5, 0, 126.5]
        x[4, 8:] = 0
    return x.astype(np.float32)


def _int8_roundtrip(x):
    tokens, dim = x.shape
    q = torch.empty((tokens, dim), dtype=torch.int8, device="cuda")
    s = torch.empty((tokens,), dtype=torch.float32, device="cuda")
    out = torch.empty((tokens, dim), dtype=torch.float32, device="cuda")
    xd = _dev(x)
    qdl.kv_quant_int8(xd, tokens, dim, q, s)
    qdl.kv_dequant_int8(q, s, tokens, dim, out)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy(), out.cpu().numpy()


@pytest.mark.parametrize("tokens,dim", [(1, 4), (7, 128), (33, 64), (1000, 128), (5, 256), (9, 500),
                                        (3, 512), (17, 1000), (6, 2048)])
def test_kv_int8_bit_exact(tokens, dim):
    """warp-per-token kernels with 1, 2, 4 chunks per lane and the wide
    two-pass kernel (head_dim > 512), ragged last warp"""
    x = _values(tokens, dim, seed=tokens + dim)
    q, s, out = _int8_roundtrip(x)
    qo, so = oracle.kv_quant_int8(x)
    assert _bits_equal(s, so)
    assert _bits_equal(q, qo)
    assert _bits_equal(out, oracle.kv_dequant_int8(qo, so))


def _int4_roundtrip(x, group):
    tokens, dim = x.shape
    n = tokens * dim
    packed = torch.empty((n // 2,), dtype=torch.uint8, device="cuda")
    sc = torch.empty((n // group,), dtype=torch.float32, device="cuda")
    zr = torch.empty((n // group,), dtype=torch.float32, device="cuda")
    out = torch.empty((tokens, dim), dtype=torch.float32, device="cuda")
    qdl.kv_quant_int4(_dev(x), tokens, dim, group, packed, sc, zr)
    qdl.kv_dequant_int4(packed, sc, zr, tokens, dim, group, out)
    torch.cuda.synchronize()
    return packed.cpu().numpy(), sc.cpu().numpy(), zr.cpu().numpy(), out.cpu().numpy()


@pytest.mark.parametrize("tokens,dim,group", [(1, 8, 8), (4, 16, 16), (8, 32, 32), (16, 128, 64), (100, 128, 128),
                                              (64, 128, 256), (4, 8, 16), (10, 96, 24), (5, 1024, 512),
                                              (3, 40, 40), (333, 128, 128)])
def test_kv_int4_bit_exact(tokens, dim, group):
    """lane segments of 1..32 lanes per group (group 8..256), groups spanning
    two tokens, the wide kernel for other group sizes, ragged last warp"""
    x = _values(tokens, dim, seed=7 * tokens + dim)
    packed, sc, zr, out = _int4_roundtrip(x, group)
    po, so, zo = oracle.kv_quant_int4(x, group)
    assert _bits_equal(sc, so)
    assert _bits_equal(zr, zo)
    assert _bits_equal(packed, po)
    assert _bits_equal(out.reshape(-1), oracle.kv_dequant_int4(po, so, zo, tokens * dim, group))


def test_kv_full_size_bit_exact():
    """the benchmark's KV block: 32768 tokens x 128, int8 and INT4 group 128"""
    tokens, dim = 32768, 128
    x = syn.normal_f32((tokens, dim), seed=11)
    q, s, out = _int8_roundtrip(x)
    qo, so = oracle.kv_quant_int8(x)
    assert _bits_equal(s, so) and _bits_equal(q, qo)
    assert _bits_equal(out, oracle.kv_dequant_int8(qo, so))
    packed, sc, zr, out4 = _int4_roundtrip(x, 128)
    po, so4, zo = oracle.kv_quant_int4(x, 128)
    assert _bits_equal(sc, so4) and _bits_equal(zr, zo) and _bits_equal(packed, po)
    assert _bits_equal(out4.reshape(-1), oracle.kv_dequant_int4(po, so4, zo, tokens * dim, 128))
