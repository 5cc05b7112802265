"""GPU parity: weight preparation against the oracle, bit for bit.

FP8 weight quantisation per output row or per 128x128 block (scale =
absmax / 448, the scale layouts of w8a8_decode.rs enum W8a8Scale) from f32
and bf16 weights, and AWQ packing in the shift order of fused_int4_qkv.rs
(QKV_AWQ_SHIFTS).  Codes, scales and packed words must be identical; a
weight quantised on the GPU then feeds the decode projection."""
import numpy as np
import pytest
import torch

import oracle
import quantized_decode_linear_gb300 as qdl
from quantized_decode_linear_gb300 import synthetic as syn
from _gpu import bf16_dev, check_close, dev, f32_bits_equal, host, scratch, upload_weight

pytestmark = pytest.mark.gpu


def _bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _weight(n, ldw, seed, bf16):
    w = syn.normal_f32((n, ldw), seed=seed, std=0.02)
    if n >= 4:
        w[0] = 0.0
        w[1] = -0.0
        w[2] = 1e-6
        w[2, 3] = -2.5
        w[3] = np.float32(0.75)
    if bf16:
        bits = syn.to_bf16_bits(w)
        return bits, _bf16_to_f32(bits)
    return w, w


def _gpu_quant(fmt, w_host, bf16, n, k, ldw):
    wd = bf16_dev(w_host) if bf16 else dev(w_host)
    codes = torch.full((n, k), 0xAB, dtype=torch.uint8, device="cuda")
    shape = (n,) if fmt == qdl.PER_ROW else ((n + 127) // 128, k // 128)
    scales = torch.full(shape, float("nan"), device="cuda")
    qdl.fp8_weight_quant(fmt, wd, qdl.IN_BF16 if bf16 else qdl.IN_F32, ldw, n, k, codes, scales)
    torch.cuda.synchronize()
    return host(codes), host(scales)


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("n,k,ldw", [(1, 128, 128), (37, 384, 392), (200, 256, 256), (300, 1024, 1040),
                                     (129, 20480, 20480)])
def test_fp8_weight_quant_bit_exact(fmt, bf16, n, k, ldw):
    """rows of one and several 128-row blocks, ragged last block row, row
    strides beyond k, rows longer than the registers a thread keeps (20480),
    special rows (zeros, negative zeros, one large value over tiny ones, a
    constant row)"""
    w_host, w32 = _weight(n, ldw, seed=n + k, bf16=bf16)
    codes, scales = _gpu_quant(fmt, w_host, bf16, n, k, ldw)
    ref_codes, ref_scales = oracle.fp8_weight_quant(fmt, np.ascontiguousarray(w32[:, :k]))
    assert f32_bits_equal(scales, ref_scales)
    assert np.array_equal(codes, ref_codes)


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
def test_fp8_weight_quant_full_gateup(fmt):
    """the gate/up weight of the M-sweep workload: [2 x 14336, 8192] from bf16"""
    n, k = 28672, 8192
    w_bits = syn.bf16_normal((n, k), seed=9, std=0.015)
    codes, scales = _gpu_quant(fmt, w_bits, True, n, k, k)
    ref_codes, ref_scales = oracle.fp8_weight_quant(fmt, _bf16_to_f32(w_bits))
    assert f32_bits_equal(scales, ref_scales)
    assert np.array_equal(codes, ref_codes)


@pytest.mark.parametrize("k,n", [(1, 8), (16, 64), (37, 200), (4096, 4096), (4096, 1024)])
def test_awq_pack_bit_exact(k, n):
    """random bytes (the high nibble must be ignored) -> packed words"""
    rng = np.random.default_rng(k * 31 + n)
    nib = rng.integers(0, 256, size=(k, n), dtype=np.uint8)
    qw = torch.full((k, n // 8), -1, dtype=torch.int32, device="cuda")
    qdl.awq_pack(dev(nib), k, n, qw)
    torch.cuda.synchronize()
    assert np.array_equal(host(qw).view(np.uint32), oracle.awq_pack(nib & 0xF))


def test_quantised_weight_feeds_the_projection():
    """a bf16 QKV weight quantised on the GPU (Block128), then the decode
    projection on it: the same result as the oracle's GEMV on the oracle's
    quantisation of that weight"""
    fmt, k, sizes, rows = qdl.BLOCK128, 1024, [512, 128, 128], 8
    segs_dev, segs_host = [], []
    for i, n in enumerate(sizes):
        bits = syn.bf16_normal((n, k), seed=60 + i, std=0.02)
        codes, scales = _gpu_quant(fmt, bits, True, n, k, k)
        ref = oracle.fp8_weight_quant(fmt, _bf16_to_f32(bits))
        assert np.array_equal(codes, ref[0]) and f32_bits_equal(scales, ref[1])
        segs_host.append((codes, scales))
    w, _keep = upload_weight(segs_host, fmt)
    x = syn.bf16_normal((rows, k), seed=70)
    qo, so = oracle.act_quant(fmt, x, k)
    yo, bo = oracle.w8a8_gemv(fmt, qo, so, segs_host)
    q, s = scratch(rows, k, fmt)
    out = torch.full((rows, w.n), float("nan"), device="cuda")
    qdl.w8a8_proj(w, bf16_dev(x), rows, out, q, s)
    torch.cuda.synchronize()
    check_close(host(out), yo, bo, what="gpu-quantised weight")


def _boundary_values() -> np.ndarray:
    """f32 values at and around every E4M3 rounding decision in [-448, 448]:
    +-64 ulps about each grid point and each midpoint between neighbours,
    every in-range bf16 pattern, and random in-range bit patterns"""
    grid = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))  # 0 .. 448, codes 0x00..0x7E
    grid = np.unique(grid.astype(np.float64))
    mids = (grid[:-1] + grid[1:]) / 2.0
    centres = np.concatenate([grid, mids]).astype(np.float32).view(np.int32)
    offs = np.arange(-64, 65, dtype=np.int32)
    near = (centres[:, None] + offs[None, :]).reshape(-1)
    near = near[(near >= 0)].view(np.float32)
    bf = (np.arange(0, 1 << 16, dtype=np.uint32) << 16).view(np.float32)
    rnd = np.random.default_rng(123).integers(0, 0x43E00001, size=4 << 20, dtype=np.uint32).view(np.float32)
    v = np.concatenate([near, bf, rnd])
    v = v[np.isfinite(v) & (np.abs(v) <= 448.0)]
    return np.concatenate([v, -v]).astype(np.float32)


def test_hardware_e4m3_encoding_matches_oracle_at_every_rounding_boundary():
    """The device conversion (cvt.rn.satfinite.e4m3x2.f32, through the
    per-row weight quantiser with every row's absmax 448, so s = 1 and the
    codes are e4m3(v)) against the oracle's encoder written from the OCP
    definition"""
    v = _boundary_values()
    k = 8192
    per_row = k - 1
    rows = -(-v.size // per_row)
    w = np.zeros((rows, k), np.float32)
    w[:, 0] = 448.0
    flat = w[:, 1:].reshape(-1)
    flat[:v.size] = v
    w[:, 1:] = flat.reshape(rows, per_row)
    codes, scales = _gpu_quant(qdl.PER_ROW, w, False, rows, k, k)
    assert np.all(scales == 1.0)
    got = codes[:, 1:].reshape(-1)[:v.size]
    want = oracle.e4m3_encode(v)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (bad.size, v[bad[:5]], got[bad[:5]], want[bad[:5]])
