"""Guard bands around every output: each kernel family writes only inside its
output (the tensors below sit in the middle of a larger buffer whose bands
hold a sentinel that must survive the call), for the W8A8 projections with
f32 and bf16 output and ragged widths, the AWQ INT4 kernels (CUDA-core and
tcgen05 paths, ragged tiles), the KV-cache codecs and the weight
preparation."""
import numpy as np
import pytest
import torch

import oracle
import quantized_decode_linear_gb300 as qdl
from quantized_decode_linear_gb300 import synthetic as syn
from _gpu import bf16_dev, check_close, dev, host, scratch, u32_dev, upload_weight

pytestmark = pytest.mark.gpu

BAND = 4096  # bytes of guard band on each side


def _guarded(shape, dtype, fill):
    """a tensor of `shape` in the middle of a buffer with BAND-byte bands
    holding `fill`; returns (view, buffer, band elements)"""
    el = torch.tensor([], dtype=dtype).element_size()
    band = BAND // el
    n = int(np.prod(shape))
    buf = torch.full((band + n + band,), fill, dtype=dtype, device="cuda")
    return buf[band:band + n].view(*shape), buf, band


def _bands_intact(buf, band, fill):
    b = torch.cat([buf[:band], buf[-band:]]).cpu()
    if b.dtype.is_floating_point and np.isnan(fill):
        return bool(torch.isnan(b.float()).all())
    return bool((b == fill).all())


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
@pytest.mark.parametrize("out_dtype", [qdl.OUT_F32, qdl.OUT_BF16])
@pytest.mark.parametrize("rows", [1, 8, 40, 300])
def test_w8a8_projection_stays_inside_its_output(fmt, out_dtype, rows):
    k = 512
    sizes = [256, 128, 72] if fmt == qdl.PER_ROW else [256, 128, 200]
    segs = [syn.fp8_weight(n, k, fmt, 0.02, seed=i) for i, n in enumerate(sizes)]
    w, _keep = upload_weight(segs, fmt)
    x = syn.bf16_normal((rows, k), seed=rows)
    tdt = torch.float32 if out_dtype == qdl.OUT_F32 else torch.bfloat16
    out, buf, band = _guarded((rows, w.n), tdt, float("nan"))
    q, s = scratch(min(rows, 256), k, fmt)
    qdl.w8a8_proj(w, bf16_dev(x), rows, out, q, s, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert _bands_intact(buf, band, float("nan"))
    assert not torch.isnan(out.float()).any()


@pytest.mark.parametrize("m", [1, 3, 8, 20])
def test_int4_stays_inside_its_outputs(m):
    k, nq, nkv, group = 1024, 288, 96, 128  # ragged 256- and 128-column tiles
    x = syn.normal_f32((m, k), seed=m)
    ws = [syn.int4_awq(k, n, group, seed=p + 1) for p, n in enumerate((nq, nkv, nkv))]
    guarded = [_guarded((m, n), torch.float32, float("nan")) for n in (nq, nkv, nkv)]
    outs = [g[0] for g in guarded]
    qdl.int4_qkv_gemv(dev(x), m, k, nq, nkv, group, [u32_dev(w[0]) for w in ws], [dev(w[1]) for w in ws],
                      [dev(w[2]) for w in ws], outs)
    torch.cuda.synchronize()
    for o, buf, band in guarded:
        assert _bands_intact(buf, band, float("nan"))
        assert not torch.isnan(o).any()
    ref, bound = oracle.int4_qkv(x, nq, nkv, group, [w[0] for w in ws], [w[1] for w in ws], [w[2] for w in ws])
    for p in range(3):
        check_close(host(outs[p]), ref[p], bound[p], what=f"proj {p}")


def test_kv_codecs_stay_inside_their_outputs():
    tokens, dim, group = 37, 128, 64
    x = dev(syn.normal_f32((tokens, dim), seed=4))
    q, qb, qband = _guarded((tokens, dim), torch.int8, 0x5A)
    s, sb, sband = _guarded((tokens,), torch.float32, float("nan"))
    qdl.kv_quant_int8(x, tokens, dim, q, s)
    out, ob, oband = _guarded((tokens, dim), torch.float32, float("nan"))
    qdl.kv_dequant_int8(q, s, tokens, dim, out)
    n = tokens * dim
    p4, pb, pband = _guarded((n // 2,), torch.uint8, 0xA5)
    s4, s4b, s4band = _guarded((n // group,), torch.float32, float("nan"))
    z4, z4b, z4band = _guarded((n // group,), torch.float32, float("nan"))
    qdl.kv_quant_int4(x, tokens, dim, group, p4, s4, z4)
    o4, o4b, o4band = _guarded((tokens, dim), torch.float32, float("nan"))
    qdl.kv_dequant_int4(p4, s4, z4, tokens, dim, group, o4)
    torch.cuda.synchronize()
    assert _bands_intact(qb, qband, 0x5A) and _bands_intact(pb, pband, 0xA5)
    for b, band in ((sb, sband), (ob, oband), (s4b, s4band), (z4b, z4band), (o4b, o4band)):
        assert _bands_intact(b, band, float("nan"))


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
def test_weight_preparation_stays_inside_its_outputs(fmt):
    n, k = 200, 384
    w = syn.bf16_normal((n, k), seed=5, std=0.02)
    codes, cb, cband = _guarded((n, k), torch.uint8, 0x77)
    shape = (n,) if fmt == qdl.PER_ROW else ((n + 127) // 128, k // 128)
    scales, sb, sband = _guarded(shape, torch.float32, float("nan"))
    qdl.fp8_weight_quant(fmt, bf16_dev(w), qdl.IN_BF16, k, n, k, codes, scales)
    nib = np.random.default_rng(6).integers(0, 16, size=(24, 72), dtype=np.uint8)
    qw, qb, qband = _guarded((24, 9), torch.int32, -7)
    qdl.awq_pack(dev(nib), 24, 72, qw)
    torch.cuda.synchronize()
    assert _bands_intact(cb, cband, 0x77) and _bands_intact(sb, sband, float("nan"))
    assert _bands_intact(qb, qband, -7)
    assert np.array_equal(host(qw).view(np.uint32), oracle.awq_pack(nib))
