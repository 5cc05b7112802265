"""GPU parity: AWQ INT4 fused QKV against the oracle (fused_int4_qkv.rs:
fused_int4_qkv_q/_k/_v, unpack_awq_qkv).  Outputs within 2e-3 * sum_k |x w|."""
import numpy as np
import pytest
import torch

import oracle
import quantized_decode_linear_gb300 as qdl
from quantized_decode_linear_gb300 import synthetic as syn
from _gpu import check_close, dev, host, u32_dev

pytestmark = pytest.mark.gpu


def _run(x, nq, nkv, group, ws):
    m, k = x.shape
    dqw = [u32_dev(w[0]) for w in ws]
    dsc = [dev(w[1]) for w in ws]
    dzr = [dev(w[2]) for w in ws]
    outs = [torch.full((m, n), float("nan"), device="cuda") for n in (nq, nkv, nkv)]
    qdl.int4_qkv_gemv(dev(x), m, k, nq, nkv, group, dqw, dsc, dzr, outs)
    torch.cuda.synchronize()
    return [host(o) for o in outs]


@pytest.mark.parametrize("m", [1, 4, 8, 9, 16, 17, 33])
@pytest.mark.parametrize("k,nq,nkv,group", [(128, 128, 128, 128), (256, 136, 8, 32),
                                            (512, 384, 256, 16), (1024, 1000, 200, 128),
                                            (4096, 256, 128, 64)])
def test_int4_small(m, k, nq, nkv, group):
    x = syn.normal_f32((m, k), seed=m + k)
    ws = [syn.int4_awq(k, n, group, seed=p + nq) for p, n in enumerate((nq, nkv, nkv))]
    outs = _run(x, nq, nkv, group, ws)
    ref, bound = oracle.int4_qkv(x, nq, nkv, group, [w[0] for w in ws], [w[1] for w in ws],
                                 [w[2] for w in ws])
    for p in range(3):
        check_close(outs[p], ref[p], bound[p], what=f"proj {p}")


@pytest.mark.parametrize("m", [1, 2, 9, 16, 17, 32, 33, 70])
@pytest.mark.parametrize("k,nq,nkv", [(128, 96, 32), (256, 128, 128), (2048, 640, 160), (1024, 4096, 1024),
                                      (16384, 128, 32)])
def test_int4_tensor_core_path(m, k, nq, nkv):
    """group 128 and widths multiple of 32: the tcgen05 kernel (ragged last
    128-column tiles, K ranges from one 64-row unit to more units per CTA than
    its code ring holds, several passes of 32 rows)"""
    group = 128
    x = syn.normal_f32((m, k), seed=2 * m + k)
    ws = [syn.int4_awq(k, n, group, seed=p + 3 * nq) for p, n in enumerate((nq, nkv, nkv))]
    outs = _run(x, nq, nkv, group, ws)
    ref, bound = oracle.int4_qkv(x, nq, nkv, group, [w[0] for w in ws], [w[1] for w in ws],
                                 [w[2] for w in ws])
    for p in range(3):
        check_close(outs[p], ref[p], bound[p], what=f"proj {p}")


@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("k,nq,nkv,group", [(128, 32, 32, 128), (1040, 96, 32, 16), (512, 288, 64, 32),
                                            (4096, 512, 256, 64), (2048, 640, 160, 128), (8192, 32, 64, 128),
                                            (16, 64, 32, 16), (48, 96, 64, 16), (960, 256, 96, 48),
                                            (4096, 4096, 1024, 128)])
def test_int4_cuda_core_path(m, k, nq, nkv, group):
    """widths multiple of 32 with 1-4 rows, and 5-8 rows with group != 128:
    the CUDA-core stream-K kernel (ragged 256-column tiles, K below one 32-row
    stage and ending inside one, groups that end in the middle of a stage (16,
    48), ranges over several tiles, every token-count variant); 5-8 rows with
    group 128 take the tcgen05 kernel"""
    x = syn.normal_f32((m, k), seed=5 * m + k)
    ws = [syn.int4_awq(k, n, group, seed=p + 7 * nq) for p, n in enumerate((nq, nkv, nkv))]
    outs = _run(x, nq, nkv, group, ws)
    ref, bound = oracle.int4_qkv(x, nq, nkv, group, [w[0] for w in ws], [w[1] for w in ws],
                                 [w[2] for w in ws])
    for p in range(3):
        check_close(outs[p], ref[p], bound[p], what=f"proj {p}")


def test_int4_continuous_zeros():
    m, k, nq, nkv, group = 5, 1024, 512, 128, 128
    x = syn.normal_f32((m, k), seed=3)
    ws = [syn.int4_awq(k, n, group, seed=20 + p, integer_zeros=False)
          for p, n in enumerate((nq, nkv, nkv))]
    outs = _run(x, nq, nkv, group, ws)
    ref, bound = oracle.int4_qkv(x, nq, nkv, group, [w[0] for w in ws], [w[1] for w in ws],
                                 [w[2] for w in ws])
    for p in range(3):
        check_close(outs[p], ref[p], bound[p], what=f"proj {p}")


@pytest.mark.parametrize("m", [1, 4, 16])
def test_int4_full_qkv_k4096(m):
    wl = syn.WORKLOADS["int4_awq_qkv_k4096_nq4096_nkv1024_g128"]
    ws = syn.int4_weights(wl)
    x = syn.int4_activations(wl, m)
    outs = _run(x, wl.nq, wl.nkv, wl.group, ws)
    ref, bound = oracle.int4_qkv(x, wl.nq, wl.nkv, wl.group, [w[0] for w in ws],
                                 [w[1] for w in ws], [w[2] for w in ws])
    for p in range(3):
        check_close(outs[p], ref[p], bound[p], what=f"proj {p} m={m}")


@pytest.mark.parametrize("m", [1, 3])
def test_int4_cuda_core_unaligned_outputs(m):
    """outputs that start 4 bytes past a 16-byte boundary: the CUDA-core
    kernel adds its totals with scalar atomics instead of 4-wide ones"""
    k, nq, nkv, group = 1024, 512, 256, 64
    x = syn.normal_f32((m, k), seed=40 + m)
    ws = [syn.int4_awq(k, n, group, seed=41 + p) for p, n in enumerate((nq, nkv, nkv))]
    bufs = [torch.full((m * n + 1,), float("nan"), device="cuda") for n in (nq, nkv, nkv)]
    outs = [b[1:].view(m, n) for b, n in zip(bufs, (nq, nkv, nkv))]
    assert all(o.data_ptr() % 16 == 4 for o in outs)
    qdl.int4_qkv_gemv(dev(x), m, k, nq, nkv, group, [u32_dev(w[0]) for w in ws], [dev(w[1]) for w in ws],
                      [dev(w[2]) for w in ws], outs)
    torch.cuda.synchronize()
    ref, bound = oracle.int4_qkv(x, nq, nkv, group, [w[0] for w in ws], [w[1] for w in ws],
                                 [w[2] for w in ws])
    for p in range(3):
        check_close(host(outs[p]), ref[p], bound[p], what=f"proj {p}")


def test_int4_cuda_core_many_tiles():
    """K = 16 (one stage per tile) over 576 tiles: more CTAs than SMs, since
    each CTA's range may touch at most four tiles"""
    m, k, nq, nkv, group = 2, 16, 131072, 8192, 16
    x = syn.normal_f32((m, k), seed=50)
    ws = [syn.int4_awq(k, n, group, seed=51 + p) for p, n in enumerate((nq, nkv, nkv))]
    outs = _run(x, nq, nkv, group, ws)
    ref, bound = oracle.int4_qkv(x, nq, nkv, group, [w[0] for w in ws], [w[1] for w in ws],
                                 [w[2] for w in ws])
    for p in range(3):
        check_close(outs[p], ref[p], bound[p], what=f"proj {p}")
