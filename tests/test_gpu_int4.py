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


@pytest.mark.parametrize("m", [1, 2, 3, 4])
@pytest.mark.parametrize("k,nq,nkv,group", [(128, 32, 32, 128), (1040, 96, 32, 16), (512, 288, 64, 32),
                                            (4096, 512, 256, 64), (2048, 640, 160, 128), (8192, 32, 64, 128)])
def test_int4_cuda_core_path(m, k, nq, nkv, group):
    """widths multiple of 32 with 1-4 rows and group != 128: the CUDA-core
    kernel (ragged 256-column tiles, K not a multiple of its 64-row stage,
    groups 16..64, split-K clusters up to 8); the group-128 cases here cover
    the tcgen05 kernel's small-row passes"""
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
