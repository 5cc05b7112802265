"""Back-to-back calls with programmatic launch overlap.

The library's kernels start early (before the previous kernel finishes) to
stream their weights, and wait for the previous kernel only before they read
activations or write scratch and outputs.  These tests issue calls
back-to-back on one stream with no host synchronisation in between, sharing
the activation scratch: if any kernel touched shared data before its wait, an
earlier call's output would be computed from a later call's codes and miss the
oracle.  Also checks the launch plan that qdl_w8a8_plan reports."""
import numpy as np
import pytest
import torch

import oracle
import quantized_decode_linear_gb300 as qdl
from quantized_decode_linear_gb300 import synthetic as syn
from _gpu import bf16_dev, check_close, host, upload_weight

pytestmark = pytest.mark.gpu


def test_chain_of_projections_sharing_scratch():
    # alternating formats, widths and row counts, so several kernel variants
    # follow one another
    cases = [(qdl.BLOCK128, 8, 1024, (512, 256)), (qdl.PER_ROW, 4, 512, (384,)),
             (qdl.BLOCK128, 40, 512, (256, 128, 100)), (qdl.PER_ROW, 16, 1024, (256, 64)),
             (qdl.BLOCK128, 1, 2048, (1024,)), (qdl.BLOCK128, 130, 256, (256,))]
    kmax = max(c[2] for c in cases)
    rmax = max(c[1] for c in cases)
    q = torch.empty((rmax, kmax), dtype=torch.uint8, device="cuda")
    s = torch.empty((rmax, kmax // 128), dtype=torch.float32, device="cuda")
    keep, outs, refs = [], [], []
    for i, (fmt, rows, k, sizes) in enumerate(cases):
        segs = [syn.fp8_weight(n, k, fmt, 0.02, 100 * i + j) for j, n in enumerate(sizes)]
        w, dsegs = upload_weight(segs, fmt)
        xb = syn.bf16_normal((rows, k), seed=7 * i)
        x = bf16_dev(xb)
        out = torch.empty((rows, w.n), device="cuda")
        keep += [w, dsegs, x]
        outs.append(out)
        qo, so = oracle.act_quant(fmt, xb, k)
        refs.append(oracle.w8a8_gemv(fmt, qo, so, segs))
    torch.cuda.synchronize()
    for rep in range(3):
        for i, (fmt, rows, k, sizes) in enumerate(cases):
            w, x, out = keep[3 * i], keep[3 * i + 2], outs[i]
            qdl.w8a8_proj(w, x, rows, out, q, s)  # the same scratch for every call
        torch.cuda.synchronize()
        for i in range(len(cases)):
            check_close(host(outs[i]), refs[i][0], refs[i][1], what=f"call {i} repeat {rep}")


def test_chain_of_gemvs_writing_one_output():
    fmt, rows, k = qdl.BLOCK128, 8, 1024
    weights = []
    for i in range(4):
        segs = [syn.fp8_weight(768, k, fmt, 0.02, 50 + i)]
        weights.append((segs, *upload_weight(segs, fmt)))
    xb = syn.bf16_normal((rows, k), seed=3)
    qo, so = oracle.act_quant(fmt, xb, k)
    q = torch.from_numpy(qo).cuda()
    s = torch.from_numpy(so).cuda()
    out = torch.empty((rows, 768), device="cuda")
    for _ in range(5):
        for segs, w, _d in weights:
            qdl.w8a8_gemv(w, q, s, rows, out)  # the last call's result must win
    torch.cuda.synchronize()
    yo, bo = oracle.w8a8_gemv(fmt, qo, so, weights[-1][0])
    check_close(host(out), yo, bo)


@pytest.mark.parametrize("fmt,n,k,rows", [(qdl.BLOCK128, 6144, 4096, 8), (qdl.PER_ROW, 1024, 1024, 1),
                                          (qdl.BLOCK128, 28672, 8192, 256), (qdl.PER_ROW, 4096, 14336, 64),
                                          (qdl.BLOCK128, 28672, 8192, 64), (qdl.BLOCK128, 6144, 4096, 20)])
def test_plan_is_consistent(fmt, n, k, rows):
    codes = torch.zeros((n, k), dtype=torch.uint8, device="cuda")
    scale = torch.ones(((n + 127) // 128 * (k // 128)) if fmt == qdl.BLOCK128 else n, device="cuda")
    w = qdl.w8a8_weight_init([(codes, scale)], fmt)
    p = qdl.w8a8_plan(w, rows)
    assert p["kernel"] == 0 and p["mma_n"] >= rows and p["mma_n"] in (16, 32, 64, 128, 256)
    assert p["tiles"] == (n + 127) // 128
    assert 1 <= p["split_k"] <= min(8, k // 128)
    assert p["stages"] >= 3 and p["threads"] % 32 == 0 and p["smem_bytes"] <= 232448
    assert p["resident_clusters"] >= 1
    # the quantiser, then the GEMV
    assert p["proj_launches"] == 2
    # the f32 projection accumulates when K is split or Block128 runs stream-K
    streamk = fmt == qdl.BLOCK128 and 16 < rows <= 128
    # (the 256-token bucket may split K only when its ranks add atomically, so
    # the projection can accumulate where the plain GEMV's plan has no split)
    must = p["split_k"] > 1 or streamk
    assert p["proj_accumulates"] in ((1,) if must else (0, 1))
    if p["proj_accumulates"] and not must:
        assert fmt == qdl.BLOCK128 and rows > 128
    assert p["proj_streamk"] == (1 if streamk else 0)
