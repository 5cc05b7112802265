"""The no-allocation decode projection, qdl_w8a8_proj_static.

Some callers cannot allocate device memory -- a plugin that its host
framework hands only input and output buffers, or a decode loop that may not
risk cudaMalloc's implicit synchronisation or an allocation failure.  For them
the library keeps its activation scratch in a built-in device array.  These
tests check, through the C ABI, that this entry point gives the same outputs
as qdl_w8a8_proj with caller scratch, on two calls in a row (the second with
different shapes, so a stale array from the first call would show), and that
oversize calls are refused before any device work.

This file is collected last so that a failure here never hides another test.
"""
import numpy as np
import pytest
import torch

import quantized_decode_linear_gb300 as qdl
from quantized_decode_linear_gb300 import synthetic as syn
from _gpu import TOL, bf16_dev, host, scratch, upload_weight


def _case(fmt, rows, k, sizes, seed):
    segs = [syn.fp8_weight(n, k, fmt, 0.02, seed + i) for i, n in enumerate(sizes)]
    x = syn.bf16_normal((rows, k), seed=seed + 50)
    return segs, x


def _both(fmt, rows, k, sizes, seed):
    segs, xb = _case(fmt, rows, k, sizes, seed)
    w, _keep = upload_weight(segs, fmt)
    x = bf16_dev(xb)
    ref = torch.empty((rows, w.n), device="cuda")
    q, s = scratch(rows, k, fmt)
    qdl.w8a8_proj(w, x, rows, ref, q, s)
    out = torch.full((rows, w.n), float("nan"), device="cuda")
    qdl.w8a8_proj_static(w, x, rows, out)
    torch.cuda.synchronize()
    return host(out), host(ref)


@pytest.mark.gpu
def test_static_scratch_matches_caller_scratch_twice():
    # first call: Block128, 3 segments, 16 rows; second: PerRow, more rows and a
    # longer K, so it overwrites more of the shared array than the first did
    calls = [(qdl.BLOCK128, 16, 1024, (512, 256, 200), 1),
             (qdl.PER_ROW, 40, 4096, (1024, 96), 2)]
    for fmt, rows, k, sizes, seed in calls:
        out, ref = _both(fmt, rows, k, sizes, seed)
        scale = np.abs(ref).max() + 1e-30
        assert np.all(np.isfinite(out))
        # both paths run the same kernels on the same codes; allow the parity
        # tolerance anyway
        assert np.max(np.abs(out - ref)) <= TOL * scale


@pytest.mark.gpu
def test_static_scratch_limit_is_refused():
    fmt, k = qdl.PER_ROW, 16384
    segs = [syn.fp8_weight(16, k, fmt, 0.02, 3)]
    w, _keep = upload_weight(segs, fmt)
    rows = 256  # 256 * 16384 codes plus scales exceed the 4 MiB array
    x = torch.zeros((rows, k), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((rows, 16), device="cuda")
    with pytest.raises(qdl.QdlError) as e:
        qdl.w8a8_proj_static(w, x, rows, out)
    assert e.value.status == 3 and "static scratch" in e.value.message
