"""The no-allocation decode projection, qdl_w8a8_proj_static.

Some callers cannot allocate device memory -- a plugin that its host
framework hands only input and output buffers, or a decode loop that may not
risk cudaMalloc's implicit synchronisation or an allocation failure.  For them
the library keeps its activation scratch in a built-in device array.

These tests call that entry point through the C ABI twice in a row, first a
large call and then a smaller one of the other scale format, and check each
output element against the oracle within the GEMV tolerance
(2e-3 * sum_k |x_hat w_hat|, plus bf16 rounding for bf16 output).  The codes
the static array holds are checked indirectly but exactly: the output must
equal, bit for bit, the deterministic qdl_w8a8_gemv run on the oracle's own
codes and scales, which holds only if the array held exactly those codes and
scales.  Oversize calls must be refused before any device work.

This file is collected last so that a failure here never hides another test.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_decode_linear_gb300 as qdl
from quantized_decode_linear_gb300 import synthetic as syn
from _gpu import BF16_REL, bf16_dev, check_close, dev, f32_bits_equal, host, upload_weight

# (format, rows, k, ldx, segment sizes, out dtype, seed).  The first call
# writes more of the shared array than the second, which uses the other
# scale layout, so a second call reading anything it did not write itself
# (a wrong offset, a stale scale) would read the first call's bytes.
CALLS = [
    (qdl.PER_ROW, 40, 4096, 4096 + 64, (1024, 96), qdl.OUT_F32, 2),
    (qdl.BLOCK128, 16, 1024, 1024, (512, 256, 200), qdl.OUT_BF16, 1),
]


def _static_call(fmt, rows, k, ldx, sizes, out_dtype, seed):
    segs = [syn.fp8_weight(n, k, fmt, 0.02, seed + i) for i, n in enumerate(sizes)]
    xb = syn.bf16_normal((rows, ldx), seed=seed + 50)
    w, keep = upload_weight(segs, fmt)
    tdt = torch.bfloat16 if out_dtype == qdl.OUT_BF16 else torch.float32
    out = torch.full((rows, w.n), float("nan"), device="cuda", dtype=tdt)
    qdl.w8a8_proj_static(w, bf16_dev(xb), rows, out, out_dtype=out_dtype, ldx=ldx)
    torch.cuda.synchronize()
    return segs, xb, w, keep, host(out.float())


def _check(call, segs, xb, w, out):
    fmt, rows, k, ldx, sizes, out_dtype, seed = call
    qo, so = oracle.act_quant(fmt, xb, k)
    yo, bo = oracle.w8a8_gemv(fmt, qo, so, segs)
    bf16 = out_dtype == qdl.OUT_BF16
    assert np.all(np.isfinite(out))
    check_close(out, yo, bo, extra_rel=BF16_REL if bf16 else 0.0, what=f"static fmt={fmt} rows={rows}")
    # the same GEMV on the oracle's codes and scales (fixed-order reduction,
    # so reproducible bit for bit) must give exactly the same output
    tdt = torch.bfloat16 if bf16 else torch.float32
    ref = torch.full((rows, w.n), float("nan"), device="cuda", dtype=tdt)
    qdl.w8a8_gemv(w, dev(qo), dev(so if fmt == qdl.BLOCK128 else so[:, None]), rows, ref, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert f32_bits_equal(out, host(ref.float())), f"static fmt={fmt}: output differs from the GEMV on the oracle codes"


@pytest.mark.gpu
def test_static_scratch_against_the_oracle_twice():
    results = [(c, _static_call(*c)) for c in CALLS]  # two calls in a row, no host check between
    for call, (segs, xb, w, _keep, out) in results:
        _check(call, segs, xb, w, out)
    # and once more in the other order, each checked straight after its call
    for call in reversed(CALLS):
        segs, xb, w, _keep, out = _static_call(*call)
        _check(call, segs, xb, w, out)


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
