"""Failure detection without a GPU fault: the GEMV's device-side waits are
bounded.  The self-test entry point withholds one pipeline stage, so the
kernel's waits run out after a short limit; the kernel records the timeout and
returns, the host reads QDL_ERR_DEVICE_TIMEOUT, and the context stays usable
(a normal call afterwards is still correct)."""
import numpy as np
import pytest
import torch

import oracle
import quantized_decode_linear_gb300 as qdl
from quantized_decode_linear_gb300 import synthetic as syn
from _gpu import check_close, dev, host, upload_weight

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,k", [(4, 1024), (12, 512)])
def test_bounded_wait_times_out_and_context_survives(rows, k):
    fmt = qdl.BLOCK128
    segs = [syn.fp8_weight(n, k, fmt, 0.02, 30 + i) for i, n in enumerate((256, 128))]
    w, _keep = upload_weight(segs, fmt)
    x = syn.bf16_normal((rows, k), seed=31)
    qo, so = oracle.act_quant(fmt, x, k)
    q, s = dev(qo), dev(so)
    out = torch.empty((rows, w.n), device="cuda")
    status = qdl.selftest_bounded_wait(w, q, s, rows, out, limit_us=20000)
    assert status == 5, qdl.last_error()
    assert "gave up" in qdl.last_error()
    qdl.check_device_fault()  # the fault word was cleared by the self-test
    qdl.w8a8_gemv(w, q, s, rows, out)
    qdl.check_device_fault()
    torch.cuda.synchronize()
    yo, bo = oracle.w8a8_gemv(fmt, qo, so, segs)
    check_close(host(out), yo, bo)
