"""Helpers shared by the GPU parity tests: device upload, oracle comparison and
the parity tolerance.  Imports the oracle (tests only)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import quantized_decode_linear_gb300 as qdl
from quantized_decode_linear_gb300 import synthetic as syn

# GEMV tolerance per output element: |y - y_ref| <= TOL * sum_k |x_hat w_hat|
TOL = 2e-3
# bf16 output adds its own rounding (unit roundoff 2^-8 relative)
BF16_REL = 2.0**-8


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def u32_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def f32_bits_equal(a: np.ndarray, b: np.ndarray) -> bool:
    return np.array_equal(np.ascontiguousarray(a, np.float32).view(np.uint32),
                          np.ascontiguousarray(b, np.float32).view(np.uint32))


def scratch(rows: int, k: int, fmt: int):
    q = torch.empty((rows, k), dtype=torch.uint8, device="cuda")
    spr = 1 if fmt == qdl.PER_ROW else k // 128
    s = torch.empty((rows, spr), dtype=torch.float32, device="cuda")
    return q, s


def upload_weight(segments, fmt: int):
    """segments: list of (codes, scales) numpy -> (W8A8Weight, device tensors)"""
    dsegs = [(dev(c), dev(s)) for c, s in segments]
    return qdl.w8a8_weight_init(dsegs, fmt), dsegs


def check_close(y: np.ndarray, ref: np.ndarray, bound: np.ndarray, extra_rel: float = 0.0, what=""):
    err = np.abs(y.astype(np.float64) - ref)
    lim = TOL * bound + extra_rel * np.abs(ref) + 1e-30
    bad = err > lim
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {tuple(i)}: "
                             f"got {y[tuple(i)]}, want {ref[tuple(i)]}, bound {bound[tuple(i)]}")
    return float((err / (bound + 1e-30)).max())
