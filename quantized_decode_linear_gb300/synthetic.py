"""Seeded synthetic inputs for the quantized decode-time linear layer.

This module only draws random numbers and stores them in the layouts the
library expects.  It holds none of the layer's arithmetic (no activation
quantisation, no GEMV, no nibble unpacking) and is shared by the tests (which
feed the oracle) and the benchmark (which feeds the CUDA path).

Recipe (LLM-shaped decode workloads):

* activations: N(0, 1) drawn in float32 with numpy's PCG64 generator and
  rounded to bfloat16 (round to nearest even, by torch's dtype cast);
* FP8 weights: N(0, std) float32 rows, scaled per output row or per 128x128
  block by ``absmax / 448`` and cast to ``torch.float8_e4m3fn`` (a library cast;
  weight preparation is not part of the decode path, which receives the codes
  and scales as inputs);
* AWQ INT4: packed words of uniform random bits (so every nibble is uniform on
  0..15), scales U(0.001, 0.02), zeros uniform on 0..15 (integers by default,
  continuous U(0, 15) on request);
* KV-cache blocks: float32 N(0, 1) rows of head_dim values;
* weight preparation: bf16 weights N(0, std) to quantise, uniform 4-bit codes
  (one per byte) to pack.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

PER_ROW = 0
BLOCK128 = 1


def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def normal_f32(shape, seed: int, std: float = 1.0) -> np.ndarray:
    x = _rng(seed).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 (round to nearest even), returned as uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_normal(shape, seed: int, std: float = 1.0) -> np.ndarray:
    return to_bf16_bits(normal_f32(shape, seed, std))


def _fp8_cast(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def fp8_weight(n: int, k: int, fmt: int, std: float, seed: int, chunk_rows: int = 4096):
    """FP8 E4M3 weight [n, k] with f32 scales: [n] (PER_ROW) or
    [ceil(n/128), k/128] (BLOCK128).  Generated in row chunks to bound memory."""
    assert k % 128 == 0
    rng = _rng(seed)
    codes = np.empty((n, k), np.uint8)
    if fmt == PER_ROW:
        scales = np.empty((n,), np.float32)
    else:
        scales = np.empty(((n + 127) // 128, k // 128), np.float32)
    chunk_rows = max(128, (chunk_rows // 128) * 128)
    for r0 in range(0, n, chunk_rows):
        r1 = min(n, r0 + chunk_rows)
        w = rng.standard_normal((r1 - r0, k), dtype=np.float32)
        w *= np.float32(std)
        if fmt == PER_ROW:
            s = np.abs(w).max(axis=1) / np.float32(448.0)
            scales[r0:r1] = s
            div = np.where(s == 0, np.float32(1.0), s)[:, None]
        else:
            rows = r1 - r0
            pad = (-rows) % 128
            wp = np.pad(np.abs(w), ((0, pad), (0, 0))) if pad else np.abs(w)
            nb = wp.shape[0] // 128
            s = wp.reshape(nb, 128, k // 128, 128).max(axis=(1, 3)) / np.float32(448.0)
            scales[r0 // 128:r0 // 128 + nb] = s
            s_safe = np.where(s == 0, np.float32(1.0), s)
            div = np.repeat(np.repeat(s_safe, 128, axis=0)[:rows], 128, axis=1)
        codes[r0:r1] = _fp8_cast(w / div)
    return codes, scales


def int4_awq(k: int, n: int, group: int, seed: int, integer_zeros: bool = True):
    """AWQ INT4 weight for one projection: qweight uint32 [k, n/8], scales and
    zeros f32 [k/group, n]."""
    assert n % 8 == 0 and k % group == 0
    rng = _rng(seed)
    qw = rng.integers(0, 2**32, size=(k, n // 8), dtype=np.uint32)
    sc = rng.uniform(0.001, 0.02, size=(k // group, n)).astype(np.float32)
    if integer_zeros:
        zr = rng.integers(0, 16, size=(k // group, n)).astype(np.float32)
    else:
        zr = rng.uniform(0.0, 15.0, size=(k // group, n)).astype(np.float32)
    return qw, sc, zr


# ---------------------------------------------------------------------------
# Workloads (LLM decode shapes).  Seeds: activations seed, weight segment s at
# seed + 1 + s, INT4 projection p at seed + 10 + p.
# ---------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class W8A8Workload:
    name: str
    fmt: int
    k: int
    segments: tuple
    rows: tuple
    w_std: float
    silu: bool = False
    seed: int = 0

    @property
    def n(self) -> int:
        return int(sum(self.segments))


@dataclasses.dataclass(frozen=True)
class Int4Workload:
    name: str
    k: int
    nq: int
    nkv: int
    group: int
    rows: tuple
    seed: int = 0


@dataclasses.dataclass(frozen=True)
class KvWorkload:
    """A block of KV-cache rows (token x head) of head_dim values; group 0
    means per-token int8, otherwise per-group INT4."""
    name: str
    head_dim: int
    group: int
    rows: tuple
    seed: int = 0


@dataclasses.dataclass(frozen=True)
class WeightPrepWorkload:
    """Weight preparation: `prep` "fp8" quantises a bf16 weight [n, k] ~ N(0, w_std)
    to FP8 with the given scale layout; "awq" packs uniform 4-bit codes [k, n]."""
    name: str
    prep: str
    n: int
    k: int
    scale_format: int = BLOCK128
    w_std: float = 0.015
    rows: tuple = (1,)
    seed: int = 0


WORKLOADS = {
    "w8a8_perrow_m1_k1024_n1024": W8A8Workload(
        "w8a8_perrow_m1_k1024_n1024", PER_ROW, 1024, (1024,), (1,), 0.02),
    "w8a8_block128_qkv_m8_k4096_n4096+1024+1024": W8A8Workload(
        "w8a8_block128_qkv_m8_k4096_n4096+1024+1024", BLOCK128, 4096, (4096, 1024, 1024),
        (8,), 0.02),
    "w8a8_perrow_silu_down_m64_k14336_n4096": W8A8Workload(
        "w8a8_perrow_silu_down_m64_k14336_n4096", PER_ROW, 14336, (4096,), (64,), 0.02,
        silu=True),
    "int4_awq_qkv_k4096_nq4096_nkv1024_g128": Int4Workload(
        "int4_awq_qkv_k4096_nq4096_nkv1024_g128", 4096, 4096, 1024, 128, (1, 4, 16)),
    "w8a8_block128_gateup_k8192_n14336+14336": W8A8Workload(
        "w8a8_block128_gateup_k8192_n14336+14336", BLOCK128, 8192, (14336, 14336),
        (1, 2, 4, 8, 16, 32, 64, 128, 256), 0.015),
    "kv_int8_t32768_d128": KvWorkload("kv_int8_t32768_d128", 128, 0, (32768,)),
    "kv_int4_t32768_d128_g128": KvWorkload("kv_int4_t32768_d128_g128", 128, 128, (32768,)),
    "fp8_weight_quant_block128_bf16_n28672_k8192": WeightPrepWorkload(
        "fp8_weight_quant_block128_bf16_n28672_k8192", "fp8", 28672, 8192),
    "awq_pack_k4096_n6144": WeightPrepWorkload("awq_pack_k4096_n6144", "awq", 6144, 4096),
}

HEADLINE = "w8a8_block128_gateup_k8192_n14336+14336"


def w8a8_weights(wl: W8A8Workload):
    return [fp8_weight(n, wl.k, wl.fmt, wl.w_std, wl.seed + 1 + s)
            for s, n in enumerate(wl.segments)]


def w8a8_activations(wl: W8A8Workload, rows: int):
    """bf16 bits: x [rows, k], or for SiLU workloads one buffer [rows, 2k]
    holding gate (columns 0..k-1) then up (columns k..2k-1)."""
    width = 2 * wl.k if wl.silu else wl.k
    return bf16_normal((rows, width), wl.seed)


def int4_weights(wl: Int4Workload, integer_zeros: bool = True):
    ns = (wl.nq, wl.nkv, wl.nkv)
    return [int4_awq(wl.k, n, wl.group, wl.seed + 10 + p, integer_zeros)
            for p, n in enumerate(ns)]


def int4_activations(wl: Int4Workload, rows: int) -> np.ndarray:
    return normal_f32((rows, wl.k), wl.seed)


def kv_values(wl: KvWorkload, rows: int, copy: int = 0) -> np.ndarray:
    """K or V rows ~ N(0, 1), float32 [rows, head_dim]"""
    return normal_f32((rows, wl.head_dim), wl.seed + 100 + copy)


def prep_weight_bf16(wl: WeightPrepWorkload, rows: int | None = None) -> np.ndarray:
    """bf16 bits [rows or n, k] ~ N(0, w_std)"""
    return bf16_normal((rows or wl.n, wl.k), wl.seed + 1, wl.w_std)


def prep_codes(wl: WeightPrepWorkload, rows: int | None = None) -> np.ndarray:
    """uniform 4-bit codes, one per byte, [rows or k, n]"""
    return _rng(wl.seed + 2).integers(0, 16, size=(rows or wl.k, wl.n), dtype=np.uint8)
