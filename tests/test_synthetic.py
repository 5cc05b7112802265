"""Pins of the seeded input recipe (quantized_decode_linear_gb300/synthetic.py):
every input is reproducible from its seed, has the stated distribution and
layout, and every workload's name matches its shapes.  The generator is
checked here against independent statements of the recipe (integer
round-to-nearest-even for bf16, the E4M3 grid for the weight codes), not
against itself."""
import re

import numpy as np
import pytest
import torch

from quantized_decode_linear_gb300 import synthetic as syn


def _bf16_rne_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bits by integer round to nearest, ties to even
    (finite inputs)"""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _e4m3_values() -> np.ndarray:
    """all finite non-negative E4M3 values, from the format's definition"""
    vals = [m * 2.0**-9 for m in range(8)]  # subnormals (and zero)
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:
                continue  # NaN
            vals.append((1 + m / 8) * 2.0 ** (e - 7))
    return np.array(sorted(vals))


def test_seeds_reproduce_and_differ():
    a = syn.bf16_normal((4, 256), seed=3)
    assert np.array_equal(a, syn.bf16_normal((4, 256), seed=3))
    assert not np.array_equal(a, syn.bf16_normal((4, 256), seed=4))
    w1 = syn.fp8_weight(256, 256, syn.BLOCK128, 0.02, seed=5)
    w2 = syn.fp8_weight(256, 256, syn.BLOCK128, 0.02, seed=5)
    assert all(np.array_equal(p, q) for p, q in zip(w1, w2))


def test_activations_are_bf16_rne_of_f32_normals():
    x = syn.normal_f32((64, 512), seed=11)
    assert x.dtype == np.float32
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1.0) < 0.02
    assert np.array_equal(syn.bf16_normal((64, 512), seed=11), _bf16_rne_bits(x))
    # ties: a value halfway between two bf16 numbers goes to the even one
    ties = np.array([0x3F808000, 0x3F818000, 0xBF808000], np.uint32).view(np.float32)
    assert list(syn.to_bf16_bits(ties)) == [0x3F80, 0x3F82, 0xBF80]


@pytest.mark.parametrize("fmt", [syn.PER_ROW, syn.BLOCK128])
def test_fp8_weights_follow_the_absmax_448_recipe(fmt):
    n, k, std, seed = 300, 384, 0.02, 21
    codes, scales = syn.fp8_weight(n, k, fmt, std, seed)
    assert codes.shape == (n, k) and codes.dtype == np.uint8
    w = np.random.default_rng(seed).standard_normal((n, k), dtype=np.float32) * np.float32(std)
    if fmt == syn.PER_ROW:
        assert scales.shape == (n,)
        s_full = np.repeat(scales[:, None], k, axis=1)
        absmax = np.abs(w).max(axis=1)
        assert np.array_equal(scales, absmax / np.float32(448.0))
    else:
        assert scales.shape == ((n + 127) // 128, k // 128)
        s_full = np.repeat(np.repeat(scales, 128, axis=0)[:n], 128, axis=1)
        for b in range(scales.shape[0]):
            for g in range(scales.shape[1]):
                blk = np.abs(w[128 * b:128 * b + 128, 128 * g:128 * g + 128])
                assert scales[b, g] == blk.max() / np.float32(448.0)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    # each code is the E4M3 value nearest w / s (within half a grid step)
    v = w.astype(np.float64) / s_full
    grid = _e4m3_values()
    i = np.clip(np.searchsorted(grid, np.abs(v)), 1, len(grid) - 1)
    step = grid[i] - grid[i - 1]
    assert np.all(np.abs(dec - v) <= step / 2 * (1 + 1e-6))
    # the largest magnitude of every row or block codes to +-448
    assert np.all(np.abs(dec).max(axis=1 if fmt == syn.PER_ROW else None) == 448.0)


def test_awq_weights_recipe():
    qw, sc, zr = syn.int4_awq(256, 512, 128, seed=7)
    assert qw.shape == (256, 64) and qw.dtype == np.uint32
    assert sc.shape == zr.shape == (2, 512)
    nib = np.stack([(qw >> (4 * p)) & 0xF for p in range(8)]).ravel()
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.8 * nib.size / 16 and counts.max() < 1.2 * nib.size / 16
    assert sc.min() >= 0.001 and sc.max() < 0.02
    assert np.array_equal(zr, np.round(zr)) and zr.min() >= 0 and zr.max() <= 15
    _, _, zc = syn.int4_awq(256, 512, 128, seed=7, integer_zeros=False)
    assert not np.array_equal(zc, np.round(zc)) and zc.min() >= 0 and zc.max() < 15


def test_workload_seeds():
    """activations at the workload seed, INT4 projection p at seed + 10 + p,
    W8A8 segment s at seed + 1 + s"""
    small = syn.Int4Workload("small", 256, 64, 32, 128, (1,), seed=4)
    ws = syn.int4_weights(small)
    for p, n in enumerate((64, 32, 32)):
        ref = syn.int4_awq(256, n, 128, seed=4 + 10 + p)
        assert all(np.array_equal(a, b) for a, b in zip(ws[p], ref))
    assert np.array_equal(syn.int4_activations(small, 3), syn.normal_f32((3, 256), 4))
    w8 = syn.W8A8Workload("small", syn.PER_ROW, 256, (32, 16), (1,), 0.02, seed=6)
    for s_, (c, sc) in enumerate(syn.w8a8_weights(w8)):
        rc, rs = syn.fp8_weight(w8.segments[s_], 256, syn.PER_ROW, 0.02, 6 + 1 + s_)
        assert np.array_equal(c, rc) and np.array_equal(sc, rs)
    assert np.array_equal(syn.w8a8_activations(w8, 2), syn.bf16_normal((2, 256), 6))


def test_workload_names_match_shapes():
    for name, wl in syn.WORKLOADS.items():
        assert wl.name == name
        if isinstance(wl, syn.W8A8Workload):
            assert f"_k{wl.k}_" in name
            assert "+".join(str(n) for n in wl.segments) in name
            assert ("block128" in name) == (wl.fmt == syn.BLOCK128)
            assert ("silu" in name) == wl.silu
            m = re.search(r"_m(\d+)_", name)
            if m:
                assert wl.rows == (int(m.group(1)),)
            # non-last segments keep the format's row alignment
            align = 16 if wl.fmt == syn.PER_ROW else 128
            assert all(n % align == 0 for n in wl.segments[:-1])
        elif isinstance(wl, syn.Int4Workload):
            assert f"_k{wl.k}_nq{wl.nq}_nkv{wl.nkv}_g{wl.group}" in name
        elif isinstance(wl, syn.KvWorkload):
            assert f"_t{wl.rows[0]}_d{wl.head_dim}" in name
            assert ("int4" in name) == (wl.group > 0)
        else:
            assert f"_n{wl.n}_k{wl.k}" in name or f"_k{wl.k}_n{wl.n}" in name
    assert syn.HEADLINE in syn.WORKLOADS


def test_silu_activation_buffer_holds_gate_then_up():
    wl = syn.WORKLOADS["w8a8_perrow_silu_down_m64_k14336_n4096"]
    x = syn.w8a8_activations(wl, 2)
    assert x.shape == (2, 2 * wl.k) and x.dtype == np.uint16
    assert np.array_equal(x, syn.bf16_normal((2, 2 * wl.k), wl.seed))
