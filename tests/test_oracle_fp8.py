"""Pins for the oracle's FP8 E4M3 codec (OCP OFP8 E4M3, RNE, satfinite).

The oracle is checked against things other than itself: hand-computed cases,
torch's float8_e4m3fn dtype (a library decode and a library round-to-nearest
cast), and a brute-force nearest-value search over the 127 finite non-negative
grid values taken from the library decode.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lib_grid():
    """decode of codes 0..126 by torch (library), float64"""
    codes = torch.arange(0, 127, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _brute_encode(v: np.ndarray) -> np.ndarray:
    """nearest grid value, ties to the even code, |v| >= 448 saturates"""
    grid = _lib_grid()
    a = np.abs(v.astype(np.float64))
    sign = np.signbit(v).astype(np.uint8) << 7
    i = np.clip(np.searchsorted(grid, a, side="right") - 1, 0, 125)
    lo, hi = grid[i], grid[i + 1]
    d0, d1 = a - lo, hi - a
    pick = np.where(d0 < d1, i, np.where(d1 < d0, i + 1, np.where(i % 2 == 0, i, i + 1)))
    pick = np.where(a >= 448.0, 126, pick)
    return (pick.astype(np.uint8) | sign).astype(np.uint8)


def test_decode_all_codes_match_library():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    nan_ours = np.isnan(ours)
    assert np.array_equal(nan_ours, np.isnan(lib))
    assert set(np.nonzero(nan_ours)[0]) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan_ours].view(np.uint32), lib[~nan_ours].view(np.uint32))


def test_encode_hand_cases():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_encode_cases.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                parts = line.split()
                rows.append((float(parts[0]), int(parts[1], 16)))
    vals = np.array([r[0] for r in rows], np.float32)
    want = np.array([r[1] for r in rows], np.uint8)
    got = oracle.e4m3_encode(vals)
    bad = [(float(v), hex(g), hex(w)) for v, g, w in zip(vals, got, want) if g != w]
    assert not bad, bad


def test_encode_every_bf16_pattern_brute_force():
    bits = np.arange(65536, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    v = v[~np.isnan(v)]
    assert np.array_equal(oracle.e4m3_encode(v), _brute_encode(v))


def test_encode_random_and_midpoints_brute_force():
    rng = np.random.default_rng(123)
    grid = _lib_grid()
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    around = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                             np.nextafter(mids, np.float32(1e9)), grid.astype(np.float32)])
    rnd = np.concatenate([
        rng.standard_normal(200_000).astype(np.float32) * 100,
        rng.uniform(-0.02, 0.02, 100_000).astype(np.float32),
        (rng.integers(0, 2**31, 100_000, dtype=np.uint32)).view(np.float32),
    ])
    v = np.concatenate([around, -around, rnd])
    v = v[np.isfinite(v)]
    assert np.array_equal(oracle.e4m3_encode(v), _brute_encode(v))


def test_encode_matches_library_rne_cast_in_range():
    # torch's cast rounds to nearest even but does not saturate: compare where
    # the nearest value is finite (|v| < 464).
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(300_000).astype(np.float32) * 60,
                        rng.uniform(-463.9, 463.9, 100_000).astype(np.float32)])
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(v), lib)


@pytest.mark.parametrize("v", [448.0, 449.0, 463.99, 464.0, 480.0, 1e5, 3.4e38, np.inf])
def test_encode_saturates(v):
    got = oracle.e4m3_encode(np.array([v, -v], np.float32))
    assert list(got) == [0x7E, 0xFE]


def test_roundtrip_is_identity_on_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)
