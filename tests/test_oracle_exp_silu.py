"""Pins for the oracle's exp specification and SiLU(gate) * up.

The exp is the library's own written specification (Cody and Waite reduction
plus a degree-7 Taylor polynomial); its pins are the mathematics: double
precision exp within 2 ulp, exact special values, and the limits of SiLU.
"""
import math

import numpy as np

import oracle


def _ulp_err(got: np.ndarray, exact: np.ndarray) -> np.ndarray:
    g = got.astype(np.float64)
    ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
    return np.abs(g - exact) / ulp


def test_exp_within_two_ulp_of_double():
    x = np.concatenate([
        np.linspace(-87.0, 88.7, 2_000_001, dtype=np.float32),
        np.random.default_rng(0).uniform(-20, 20, 1_000_000).astype(np.float32),
        np.linspace(-1e-3, 1e-3, 10_001, dtype=np.float32),
    ])
    got = oracle.expf(x)
    exact = np.exp(x.astype(np.float64))
    err = _ulp_err(got, exact)
    assert err.max() <= 2.0, (float(err.max()), float(x[np.argmax(err)]))


def test_exp_subnormal_range_close():
    x = np.linspace(-103.9, -87.4, 100_001, dtype=np.float32)
    got = oracle.expf(x).astype(np.float64)
    exact = np.exp(x.astype(np.float64))
    # below 2^-126 the result has fewer significant bits: absolute error of a
    # couple of subnormal steps (2^-149) is the meaningful bound there
    assert np.max(np.abs(got - exact)) <= 3 * 2.0**-149 + 2 * np.spacing(np.float32(2.0**-126))


def test_exp_special_values():
    x = np.array([0.0, -0.0, 1.0, 88.8, 1000.0, -104.0, -1000.0, np.inf, -np.inf, np.nan],
                 np.float32)
    got = oracle.expf(x)
    assert got[0] == 1.0 and got[1] == 1.0
    assert abs(float(got[2]) - math.e) <= float(np.spacing(np.float32(math.e)))
    assert np.isinf(got[3]) and np.isinf(got[4]) and np.isinf(got[7])
    assert got[5] == 0.0 and got[6] == 0.0 and got[8] == 0.0
    assert np.isnan(got[9])


def test_silu_mul_limits_and_accuracy():
    g = np.array([0.0, 30.0, 100.0, -120.0, -200.0], np.float32)
    u = np.ones_like(g)
    s = oracle.silu_mul(g, u)
    assert s[0] == 0.0
    assert s[1] == np.float32(30.0) and s[2] == np.float32(100.0)  # e^-g vanishes next to 1
    assert s[3] == 0.0 and np.signbit(s[3])  # g / inf = -0
    assert s[4] == 0.0 and np.signbit(s[4])
    rng = np.random.default_rng(1)
    g = rng.standard_normal(500_000).astype(np.float32) * 4
    u = rng.standard_normal(500_000).astype(np.float32)
    got = oracle.silu_mul(g, u).astype(np.float64)
    g64, u64 = g.astype(np.float64), u.astype(np.float64)
    exact = g64 / (1.0 + np.exp(-g64)) * u64
    # four roundings of at most ~half an ulp each plus exp's 2 ulp
    err = np.abs(got - exact) / np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
    assert np.max(err[np.abs(exact) > 1e-30]) <= 4.0
