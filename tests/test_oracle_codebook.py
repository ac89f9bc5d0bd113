"""Pins of the oracle's TQ-MSE scalar codebook (Lloyd-Max for N(0,1)).

The pages call TQ-MSE near-optimal in distortion rate ("RoPE-Aware Bit
Allocation for KV-Cache Quantization" review, §1 Key Terms) without printing
the codebook; the build reads it as the Lloyd-Max quantiser of a unit
Gaussian.  Pins: the b = 1 closed form, the published table of J. Max (1960),
the optimality conditions by independent quadrature, symmetry, the
high-rate asymptote, and brute-force nearest-centroid coding.
"""

import math
import os

import numpy as np
import pytest
from scipy import integrate

from oracle import bgtq_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "lloyd_max_gaussian.txt")


def load_max_table():
    tab = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        tab[(int(parts[0]), parts[1])] = [float(v) for v in parts[2:]]
    return tab


def pdf(x):
    return math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)


def quad_moments(a, b):
    m0 = integrate.quad(pdf, a, b, epsabs=1e-15, epsrel=1e-13, limit=200)[0]
    m1 = integrate.quad(lambda x: x * pdf(x), a, b, epsabs=1e-15, epsrel=1e-13, limit=200)[0]
    return m0, m1


def distortion(cent, thr):
    edges = [-np.inf] + list(thr) + [np.inf]
    tot = 0.0
    for k, c in enumerate(cent):
        tot += integrate.quad(lambda x: (x - c) ** 2 * pdf(x), edges[k], edges[k + 1],
                              epsabs=1e-15, epsrel=1e-12, limit=200)[0]
    return tot


def test_one_bit_closed_form():
    c, t = O.lloyd_max_fp64(1)
    assert math.isclose(c[1], math.sqrt(2 / math.pi), rel_tol=1e-15)
    cent, thr = O.codebook(1)
    assert cent[1] == np.float32(np.float16(math.sqrt(2 / math.pi)))
    assert thr[0] == 0.0
    assert math.isclose(distortion(c, t), 1 - 2 / math.pi, rel_tol=1e-9)


def test_published_table():
    tab = load_max_table()
    for levels in (2, 4, 8, 16):
        b = int(math.log2(levels))
        c, t = O.lloyd_max_fp64(b)
        pos_c = c[levels // 2:]
        assert np.allclose(pos_c, tab[(levels, "output")], atol=1.5e-3, rtol=0)
        if (levels, "threshold") in tab:
            assert np.allclose(t[levels // 2:], tab[(levels, "threshold")], atol=1.5e-3, rtol=0)
        d = distortion(c, t)
        assert math.isclose(d, tab[(levels, "distortion")][0], rel_tol=2e-3)


@pytest.mark.parametrize("b", range(2, 9))
def test_optimality_conditions_by_quadrature(b):
    c, t = O.lloyd_max_fp64(b)
    edges = [-np.inf] + list(t) + [np.inf]
    # every threshold is the midpoint of its neighbours
    assert np.max(np.abs(t - 0.5 * (c[:-1] + c[1:]))) < 1e-12
    # every centroid is the conditional mean of its cell (independent quadrature)
    for k in range(0, len(c), max(1, len(c) // 16)):
        m0, m1 = quad_moments(edges[k], edges[k + 1])
        assert abs(m1 / m0 - c[k]) < 1e-9
    # symmetric and strictly increasing
    assert np.allclose(c, -c[::-1], atol=0, rtol=0)
    assert np.all(np.diff(c) > 0)


@pytest.mark.parametrize("b", range(1, 9))
def test_fp16_rounding_is_robust_and_distinct(b):
    c, _ = O.lloyd_max_fp64(b)
    cent, thr = O.codebook(b)
    assert np.all(np.diff(cent) > 0)
    assert np.all(cent.astype(np.float16).astype(np.float32) == cent)
    # each centroid is far (>= 1e-9) from an fp16 rounding boundary, so any
    # correct float64 solver rounds to the same fp16 codebook
    for x in c:
        h = np.float16(x)
        up = np.nextafter(h, np.float16(np.inf))
        dn = np.nextafter(h, np.float16(-np.inf))
        mid_up = 0.5 * (float(h) + float(up))
        mid_dn = 0.5 * (float(h) + float(dn))
        assert min(abs(x - mid_up), abs(x - mid_dn)) > 1e-9
    # thresholds are exact midpoints of the rounded centroids
    mids = 0.5 * (cent[:-1].astype(np.float64) + cent[1:].astype(np.float64))
    assert np.array_equal(thr.astype(np.float64), mids)


def test_distortion_falls_about_4x_per_bit_and_meets_high_rate_limit():
    d = []
    for b in range(1, 9):
        c, t = O.lloyd_max_fp64(b)
        d.append(distortion(c, t))
    ratios = [d[i] / d[i + 1] for i in range(len(d) - 1)]
    assert all(2.8 < r < 4.3 for r in ratios)
    assert all(ratios[i] < ratios[i + 1] for i in range(len(ratios) - 1))
    panter_dite = math.sqrt(3) * math.pi / 2
    assert abs(d[-1] * 4 ** 8 / panter_dite - 1) < 0.03


@pytest.mark.parametrize("b", range(1, 9))
def test_threshold_count_equals_nearest_centroid(b):
    """code = #{thresholds <= u} equals argmin |u - c_k| with ties to the larger k.

    Inputs: every finite fp16 value (distances to fp16 centroids are exact in
    float64) and every threshold with its two float32 neighbours (distances
    compared exactly as rationals).
    """
    from fractions import Fraction
    cent, thr = O.codebook(b)
    allh = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    u = allh[np.isfinite(allh)].astype(np.float32)
    code = np.searchsorted(thr, u, side="right")
    dist = np.abs(u[:, None].astype(np.float64) - cent[None, :].astype(np.float64))
    best = dist.min(axis=1, keepdims=True)
    brute = len(cent) - 1 - np.argmax((dist == best)[:, ::-1], axis=1)
    assert np.array_equal(code, brute)
    extra = np.concatenate([thr, np.nextafter(thr, np.float32(np.inf)), np.nextafter(thr, np.float32(-np.inf))])
    cf = [Fraction(float(c)) for c in cent]
    for x in extra.astype(np.float32):
        xf = Fraction(float(x))
        d = [abs(xf - c) for c in cf]
        m = min(d)
        want = max(k for k in range(len(cf)) if d[k] == m)
        assert int(np.searchsorted(thr, x, side="right")) == want
