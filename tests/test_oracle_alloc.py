"""Pins of the oracle's energy score and greedy bit allocation.

The allocation is Block-GTQ's greedy marginal-gain rule ("RoPE-Aware Bit
Allocation for KV-Cache Quantization": English abstract; review §3 Method).
Because the objective sum_i s_i 4^-b_i is separable and convex in b, the
greedy result must equal the exhaustive optimum; with s_i = 4^a_i it is an
integer water-filling with a closed form.
"""

import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import bgtq_oracle as O
from rope_aware_quantized_gb300 import synth


def objective(s, b):
    return sum(float(s[i]) * 4.0 ** (-int(b[i])) for i in range(len(b)))


@pytest.mark.parametrize("seed", range(12))
def test_greedy_equals_exhaustive(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 7))
    b_max = int(rng.integers(1, 5))
    budget_steps = int(rng.integers(0, n * b_max + 1))
    s_small = rng.lognormal(0.0, 1.5, n)
    s = np.zeros(O.NB)
    s[:n] = s_small
    bits = O.greedy_bits(s, 2 * budget_steps, b_max)
    assert bits[n:].sum() == 0
    best = min(objective(s_small, c) for c in itertools.product(range(b_max + 1), repeat=n)
               if sum(c) == budget_steps)
    assert math.isclose(objective(s_small, bits[:n]), best, rel_tol=1e-12)


@pytest.mark.parametrize("budget", [2, 128, 256, 384, 512, 1024])
def test_budget_exact_and_monotone(budget):
    rng = np.random.default_rng(budget)
    s = rng.lognormal(0.0, 1.2, O.NB)
    bits = O.greedy_bits(s, budget, 8)
    assert 2 * bits.sum() == budget
    assert bits.min() >= 0 and bits.max() <= 8
    for i in range(O.NB):
        for j in range(O.NB):
            if s[i] > s[j]:
                assert bits[i] >= bits[j]


def water_fill(a, total, b_max):
    """Closed form for s_i = 4^a_i: b_i = clip(a_i + lam, 0, b_max) at the
    largest level that fits, the remaining bits one each to the blocks that
    grow at the next level, smallest index first."""
    def at(lam):
        return [min(max(ai + lam, 0), b_max) for ai in a]
    lam = -max(a) - 1
    while sum(at(lam + 1)) <= total:
        lam += 1
    b = at(lam)
    rest = total - sum(b)
    nxt = at(lam + 1)
    for i in range(len(a)):
        if rest and nxt[i] > b[i]:
            b[i] += 1
            rest -= 1
    assert rest == 0
    return b


@pytest.mark.parametrize("seed", range(8))
def test_water_filling_closed_form(seed):
    rng = np.random.default_rng(100 + seed)
    a = [int(x) for x in rng.integers(-6, 7, O.NB)]
    s = np.array([math.ldexp(1.0, 2 * ai) for ai in a])
    b_max = int(rng.integers(3, 9))
    total = int(rng.integers(1, O.NB * b_max))
    bits = O.greedy_bits(s, 2 * total, b_max)
    assert bits.tolist() == water_fill(a, total, b_max)


def test_scale_invariance_and_uniform_special_case():
    rng = np.random.default_rng(7)
    s = rng.lognormal(0.0, 1.0, O.NB)
    ref = O.greedy_bits(s, 384, 8)
    for c in (0.25, 2.0, 1024.0):
        assert np.array_equal(O.greedy_bits(s * c, 384, 8), ref)
    # equal energies: Block-GTQ reduces to uniform TQ-MSE (abstract's baseline)
    for bk in (1, 2, 3, 4):
        assert np.array_equal(O.greedy_bits(np.ones(O.NB), 128 * bk, 8), np.full(O.NB, bk))


def test_greedy_rejects_bad_budgets():
    with pytest.raises(ValueError):
        O.greedy_bits(np.ones(O.NB), 3, 8)
    with pytest.raises(ValueError):
        O.greedy_bits(np.ones(O.NB), 2 * 64 * 4 + 2, 4)


def test_energy_exact_small_example():
    """Hand-checkable keys: exact rational expectation of the block energy."""
    rng = np.random.default_rng(3)
    n = 5
    x = (rng.integers(-64, 65, (n, O.D)) / 16.0).astype(np.float16)
    for layout in (0, 1):
        s = O.energy(x, layout)
        dims = O.block_dims(layout)
        for i, (a, b) in enumerate(dims):
            exact = sum(Fraction(float(x[t, a])) ** 2 + Fraction(float(x[t, b])) ** 2 for t in range(n)) / n
            assert s[i] == float(exact)


def test_energy_matches_generator_and_is_rope_invariant():
    """s_i ~ 2 sigma_i^2 (chi-square with 2n dof: rel. sd 1/sqrt(n)) and the
    post-RoPE score equals the pre-RoPE one (RoPE rotates inside each block)."""
    sig = synth.block_sigma(11, 0, 0, 1.2)
    n = 4096
    for layout in (0, 1):
        rng = np.random.default_rng(5)
        k_post = synth.draw_keys(rng, sig, np.arange(n), 5e5, layout)
        rng = np.random.default_rng(5)
        k_pre = synth.draw_keys(rng, sig, np.zeros(n, dtype=np.int64), 5e5, layout)
        s_post = O.energy(k_post, layout)
        s_pre = O.energy(k_pre, layout)
        rel = s_post / (2 * sig ** 2) - 1.0
        assert np.all(np.abs(rel) < 6.0 / math.sqrt(n))
        assert np.allclose(s_post, s_pre, rtol=2e-3)
    # the wrong pairing breaks RoPE invariance: pins the block definition
    k_post = synth.draw_keys(np.random.default_rng(5), sig, np.arange(n), 1e4, 0)
    k_pre = synth.draw_keys(np.random.default_rng(5), sig, np.zeros(n, dtype=np.int64), 1e4, 0)
    assert not np.allclose(O.energy(k_post, 1), O.energy(k_pre, 1), rtol=2e-2)
