"""Pins of the oracle's attention over the dequantised cache.

The packed-cache path must compute ordinary softmax attention over the
compressed cache without materialising an fp16 copy ("RoPE-Aware Bit
Allocation for KV-Cache Quantization": English abstract, packed-cache
serving path; review §1 "Packed-Cache").  Token order inside K/V does not
change the output (LogQuant summary page, §4 position-agnostic attention,
A·V = A_P·V_P), which also makes split-and-merge exact.
"""

import math

import numpy as np
import pytest
from scipy.special import softmax

from oracle import bgtq_oracle as O


def data(seed, t=300, g=4):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((g, 128)) * 3).astype(np.float16)
    k = rng.standard_normal((t, 128)).astype(np.float32)
    v = rng.standard_normal((t, 128)).astype(np.float32)
    return q, k, v


@pytest.mark.parametrize("seed", range(4))
def test_matches_library_softmax(seed):
    q, k, v = data(seed)
    scale = 1 / math.sqrt(128)
    ref = softmax(q.astype(np.float64) @ k.astype(np.float64).T * scale, axis=1) @ v.astype(np.float64)
    assert np.allclose(O.attention(q, k, v), ref, rtol=1e-12, atol=1e-12)


def test_single_token_and_zero_query():
    q, k, v = data(1)
    assert np.allclose(O.attention(q, k[:1], v[:1]), np.repeat(v[:1].astype(np.float64), 4, 0), atol=1e-15)
    z = np.zeros_like(q)
    assert np.allclose(O.attention(z, k, v), np.repeat(v.astype(np.float64).mean(0, keepdims=True), 4, 0))


def test_permutation_and_split_invariance():
    q, k, v = data(2, t=777)
    ref = O.attention(q, k, v)
    perm = np.random.default_rng(0).permutation(777)
    assert np.allclose(O.attention(q, k[perm], v[perm]), ref, atol=1e-12)
    cuts = [0, 5, 200, 201, 650, 777]
    parts = [O.attention_partial(q, k[a:b], v[a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    assert np.allclose(O.merge_partials(parts), ref, atol=1e-12)


def test_peaked_softmax_stays_finite():
    q, k, v = data(3)
    q = (q.astype(np.float32) * 300).astype(np.float16)
    o = O.attention(q, k, v)
    assert np.all(np.isfinite(o))
