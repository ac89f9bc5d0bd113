"""Oracle: causal prefill attention over the prompt's fp16 keys and values
(reading R21), pinned by closed forms and invariants that a dropped or
shifted mask, a missing scale or a transposed operand would break."""

import math

import numpy as np

from oracle import bgtq_oracle as O


def rnd(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float16)


def test_single_token_returns_its_value():
    q, k, v = rnd((3, 1, 128), 1), rnd((1, 128), 2), rnd((1, 128), 3)
    out = O.prefill_attention(q, k, v)
    assert np.array_equal(out, np.broadcast_to(v.astype(np.float64), (3, 1, 128)))


def test_zero_query_gives_the_running_mean_of_values():
    T = 37
    v = rnd((T, 128), 4)
    out = O.prefill_attention(np.zeros((2, T, 128), np.float16), rnd((T, 128), 5), v)
    want = np.cumsum(v.astype(np.float64), axis=0) / np.arange(1, T + 1)[:, None]
    assert np.allclose(out[0], want, rtol=0, atol=1e-12) and np.allclose(out[1], want, rtol=0, atol=1e-12)


def test_hand_example_two_tokens():
    # q_1 . k_0 = 2, q_1 . k_1 = -1 (dims 0 and 1 only), scale 0.5
    q = np.zeros((1, 2, 128), np.float16)
    k = np.zeros((2, 128), np.float16)
    v = np.zeros((2, 128), np.float16)
    q[0, 1, 0], q[0, 1, 1] = 1.0, 1.0
    k[0, 0], k[1, 1] = 2.0, -1.0
    v[0, 5], v[1, 5] = 3.0, -2.0
    v[0, 7] = 1.0
    out = O.prefill_attention(q, k, v, scale=0.5)
    e0, e1 = math.exp(1.0), math.exp(-0.5)
    assert np.allclose(out[0, 0, 5], 3.0) and np.allclose(out[0, 0, 7], 1.0)   # row 0 sees token 0 only
    assert np.allclose(out[0, 1, 5], (3.0 * e0 - 2.0 * e1) / (e0 + e1), rtol=1e-14)
    assert np.allclose(out[0, 1, 7], e0 / (e0 + e1), rtol=1e-14)


def test_last_row_is_full_attention_and_rows_ignore_the_future():
    G, T = 4, 300
    q, k, v = rnd((G, T, 128), 6), rnd((T, 128), 7), rnd((T, 128), 8)
    out = O.prefill_attention(q, k, v, rows=64)
    assert np.allclose(out[:, -1], O.attention(q[:, -1], k, v), rtol=1e-12, atol=1e-12)
    i = 123
    assert np.allclose(out[:, i], O.attention(q[:, i], k[:i + 1], v[:i + 1]), rtol=1e-12, atol=1e-12)
    k2, v2 = k.copy(), v.copy()
    k2[i + 1:] = rnd((T - i - 1, 128), 9, 3.0)
    v2[i + 1:] = rnd((T - i - 1, 128), 10, 3.0)
    out2 = O.prefill_attention(q, k2, v2, rows=50)
    assert np.array_equal(out[:, :i + 1], out2[:, :i + 1]) or np.allclose(out[:, :i + 1], out2[:, :i + 1],
                                                                           rtol=0, atol=1e-13)


def test_prefix_order_does_not_matter():
    """Permuting the (key, value) pairs of a row's prefix leaves that row's
    output unchanged (the order invariance of A.V)."""
    T = 64
    q, k, v = rnd((2, T, 128), 11), rnd((T, 128), 12), rnd((T, 128), 13)
    perm = np.random.default_rng(14).permutation(T)
    a = O.prefill_attention(q, k, v)[:, -1]
    b = O.prefill_attention(q, k[perm], v[perm])[:, -1]
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)
