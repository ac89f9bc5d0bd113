"""Oracle: attention of a later prompt chunk over the packed prefix of its
cache and its own fp16 tokens (reading R22), pinned by reductions to the
already pinned empty-cache prefill (R21) and decode attention (R14), by the
split-softmax merge identity, by a hand example and by invariants that a
shifted causal offset, a dropped prefix or a mixed-up operand would break."""

import math

import numpy as np

from oracle import bgtq_oracle as O


def rnd(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float16)


def test_an_empty_prefix_is_the_empty_cache_prefill():
    C = 75
    q, k, v = rnd((3, C, 128), 1), rnd((C, 128), 2), rnd((C, 128), 3)
    empty = np.zeros((0, 128))
    got = O.chunk_prefill_attention(q, empty, empty, k, v)
    assert np.allclose(got, O.prefill_attention(q, k, v), rtol=0, atol=1e-12)


def test_every_row_is_decode_attention_over_prefix_and_chunk_so_far():
    P0, C, G = 40, 9, 2
    kp = rnd((P0, 128), 4).astype(np.float32) * np.float32(0.9)  # dequantised prefix: any fp32 rows
    vp = rnd((P0, 128), 5).astype(np.float32)
    q, k, v = rnd((G, C, 128), 6), rnd((C, 128), 7), rnd((C, 128), 8)
    got = O.chunk_prefill_attention(q, kp, vp, k, v)
    for i in range(C):
        keys = np.concatenate([kp.astype(np.float64), k[:i + 1].astype(np.float64)])
        vals = np.concatenate([vp.astype(np.float64), v[:i + 1].astype(np.float64)])
        assert np.allclose(got[:, i], O.attention(q[:, i], keys, vals), rtol=0, atol=1e-12)


def test_split_softmax_merge_of_prefix_and_chunk_parts():
    P0, C, G = 100, 33, 4
    kp, vp = rnd((P0, 128), 9).astype(np.float32), rnd((P0, 128), 10).astype(np.float32)
    q, k, v = rnd((G, C, 128), 11), rnd((C, 128), 12), rnd((C, 128), 13)
    got = O.chunk_prefill_attention(q, kp, vp, k, v, rows=8)
    for i in (0, 1, 17, C - 1):
        a = O.attention_partial(q[:, i], kp, vp)
        b = O.attention_partial(q[:, i], k[:i + 1].astype(np.float32), v[:i + 1].astype(np.float32))
        assert np.allclose(got[:, i], O.merge_partials([a, b]), rtol=0, atol=1e-12)


def test_hand_example_one_prefix_key_two_chunk_tokens():
    # prefix key kp0; chunk keys k0, k1; row 0 sees {kp0, k0}, row 1 sees all three
    q = np.zeros((1, 2, 128), np.float16)
    q[0, 0, 0] = 1.0
    q[0, 1, 1] = 2.0
    kp = np.zeros((1, 128))
    vp = np.zeros((1, 128))
    kp[0, 0], kp[0, 1] = 0.5, 1.0      # q0 . kp0 = 0.5, q1 . kp0 = 2
    vp[0, 3] = 4.0
    k = np.zeros((2, 128), np.float16)
    v = np.zeros((2, 128), np.float16)
    k[0, 0] = -1.0                     # q0 . k0 = -1, q1 . k0 = 0
    k[1, 1] = 0.25                     # q1 . k1 = 0.5 (row 0 must not see it)
    v[0, 3], v[1, 3] = -2.0, 8.0
    out = O.chunk_prefill_attention(q, kp, vp, k, v, scale=1.0)
    e = [math.exp(0.5), math.exp(-1.0)]
    assert math.isclose(out[0, 0, 3], (4.0 * e[0] - 2.0 * e[1]) / sum(e), rel_tol=1e-12)
    e = [math.exp(2.0), math.exp(0.0), math.exp(0.5)]
    assert math.isclose(out[0, 1, 3], (4.0 * e[0] - 2.0 * e[1] + 8.0 * e[2]) / sum(e), rel_tol=1e-12)
    assert np.count_nonzero(out[0, :, np.arange(128) != 3]) == 0


def test_rows_ignore_later_chunk_tokens_and_see_the_whole_prefix():
    P0, C = 30, 20
    kp, vp = rnd((P0, 128), 14).astype(np.float32), rnd((P0, 128), 15).astype(np.float32)
    q, k, v = rnd((2, C, 128), 16), rnd((C, 128), 17), rnd((C, 128), 18)
    base = O.chunk_prefill_attention(q, kp, vp, k, v)
    k2, v2 = k.copy(), v.copy()
    k2[12:], v2[12:] = rnd((C - 12, 128), 19), rnd((C - 12, 128), 20)
    later = O.chunk_prefill_attention(q, kp, vp, k2, v2)
    assert np.array_equal(base[:, :12], later[:, :12]) and not np.allclose(base[:, 12:], later[:, 12:])
    vp2 = vp.copy()
    vp2[0] += 1.0  # the oldest prefix value reaches every row
    moved = O.chunk_prefill_attention(q, kp, vp2, k, v)
    assert (np.abs(moved - base).max(axis=2) > 0).all()


def test_the_prefix_uses_the_cached_keys_not_the_prompt_keys():
    # a cached prefix from the codec: the chunk attends the dequantised rows
    H, P0, C = 1, 64, 16
    rng = np.random.default_rng(21)
    calib = (rng.standard_normal((256, 128)) * np.linspace(0.2, 3.0, 128)).astype(np.float16)
    hs = O.head_state(calib, 256, 2, 0x123, 0)
    kfull = (rng.standard_normal((P0 + C, 128)) * np.linspace(0.2, 3.0, 128)).astype(np.float16)
    vfull = rng.standard_normal((P0 + C, 128)).astype(np.float16)
    enc = O.encode_head(hs, kfull[:P0], vfull[:P0])
    q = rnd((2, C, 128), 22, 0.3)
    got = O.chunk_prefill_attention(q, enc["khat"], enc["vhat"], kfull[P0:], vfull[P0:])
    qf = np.zeros((2, P0 + C, 128), np.float16)
    qf[:, P0:] = q
    exact = O.prefill_attention(qf, kfull, vfull)[:, P0:]  # the prefix as given instead: differs
    assert not np.allclose(got, exact, rtol=0, atol=1e-6)
    last = O.attention(q[:, C - 1], np.concatenate([enc["khat"], kfull[P0:]]), np.concatenate([enc["vhat"], vfull[P0:]]))
    assert np.allclose(got[:, C - 1], last, rtol=0, atol=1e-12)
