"""Oracle: attention with an fp16 recent-key buffer (reading R20).

Pins: a buffer of 0 keys is plain attention over the dequantised cache; a
buffer at least as long as the sequence is attention over the exact keys
(brute-force softmax); a buffer of one key replaces exactly the newest row.
"""

import math

import numpy as np
from scipy.special import softmax

from oracle import bgtq_oracle as O
from rope_aware_quantized_gb300 import synth


def _case(seed=4, t=300):
    li = synth.layer_inputs(seed, 0, 1, 4, t, 1e4, 1.0)
    hs = O.head_state(li.calib[0], 384, 3, 9, 0)
    enc = O.encode_head(hs, li.k[0], li.v[0])
    return li, enc


def test_zero_buffer_is_plain_attention():
    li, enc = _case()
    a = O.attention_recent(li.q[:4], enc["khat"], enc["vhat"], li.k[0], 0)
    b = O.attention(li.q[:4], enc["khat"], enc["vhat"])
    assert np.array_equal(a, b)


def test_full_buffer_is_exact_key_attention():
    li, enc = _case(t=50)
    got = O.attention_recent(li.q[:4], enc["khat"], enc["vhat"], li.k[0], 64)
    logits = li.q[:4].astype(np.float64) @ li.k[0].astype(np.float64).T / math.sqrt(128)
    want = softmax(logits, axis=1) @ enc["vhat"].astype(np.float64)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_one_key_buffer_replaces_the_newest_row():
    li, enc = _case(t=40)
    kk = O.keys_with_recent(enc["khat"], li.k[0], 1)
    assert np.array_equal(kk[:-1], enc["khat"][:-1].astype(np.float64))
    assert np.array_equal(kk[-1], li.k[0][-1].astype(np.float64))
