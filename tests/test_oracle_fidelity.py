"""Oracle: the RoPE-logit fidelity diagnostic and the uniform TQ-MSE baseline.

The diagnostic is the mean absolute error of the attention logits
scale * q.k_hat against scale * q.k over the cached tokens, per query head
(review §3: Block-GTQ lowers the RoPE-logit error against uniform TQ-MSE at
matched bit budgets).  Pins: a hand-computed example, the zero-error and
single-token cases, the structure of the uniform baseline, and the paper's
claim in kind on the synthetic energy model.
"""

import math

import numpy as np
import pytest

from oracle import bgtq_oracle as O
from rope_aware_quantized_gb300 import synth


def test_logit_mae_hand_example():
    # two query rows, three tokens; only dims 0 and 5 are non-zero
    q = np.zeros((2, 128), np.float16)
    q[0, 0], q[0, 5] = 2.0, -1.0
    q[1, 5] = 4.0
    k = np.zeros((3, 128), np.float16)
    k[0, 0], k[1, 5], k[2, 0], k[2, 5] = 1.0, 1.0, 0.5, 0.5
    khat = k.astype(np.float32).copy()
    khat[0, 0] += 0.25   # q0 logit off by 2 * 0.25 = 0.5, q1 by 0
    khat[1, 5] -= 0.5    # q0 off by -1 * -0.5 = 0.5, q1 by 4 * -0.5 = -2
    khat[2, 0] += 1.0    # q0 off by 2, q1 by 0
    # per row: mean |diff| * scale; scale 0.5
    want = 0.5 * np.array([(0.5 + 0.5 + 2.0) / 3.0, (0.0 + 2.0 + 0.0) / 3.0])
    got = O.logit_mae(q, k, khat, scale=0.5)
    assert np.allclose(got, want, rtol=0, atol=1e-15)


def test_logit_mae_zero_and_single_token():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((3, 128)).astype(np.float16)
    k = rng.standard_normal((9, 128)).astype(np.float16)
    assert np.all(O.logit_mae(q, k, k.astype(np.float32)) == 0.0)
    khat = k[:1].astype(np.float64) + rng.standard_normal((1, 128)) * 0.1
    want = np.abs((q.astype(np.float64) @ (k[0].astype(np.float64) - khat[0]))) / math.sqrt(128)
    assert np.allclose(O.logit_mae(q, k[:1], khat), want, rtol=1e-12)


@pytest.mark.parametrize("bits_per_key", [256, 384])
def test_uniform_baseline_structure(bits_per_key):
    hs = O.uniform_head_state(bits_per_key, 3, 77, 1)
    kc = hs.kc
    assert np.all(hs.bits == bits_per_key // 128)
    assert kc.n_coded == 128
    assert np.all(kc.psize == 128)                   # one rotation piece, as for values
    assert np.all(kc.w == 1.0) and np.all(kc.sig == 1.0)   # no whitening
    assert np.all(kc.width == bits_per_key // 128)
    assert sorted(kc.perm.tolist()) == list(range(128))


@pytest.mark.parametrize("bits_per_key,seed", [(256, 3), (384, 3), (256, 11), (384, 11)])
def test_block_gtq_lowers_logit_error_against_uniform(bits_per_key, seed):
    """The paper's claim in kind: with heavy low-frequency RoPE blocks (the
    synthetic energy model), Block-GTQ's per-block widths give a smaller
    logit error than uniform TQ-MSE at the same key budget."""
    li = synth.layer_inputs(seed, 0, 1, 8, 1024, 1e6, 1.2)
    hb = O.head_state(li.calib[0], bits_per_key, 3, 99, 0)
    hu = O.uniform_head_state(bits_per_key, 3, 99, 0)
    kb, rb = O.encode(li.k[0], hb.kc)
    ku, ru = O.encode(li.k[0], hu.kc)
    mb = O.logit_mae(li.q[0], li.k[0], O.dequant(kb, rb, hb.kc))
    mu = O.logit_mae(li.q[0], li.k[0], O.dequant(ku, ru, hu.kc))
    assert mb.mean() < 0.5 * mu.mean()
    assert np.all(mb < mu)
