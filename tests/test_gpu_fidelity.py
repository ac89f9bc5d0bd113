"""GPU: the RoPE-logit fidelity diagnostic (bgtq_logit_mae) against the oracle.

For a Block-GTQ plan and the uniform TQ-MSE plan at the same key budget
(every block at bK bits, equal energies), the kernel's per-query-head mean
absolute logit error must equal the oracle's float64 value within float32
summation error, and Block-GTQ must come out below uniform, as the oracle
says (review §3 Method & Key Results).
"""

import numpy as np
import pytest

import rope_aware_quantized_gb300 as bg
from oracle import bgtq_oracle as O
from rope_aware_quantized_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run(seed, H, G, T, bits_per_key, uniform, s_ln=1.2):
    li = synth.layer_inputs(seed, 0, H, G, T, 1e6, s_ln)
    pseed = 0x5EED + seed
    if uniform:
        bits = np.full((H, 64), bits_per_key // 128, np.uint8)
        energy = np.full((H, 64), 2.0)
        heads = [O.uniform_head_state(bits_per_key, 2, pseed, h) for h in range(H)]
    else:
        be = [bg.bgtq_alloc_bits(li.calib[h], bits_per_key) for h in range(H)]
        bits = np.stack([b for b, _ in be])
        energy = np.stack([e for _, e in be])
        heads = [O.head_state(li.calib[h], bits_per_key, 2, pseed, h) for h in range(H)]
    plan = bg.bgtq_plan_create(bits, energy, G, bits_per_key, 2, pseed)
    cache = bg.Cache(plan, 1, T + (T % 2))
    k = dev(li.k[None])
    bg.bgtq_quantize_append(plan, k, dev(li.v[None]), dev(np.array([0], np.int32)), cache)
    out = torch.empty((1, H * G), dtype=torch.float32, device="cuda")
    bg.bgtq_logit_mae(plan, dev(li.q[None]), k, cache, T, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()[0].astype(np.float64)
    want = []
    for h, hs in enumerate(heads):
        codes, rho = O.encode(li.k[h], hs.kc)
        want.append(O.logit_mae(li.q[h * G:(h + 1) * G], li.k[h], O.dequant(codes, rho, hs.kc)))
    return got, np.concatenate(want)


@pytest.mark.parametrize("H,G,T,bits_per_key", [(2, 8, 3000, 384), (2, 8, 2049, 256), (3, 4, 700, 384), (1, 2, 17, 256)])
def test_logit_mae_matches_oracle_and_block_gtq_wins(H, G, T, bits_per_key):
    gb, wb = run(60 + T, H, G, T, bits_per_key, uniform=False)
    gu, wu = run(60 + T, H, G, T, bits_per_key, uniform=True)
    for got, want in ((gb, wb), (gu, wu)):
        assert np.all(np.isfinite(got))
        assert np.allclose(got, want, rtol=2e-3, atol=1e-5), (got, want)
    assert gb.mean() < gu.mean()
