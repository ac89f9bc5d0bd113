"""GPU: the fp16 recent-key buffer (reading R20) against the oracle.

With a buffer of W keys, appends also copy the last W keys as given into
ring slot (position mod W), and decode uses those exact keys for positions
[seq_len - W, seq_len) and the packed keys before (abstract: results are
quoted "without an fp16 recent-key buffer", so the option exists).
"""

import numpy as np
import pytest

import rope_aware_quantized_gb300 as bg
from oracle import bgtq_oracle as O
from rope_aware_quantized_gb300 import synth

from tests.test_gpu_parity import check_close, dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def setup(seed, H, G, T, W, bits_per_key=384, v_bits=3, batch=1):
    li = [synth.layer_inputs(seed + 13 * b, 0, H, G, T, 1e5, 1.2) for b in range(batch)]
    be = [bg.bgtq_alloc_bits(li[0].calib[h], bits_per_key) for h in range(H)]
    pseed = 0xBEEF + seed
    plan = bg.bgtq_plan_create(np.stack([b for b, _ in be]), np.stack([e for _, e in be]), G, bits_per_key, v_bits,
                               pseed)
    cache = bg.Cache(plan, batch, T + (T % 2), recent=W)
    heads = [O.head_state(li[0].calib[h], bits_per_key, v_bits, pseed, h) for h in range(H)]
    return li, plan, cache, heads


def want_out(heads, l, q, n, G, W):
    outs = []
    for h, hs in enumerate(heads):
        enc = O.encode_head(hs, l.k[h][:n], l.v[h][:n])
        outs.append(O.attention_recent(q[h * G:(h + 1) * G], enc["khat"], enc["vhat"], l.k[h][:n], W))
    return np.concatenate(outs, axis=0)


def decode(plan, cache, q, lens, max_len):
    ws = torch.zeros(bg.bgtq_decode_attn_workspace(plan, q.shape[0], max_len), dtype=torch.uint8, device="cuda")
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bgtq_decode_attn(plan, q, cache, lens, max_len, out, ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("T,W", [(3000, 16), (3000, 100), (3000, 1000), (2049, 64), (200, 200), (777, 1)])
def test_decode_with_recent_buffer_matches_oracle(T, W):
    H, G = 2, 8
    li, plan, cache, heads = setup(30 + W, H, G, T, W)
    bg.bgtq_quantize_append(plan, dev(li[0].k[None]), dev(li[0].v[None]), dev(np.array([0], np.int32)), cache)
    # the ring holds the last W keys as given, at slot position mod W
    ring = cache.k_recent.view(1, H, W, 128).cpu().numpy()
    for h in range(H):
        for pos in range(max(0, T - W), T):
            assert np.array_equal(ring[0, h, pos % W], li[0].k[h][pos])
    got = decode(plan, cache, dev(li[0].q[None]), dev(np.array([T], np.int32)), T)
    check_close(got[0], want_out(heads, li[0], li[0].q, T, G, W))


def test_recent_buffer_fused_step_and_two_calls_agree():
    H, G, T, W = 2, 8, 1500, 96
    li, plan, cache_a, heads = setup(71, H, G, T, W)
    cache_b = bg.Cache(plan, 1, cache_a.capacity, recent=W)
    for c in (cache_a, cache_b):
        bg.bgtq_quantize_append(plan, dev(li[0].k[None, :, :T - 1]), dev(li[0].v[None, :, :T - 1]),
                                dev(np.array([0], np.int32)), c)
    k_new = li[0].k[:, T - 1][None]
    v_new = li[0].v[:, T - 1][None]
    pos = dev(np.array([T - 1], np.int32))
    seq = dev(np.array([T], np.int32))
    q = dev(li[0].q[None])
    bg.bgtq_quantize_append(plan, dev(k_new[:, :, None]), dev(v_new[:, :, None]), pos, cache_a)
    a = decode(plan, cache_a, q, seq, T)
    ws = torch.zeros(bg.bgtq_decode_attn_workspace(plan, 1, T), dtype=torch.uint8, device="cuda")
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    bg.bgtq_decode_step(plan, q, dev(k_new), dev(v_new), pos, cache_b, seq, T, out, ws)
    torch.cuda.synchronize()
    b = out.cpu().numpy().astype(np.float64)
    assert torch.equal(cache_a.k_recent, cache_b.k_recent)
    assert torch.equal(cache_a.k_codes, cache_b.k_codes)
    assert np.array_equal(a, b)
    check_close(b[0], want_out(heads, li[0], li[0].q, T, G, W))


def test_recent_buffer_ragged_batch():
    H, G, T, W = 2, 4, 1200, 48
    li, plan, cache, heads = setup(5, H, G, T, W, bits_per_key=256, v_bits=2, batch=3)
    lens = np.array([1200, 37, 600], np.int32)
    for b in range(3):
        view = cache.sequence_view(b)
        n = int(lens[b])
        bg.bgtq_quantize_append(plan, dev(li[b].k[None, :, :n]), dev(li[b].v[None, :, :n]),
                                dev(np.array([0], np.int32)), view)
    q = np.stack([l.q for l in li])
    got = decode(plan, cache, dev(q), dev(lens), T)
    for b in range(3):
        check_close(got[b], want_out(heads, li[b], q[b], int(lens[b]), G, W))


@pytest.mark.parametrize("layout", ["uniform3", "wide8"])
def test_recent_buffer_both_kernel_paths(layout):
    """Explicit widths that fix which decode path runs: every block at 3 bits
    (no code wider than the pair tables: the fast path) and 24 blocks at 8
    bits with the rest at 0 (wide codes in many slots: the general path),
    both at 384 bits per key."""
    H, G, T, W, v_bits = 2, 8, 2500, 200, 3
    li = synth.layer_inputs(808, 0, H, G, T, 1e5, 1.2)
    energy = np.stack([bg.bgtq_alloc_bits(li.calib[h], 384)[1] for h in range(H)])
    if layout == "uniform3":
        bits = np.full((H, 64), 3, np.uint8)
    else:
        bits = np.zeros((H, 64), np.uint8)
        bits[0, :24] = 8
        bits[1, 40:] = 8
    pseed = 0xA11CE
    plan = bg.bgtq_plan_create(bits, energy, G, 384, v_bits, pseed)
    cache = bg.Cache(plan, 1, T, recent=W)
    heads = [O.HeadState(O.k_codec(bits[h].astype(np.int64), energy[h], pseed, h), O.v_codec(v_bits, pseed, h),
                         bits[h].astype(np.int64), energy[h], 3, v_bits) for h in range(H)]
    bg.bgtq_quantize_append(plan, dev(li.k[None]), dev(li.v[None]), dev(np.array([0], np.int32)), cache)
    got = decode(plan, cache, dev(li.q[None]), dev(np.array([T], np.int32)), T)
    check_close(got[0], want_out(heads, li, li.q, T, G, W))
    # the same cache without the window path gives the packed-key result
    plain = bg.Cache(plan, 1, T)
    bg.bgtq_quantize_append(plan, dev(li.k[None]), dev(li.v[None]), dev(np.array([0], np.int32)), plain)
    got0 = decode(plan, plain, dev(li.q[None]), dev(np.array([T], np.int32)), T)
    check_close(got0[0], want_out(heads, li, li.q, T, G, 0))
