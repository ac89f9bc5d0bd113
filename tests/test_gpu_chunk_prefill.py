"""GPU: a later prompt chunk onto a cache that holds the earlier tokens
packed (bgtq_prefill_chunk_attn, reading R22) against the oracle.

The cache after the call must equal, bit for bit, one append of the whole
prompt (the chunk's records are an append at pos_start = P0); each chunk row's
output must match the oracle's float64 attention over the dequantised prefix
and the chunk's own fp16 tokens within the decode tolerance (max-abs 2e-3,
relative L2 1e-3; an fp16 output may differ by half a binary16 ulp more).
"""

import numpy as np
import pytest

import rope_aware_quantized_gb300 as bg
from oracle import bgtq_oracle as O
from rope_aware_quantized_gb300 import synth

from tests.test_gpu_parity import cache_arrays, check_close, dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def build(seed, H, G, T, bits_per_key=384, v_bits=3, batch=1, page_tokens=0):
    li = [synth.layer_inputs(seed + 13 * b, 0, H, G, T, 1e5, 1.2) for b in range(batch)]
    be = [bg.bgtq_alloc_bits(li[0].calib[h], bits_per_key) for h in range(H)]
    pseed = 0x3C11 + seed
    plan = bg.bgtq_plan_create(np.stack([b for b, _ in be]), np.stack([e for _, e in be]), G, bits_per_key, v_bits,
                               pseed)
    heads = [O.head_state(li[0].calib[h], bits_per_key, v_bits, pseed, h) for h in range(H)]
    return li, plan, heads


def new_cache(plan, batch, T, page_tokens=0):
    cap = T + (T % 2)
    if page_tokens:
        cap = -(-cap // page_tokens) * page_tokens
    cache = bg.Cache(plan, batch, cap, page_tokens=page_tokens)
    if page_tokens:  # pages in a shuffled order
        perm = np.random.default_rng(7).permutation(cache.n_pages).astype(np.int32)
        cache.page_table.copy_(dev(perm.reshape(cache.page_table.shape)))
    return cache


def chunk_queries(li, G, T, seed):
    qs = []
    for l in li:
        rng = np.random.default_rng(seed)
        q = np.empty((l.k.shape[0] * G, T, 128), np.float16)
        for h in range(l.k.shape[0]):
            for g in range(G):
                q[h * G + g] = l.k[h][rng.permutation(T)]  # keys of other positions as queries
        qs.append(q)
    return np.stack(qs)


def run_chunk(plan, cache, li, p0s, C, q, out_dtype=torch.float32):
    """Prefix of p0s[b] tokens of each sequence by an append (one sequence at
    a time: the others get a start past the capacity and are skipped), then
    the chunk [p0, p0 + C) in one call."""
    B = len(li)
    for b, l in enumerate(li):
        if p0s[b] == 0:
            continue
        k = np.zeros((B,) + l.k[:, :p0s[b]].shape, np.float16)
        v = np.zeros_like(k)
        k[b], v[b] = l.k[:, :p0s[b]], l.v[:, :p0s[b]]
        ps = torch.full((B,), int(cache.capacity), dtype=torch.int32, device="cuda")
        ps[b] = 0
        bg.bgtq_quantize_append(plan, dev(k), dev(v), ps, cache)
    kc = np.stack([l.k[:, p0:p0 + C] for l, p0 in zip(li, p0s)])
    vc = np.stack([l.v[:, p0:p0 + C] for l, p0 in zip(li, p0s)])
    out = torch.full(q.shape, float("nan"), dtype=out_dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(bg.bgtq_prefill_chunk_workspace(plan, B, max(p0s)) + 1, dtype=torch.uint8, device="cuda")
    bg.bgtq_prefill_chunk_attn(plan, dev(q), dev(np.ascontiguousarray(kc)), dev(np.ascontiguousarray(vc)),
                               dev(np.asarray(p0s, np.int32)), cache, out, max_prefix=max(p0s), workspace=ws, status=st)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), int(st.item())


def check_against_oracle(got, q, li, heads, p0s, C, G, fp16_out=False):
    for b, l in enumerate(li):
        p0 = p0s[b]
        for h, hs in enumerate(heads):
            if p0 > 0:
                enc = O.encode_head(hs, l.k[h][:p0], l.v[h][:p0])
                kp, vp = enc["khat"], enc["vhat"]
            else:
                kp = vp = np.zeros((0, 128))
            want = O.chunk_prefill_attention(q[b][h * G:(h + 1) * G], kp, vp, l.k[h][p0:p0 + C], l.v[h][p0:p0 + C])
            check_close(got[b][h * G:(h + 1) * G].reshape(-1, 128), want.reshape(-1, 128), fp16_out=fp16_out)


@pytest.mark.parametrize("H,G,P0,C,bits_per_key,v_bits", [
    (2, 4, 300, 200, 384, 3),    # ragged prefix and chunk tiles
    (1, 8, 128, 128, 384, 3),    # whole tiles
    (2, 2, 1000, 1, 256, 2),     # a one-token chunk
    (1, 4, 0, 150, 384, 3),      # empty prefix: the empty-cache prefill
    (2, 3, 129, 64, 384, 4),     # odd prefix: the chunk's first token completes a V pair record; G odd
    (1, 2, 700, 333, 128, 1),
])
def test_chunk_records_and_attention_match_oracle(H, G, P0, C, bits_per_key, v_bits):
    T = P0 + C
    li, plan, heads = build(500 + P0 + C, H, G, T, bits_per_key, v_bits)
    cache = new_cache(plan, 1, T)
    q = chunk_queries([type("L", (), {"k": li[0].k[:, P0:]})()], G, C, 9)
    got, st = run_chunk(plan, cache, li, [P0], C, q)
    assert st == 0
    # the cache equals one append of the whole prompt
    ref = new_cache(plan, 1, T)
    bg.bgtq_quantize_append(plan, dev(li[0].k[None]), dev(li[0].v[None]), dev(np.array([0], np.int32)), ref)
    torch.cuda.synchronize()
    bk = bits_per_key // 128
    for a, b in zip(cache_arrays(plan, cache, H, bk, v_bits), cache_arrays(plan, ref, H, bk, v_bits)):
        assert np.array_equal(a, b)
    check_against_oracle(got, q, li, heads, [P0], C, G)


def test_ragged_batch_paged_fp16_out():
    H, G, C = 2, 4, 90
    p0s = [257, 40, 0]
    T = max(p0s) + C
    li, plan, heads = build(77, H, G, T, batch=3)
    cache = new_cache(plan, 3, T, page_tokens=64)
    q = chunk_queries([type("L", (), {"k": l.k[:, p0:p0 + C]})() for l, p0 in zip(li, p0s)], G, C, 10)
    got, st = run_chunk(plan, cache, li, p0s, C, q, out_dtype=torch.float16)
    assert st == 0
    check_against_oracle(got, q, li, heads, p0s, C, G, fp16_out=True)


def test_empty_prefix_agrees_with_the_empty_cache_prefill():
    H, G, C = 2, 8, 300
    li, plan, heads = build(91, H, G, C)
    q = chunk_queries(li, G, C, 11)
    got, st = run_chunk(plan, new_cache(plan, 1, C), li, [0], C, q)
    assert st == 0
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    bg.bgtq_prefill_attn(plan, dev(q), dev(li[0].k[None]), dev(li[0].v[None]), new_cache(plan, 1, C), out)
    torch.cuda.synchronize()
    assert np.abs(got - out.cpu().numpy()).max() <= 1e-5


def test_a_chunk_past_the_capacity_is_skipped_and_flagged():
    H, G, C = 1, 2, 64
    li, plan, heads = build(5, H, G, 256)
    cache = new_cache(plan, 1, 200)
    q = chunk_queries([type("L", (), {"k": li[0].k[:, :C]})()], G, C, 12)
    out = torch.full(q.shape, 7.0, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bgtq_prefill_chunk_attn(plan, dev(q), dev(li[0].k[None, :, :C]), dev(li[0].v[None, :, :C]),
                               dev(np.array([190], np.int32)), cache, out, max_prefix=190, status=st)
    torch.cuda.synchronize()
    assert st.item() & 1
    assert torch.count_nonzero(out) == 0
    assert torch.count_nonzero(cache.k_norm) == 0


def test_a_prefix_past_max_prefix_is_flagged():
    H, G, C, P0 = 1, 2, 32, 300
    li, plan, heads = build(6, H, G, P0 + C)
    cache = new_cache(plan, 1, P0 + C)
    bg.bgtq_quantize_append(plan, dev(li[0].k[None, :, :P0]), dev(li[0].v[None, :, :P0]), dev(np.array([0], np.int32)),
                            cache)
    q = chunk_queries([type("L", (), {"k": li[0].k[:, P0:]})()], G, C, 13)
    out = torch.full(q.shape, 7.0, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bgtq_prefill_chunk_attn(plan, dev(q), dev(li[0].k[None, :, P0:]), dev(li[0].v[None, :, P0:]),
                               dev(np.array([P0], np.int32)), cache, out, max_prefix=256, status=st)
    torch.cuda.synchronize()
    assert st.item() & 2
    assert torch.count_nonzero(out) == 0
