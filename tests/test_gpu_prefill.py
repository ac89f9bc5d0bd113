"""GPU: the fused prefill (causal attention over the prompt's fp16 K/V and
the packed records of the prompt in one launch, reading R21) against the
oracle.

Records and norms must equal the oracle's encoding bit for bit (they are the
append kernel's records); the attention output must match the oracle's
float64 causal attention within the decode tolerance (max-abs 2e-3,
relative L2 1e-3): fp16 products with fp32 accumulation and probabilities
rounded to fp16 stay well inside it.
"""

import numpy as np
import pytest

import rope_aware_quantized_gb300 as bg
from oracle import bgtq_oracle as O
from rope_aware_quantized_gb300 import synth

from tests.test_gpu_parity import cache_arrays, check_close, dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def setup(seed, H, G, T, bits_per_key=384, v_bits=3, batch=1, cap=None, recent=0, page_tokens=0):
    li = [synth.layer_inputs(seed + 17 * b, 0, H, G, T, 1e5, 1.2) for b in range(batch)]
    be = [bg.bgtq_alloc_bits(li[0].calib[h], bits_per_key) for h in range(H)]
    pseed = 0x7F11 + seed
    plan = bg.bgtq_plan_create(np.stack([b for b, _ in be]), np.stack([e for _, e in be]), G, bits_per_key, v_bits,
                               pseed)
    cap = cap or T + (T % 2)
    if page_tokens:
        cap = -(-cap // page_tokens) * page_tokens
    cache = bg.Cache(plan, batch, cap, recent=recent, page_tokens=page_tokens)
    heads = [O.head_state(li[0].calib[h], bits_per_key, v_bits, pseed, h) for h in range(H)]
    return li, plan, cache, heads


def prompt_queries(li, G, T, seed):
    """Per-position queries [B][H*G][T][128]: the synthetic keys of other
    seeds at the same positions (RoPE structure like the keys')."""
    qs = []
    for l in li:
        rng = np.random.default_rng(seed)
        q = np.empty((l.k.shape[0] * G, T, 128), np.float16)
        for h in range(l.k.shape[0]):
            for g in range(G):
                perm = rng.permutation(T)
                q[h * G + g] = l.k[h][perm]  # keys of other positions as queries: same scale, no self-match
        qs.append(q)
    return np.stack(qs)


def run(plan, cache, q, li, out_dtype=torch.float32):
    k = dev(np.stack([l.k for l in li]))
    v = dev(np.stack([l.v for l in li]))
    out = torch.empty(q.shape, dtype=out_dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bgtq_prefill_attn(plan, dev(q), k, v, cache, out, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return out.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("H,G,T,bits_per_key,v_bits,batch", [
    (2, 8, 300, 384, 3, 1),     # several tiles, ragged last block
    (1, 4, 64, 256, 2, 1),      # exactly one tile
    (2, 2, 129, 384, 4, 2),     # odd length: the last V pair is half full; two sequences
    (1, 1, 1, 384, 3, 1),       # one token
    (2, 4, 1000, 128, 1, 1),
])
def test_prefill_records_and_attention_match_oracle(H, G, T, bits_per_key, v_bits, batch):
    li, plan, cache, heads = setup(300 + T, H, G, T, bits_per_key, v_bits, batch)
    q = prompt_queries(li, G, T, 5)
    got = run(plan, cache, q, li)
    bk = bits_per_key // 128
    kc, vc, kn, vn = cache_arrays(plan, cache, H, bk, v_bits)
    for b in range(batch):
        for h, hs in enumerate(heads):
            e = O.encode_head(hs, li[b].k[h], li[b].v[h])
            assert np.array_equal(kc[b, h, :T], e["krec"])
            assert np.array_equal(kn[b, h, :T], e["krho"])
            assert np.array_equal(vn[b, h, :T], e["vrho"])
            vrec = vc[b, h, :(T + 1) // 2]
            if T % 2:  # compare the written half of the last pair record only
                assert np.array_equal(vrec[:-1], e["vrec"][:-1])
                want_last = O.unpack_v(e["vrec"][-1:], v_bits, 1)[0]
                assert np.array_equal(O.unpack_v(vrec[-1:], v_bits, 1)[0], want_last)
            else:
                assert np.array_equal(vrec, e["vrec"])
            want = O.prefill_attention(q[b][h * G:(h + 1) * G], li[b].k[h], li[b].v[h])
            check_close(got[b][h * G:(h + 1) * G].reshape(-1, 128), want.reshape(-1, 128))


def test_prefill_equals_append_and_feeds_decode():
    """The prefill's cache is the append kernel's cache, bit for bit, and a
    decode over it matches the oracle; fp16 output agrees with fp32."""
    H, G, T = 2, 8, 777
    li, plan, cache, heads = setup(41, H, G, T)
    _, _, cache2, _ = setup(41, H, G, T)
    q = prompt_queries(li, G, T, 6)
    got32 = run(plan, cache, q, li)
    got16 = run(plan, cache2, q, li, out_dtype=torch.float16)
    assert np.abs(got16 - got32).max() <= 2e-3
    ref = bg.Cache(plan, 1, cache.capacity)
    bg.bgtq_quantize_append(plan, dev(li[0].k[None]), dev(li[0].v[None]), dev(np.array([0], np.int32)), ref)
    torch.cuda.synchronize()
    for a, b in zip(cache_arrays(plan, cache, H, 3, 3), cache_arrays(plan, ref, H, 3, 3)):
        assert np.array_equal(a, b)
    from tests.test_gpu_parity import decode
    dq = li[0].q[None]
    out, st = decode(plan, cache, dev(dq), dev(np.array([T], np.int32)), T)
    assert st == 0
    for h, hs in enumerate(heads):
        e = O.encode_head(hs, li[0].k[h], li[0].v[h])
        check_close(out[0][h * G:(h + 1) * G], O.attention(dq[0][h * G:(h + 1) * G], e["khat"], e["vhat"]))


def test_prefill_paged_with_recent_buffer():
    H, G, T, W, P = 2, 4, 500, 64, 32
    li, plan, cache, heads = setup(77, H, G, T, recent=W, page_tokens=P)
    perm = np.random.default_rng(3).permutation(cache.n_pages).astype(np.int32)
    cache.page_table.copy_(dev(perm.reshape(cache.page_table.shape)))
    lc, _, cont, _ = setup(77, H, G, T, recent=W)
    q = prompt_queries(li, G, T, 8)
    got = run(plan, cache, q, li)
    got_c = run(plan, cont, q, lc)
    assert np.array_equal(got, got_c)
    assert torch.equal(cache.k_recent, cont.k_recent)
    ring = cache.k_recent.view(1, H, W, 128).cpu().numpy()
    for h in range(H):
        for pos in range(T - W, T):
            assert np.array_equal(ring[0, h, pos % W], li[0].k[h][pos])
    for h in range(H):
        want = O.prefill_attention(q[0][h * G:(h + 1) * G], li[0].k[h], li[0].v[h])
        check_close(got[0][h * G:(h + 1) * G].reshape(-1, 128), want.reshape(-1, 128))


def test_prefill_long_prompt_sampled_rows():
    """A 16384-token prompt of the Qwen2.5-3B-shaped layer (2 KV heads x 8
    query heads): rows sampled across the prompt against the oracle's
    attention over their causal prefix."""
    H, G, T = 2, 8, 16384
    li, plan, cache, heads = setup(9, H, G, T)
    q = prompt_queries(li, G, T, 10)
    got = run(plan, cache, q, li, out_dtype=torch.float16)
    rng = np.random.default_rng(11)
    for i in sorted(set([0, 1, 63, 64, T - 1] + rng.integers(0, T, 12).tolist())):
        for h in range(H):
            want = O.attention(q[0][h * G:(h + 1) * G, i], li[0].k[h][:i + 1], li[0].v[h][:i + 1])
            check_close(got[0][h * G:(h + 1) * G, i], want, fp16_out=True)


def test_prefill_rejects_a_prompt_longer_than_the_cache():
    H, G, T = 1, 2, 100
    li, plan, cache, heads = setup(1, H, G, T, cap=64)
    q = prompt_queries(li, G, T, 1)
    with pytest.raises(bg.BgtqError) as e:
        run(plan, cache, q, li)
    assert e.value.code == -3


@pytest.mark.parametrize("W", [0, 48])
def test_prefill_then_decode_steps(W):
    """A serving sequence: prefill a prompt (one launch), then two decode
    steps that append and attend (bgtq_decode_step), with and without an
    fp16 recent-key buffer; every output against the oracle over the
    tokens as appended."""
    H, G, T0, steps = 2, 8, 700, 2
    T = T0 + steps
    li, plan, cache, heads = setup(55 + W, H, G, T, recent=W)
    q_prompt = prompt_queries([type("L", (), {"k": li[0].k[:, :T0]})()], G, T0, 12)
    k = dev(np.ascontiguousarray(li[0].k[None, :, :T0]))
    v = dev(np.ascontiguousarray(li[0].v[None, :, :T0]))
    out = torch.empty(q_prompt.shape, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bgtq_prefill_attn(plan, dev(q_prompt), k, v, cache, out, status=st)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    for h in range(H):
        want = O.prefill_attention(q_prompt[0][h * G:(h + 1) * G], li[0].k[h][:T0], li[0].v[h][:T0])
        check_close(got[0][h * G:(h + 1) * G].reshape(-1, 128), want.reshape(-1, 128))
    ws = torch.zeros(bg.bgtq_decode_attn_workspace(plan, 1, T), dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(13)
    for s in range(steps):
        pos = T0 + s
        q = li[0].k[:, rng.integers(0, pos, G)].reshape(H * G, 128)[None]  # earlier keys as queries
        o = torch.empty((1, H * G, 128), dtype=torch.float32, device="cuda")
        bg.bgtq_decode_step(plan, dev(q), dev(li[0].k[None, :, pos]), dev(li[0].v[None, :, pos]),
                            dev(np.array([pos], np.int32)), cache, dev(np.array([pos + 1], np.int32)), T, o, ws,
                            status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        got = o.cpu().numpy().astype(np.float64)[0]
        for h, hs in enumerate(heads):
            e = O.encode_head(hs, li[0].k[h][:pos + 1], li[0].v[h][:pos + 1])
            want = O.attention_recent(q[0][h * G:(h + 1) * G], e["khat"], e["vhat"], li[0].k[h][:pos + 1], W)
            check_close(got[h * G:(h + 1) * G], want)
