"""GPU: the paged ragged cache (pools of P-token pages and a per-sequence page
table) against the contiguous cache and the oracle.

Paging moves records, never their contents: with the same appends, every
record and norm gathered through the page table must equal the contiguous
cache's bit for bit, decode outputs must be identical, and both must match
the oracle's attention within the decode tolerance.  Page tables are random
permutations of a pool with spare pages, so neighbouring positions of a
sequence live in unrelated pages.
"""

import numpy as np
import pytest

import rope_aware_quantized_gb300 as bg
from oracle import bgtq_oracle as O
from rope_aware_quantized_gb300 import synth

from tests.test_gpu_parity import check_close, decode, dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def setup(seed, H, G, lens, P, bits_per_key=384, v_bits=3, recent=0, spare=3):
    B, T = len(lens), max(lens)
    li = [synth.layer_inputs(seed + 17 * b, 0, H, G, T, 1e5, 1.2) for b in range(B)]
    be = [bg.bgtq_alloc_bits(li[0].calib[h], bits_per_key) for h in range(H)]
    pseed = 0x9A6E + seed
    plan = bg.bgtq_plan_create(np.stack([b for b, _ in be]), np.stack([e for _, e in be]), G, bits_per_key, v_bits,
                               pseed)
    cap = -(-(T + 2) // P) * P
    cont = bg.Cache(plan, B, cap, recent=recent)
    n_pages = B * (cap // P) + spare
    paged = bg.Cache(plan, B, cap, recent=recent, page_tokens=P, n_pages=n_pages)
    perm = np.random.default_rng(seed).permutation(n_pages)[:B * (cap // P)].astype(np.int32)
    paged.page_table.copy_(dev(perm.reshape(B, cap // P)))
    heads = [O.head_state(li[0].calib[h], bits_per_key, v_bits, pseed, h) for h in range(H)]
    return li, plan, cont, paged, heads


def append_ragged(plan, cache, li, lens, chunks):
    """Sequence b gets its first lens[b] tokens in chunks of the given sizes
    (the rest in one final chunk), each through its own batch-1 view."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for b, n in enumerate(lens):
        view = cache.sequence_view(b)
        t = 0
        for c in list(chunks) + [n]:
            c = min(c, n - t)
            if c <= 0:
                break
            bg.bgtq_quantize_append(plan, dev(li[b].k[None, :, t:t + c]), dev(li[b].v[None, :, t:t + c]),
                                    dev(np.array([t], np.int32)), view, status=st)
            t += c
    torch.cuda.synchronize()
    return int(st.item())


def gathered(plan, cache, H, lens, bk, bv):
    """Records and norms of every (b, h, pos < lens[b]) in position order."""
    P = cache.page_tokens
    kc = cache.k_codes.cpu().numpy()
    vc = cache.v_codes.cpu().numpy()
    kn = cache.k_norm.cpu().numpy()
    vn = cache.v_norm.cpu().numpy()
    pt = cache.page_table.cpu().numpy() if P else None
    out = []
    for b, n in enumerate(lens):
        pos = np.arange(n)
        for h in range(H):
            if P:
                sl = (pt[b][pos // P].astype(np.int64) * H + h) * P + pos % P
            else:
                sl = (b * H + h) * cache.capacity + pos
            krec = kc.reshape(-1, 16 * bk)[sl]
            vrec = vc.reshape(-1, 32 * bv)[sl[::2] // 2]
            out.append((krec, vrec, kn[sl], vn[sl]))
    return out


@pytest.mark.parametrize("P,lens,chunks", [
    (16, [300, 45, 129], (64, 1, 1, 37)),     # bulk then warp appends, pages smaller than a split
    (64, [1000, 777], (200, 3, 64)),
    (256, [2049, 1, 513], (1024, 1)),         # a one-token sequence; odd lengths
])
def test_paged_records_and_decode_equal_contiguous(P, lens, chunks):
    H, G = 2, 8
    li, plan, cont, paged, heads = setup(7 + P, H, G, lens, P)
    assert append_ragged(plan, cont, li, lens, chunks) == 0
    assert append_ragged(plan, paged, li, lens, chunks) == 0
    for a, b in zip(gathered(plan, cont, H, lens, 3, 3), gathered(plan, paged, H, lens, 3, 3)):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)
    q = np.stack([l.q for l in li])
    seq = dev(np.array(lens, np.int32))
    got_c, st_c = decode(plan, cont, dev(q), seq, max(lens))
    got_p, st_p = decode(plan, paged, dev(q), seq, max(lens))
    assert st_c == 0 and st_p == 0
    assert np.array_equal(got_c, got_p)
    for b, n in enumerate(lens):
        want = np.concatenate([O.attention(q[b][h * G:(h + 1) * G], *(lambda e: (e["khat"], e["vhat"]))(
            O.encode_head(hs, li[b].k[h][:n], li[b].v[h][:n]))) for h, hs in enumerate(heads)])
        check_close(got_p[b], want)


def test_paged_fused_step_and_recent_buffer():
    """bgtq_decode_step on a paged cache with an fp16 recent-key buffer equals
    the same step on a contiguous cache, cache and output."""
    H, G, P, W = 2, 8, 32, 40
    lens = [700, 90]
    li, plan, cont, paged, heads = setup(91, H, G, lens, P, recent=W)
    pre = [n - 1 for n in lens]
    append_ragged(plan, cont, li, pre, (128,))
    append_ragged(plan, paged, li, pre, (128,))
    q = dev(np.stack([l.q for l in li]))
    k_new = dev(np.stack([l.k[:, n - 1] for l, n in zip(li, lens)]))
    v_new = dev(np.stack([l.v[:, n - 1] for l, n in zip(li, lens)]))
    pos = dev(np.array(pre, np.int32))
    seq = dev(np.array(lens, np.int32))
    outs = []
    for c in (cont, paged):
        ws = torch.zeros(bg.bgtq_decode_attn_workspace(plan, 2, max(lens)), dtype=torch.uint8, device="cuda")
        out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        bg.bgtq_decode_step(plan, q, k_new, v_new, pos, c, seq, max(lens), out, ws, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        outs.append(out.cpu().numpy().astype(np.float64))
    assert np.array_equal(outs[0], outs[1])
    assert torch.equal(cont.k_recent, paged.k_recent)
    for a, b in zip(gathered(plan, cont, H, lens, 3, 3), gathered(plan, paged, H, lens, 3, 3)):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)
    for b, n in enumerate(lens):
        want = []
        for h, hs in enumerate(heads):
            e = O.encode_head(hs, li[b].k[h][:n], li[b].v[h][:n])
            want.append(O.attention_recent(li[b].q[h * G:(h + 1) * G], e["khat"], e["vhat"], li[b].k[h][:n], W))
        check_close(outs[1][b], np.concatenate(want))


def test_paged_dequant_debug_equals_contiguous():
    H, G, P = 2, 4, 16
    lens = [333]
    li, plan, cont, paged, heads = setup(5, H, G, lens, P, bits_per_key=256, v_bits=2)
    append_ragged(plan, cont, li, lens, (100,))
    append_ragged(plan, paged, li, lens, (100,))
    for h in range(H):
        outs = []
        for c in (cont, paged):
            ko = torch.empty((333, 128), dtype=torch.float32, device="cuda")
            vo = torch.empty_like(ko)
            bg.bgtq_dequant_debug(plan, c, 0, h, 0, 333, ko, vo)
            outs.append((ko, vo))
        torch.cuda.synchronize()
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_page_index_out_of_range_is_flagged_and_contained():
    """A page table entry outside [0, n_pages) is flagged by append and
    decode; the other sequence of the batch is unaffected."""
    H, G, P = 2, 8, 64
    lens = [500, 400]
    li, plan, cont, paged, heads = setup(33, H, G, lens, P, spare=0)
    pt = paged.page_table.cpu().numpy()
    pt[1, 2] = paged.n_pages + 5        # positions 128..191 of sequence 1
    paged.page_table.copy_(dev(pt))
    assert append_ragged(plan, cont, li, lens, (256,)) == 0
    assert append_ragged(plan, paged, li, lens, (256,)) & bg.STATUS_PAGE_RANGE
    q = np.stack([l.q for l in li])
    seq = dev(np.array(lens, np.int32))
    got_c, _ = decode(plan, cont, dev(q), seq, max(lens))
    got_p, st = decode(plan, paged, dev(q), seq, max(lens))
    assert st & bg.STATUS_PAGE_RANGE
    assert np.array_equal(got_c[0], got_p[0])


def test_paged_full_size_decode_equals_contiguous():
    """The bench's layer shape (2 KV heads x 8 query heads, 131072 cached
    tokens, K3V3) with 256-token pages in a shuffled pool: decode output
    identical to the contiguous cache's, in the launch configuration the
    bench uses."""
    from rope_aware_quantized_gb300 import workloads
    w = workloads.WORKLOADS["qwen3b_36l_128k"]
    a = workloads.build_layer(w, 0)
    b = workloads.build_layer(w, 0, page_tokens=256)
    assert not torch.equal(b.cache.page_table.view(-1).cpu(), torch.arange(b.cache.page_table.numel(),
                                                                            dtype=torch.int32))
    outs = []
    for ls in (a, b):
        ws = torch.zeros(bg.bgtq_decode_attn_workspace(ls.plan, w.batch, 131072), dtype=torch.uint8, device="cuda")
        out = torch.empty((w.batch, w.n_q, 128), dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        bg.bgtq_decode_step(ls.plan, ls.q, ls.new_k[:, :, 0], ls.new_v[:, :, 0], ls.pos_new, ls.cache, ls.seq_lens,
                            131072, out, ws, status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        outs.append(out.cpu())
    assert torch.equal(outs[0], outs[1])


def test_paged_general_instance_noalloc_and_fidelity():
    """Explicit widths with wide codes in many slots (the general decode
    path) on a paged cache with a recent-key buffer: decode (workspace and
    no-alloc entry points) and the logit-fidelity kernel equal the
    contiguous cache's results (decode bit for bit)."""
    H, G, T, P, W = 2, 8, 1500, 64, 100
    li = synth.layer_inputs(404, 0, H, G, T, 1e5, 1.2)
    energy = np.stack([bg.bgtq_alloc_bits(li.calib[h], 384)[1] for h in range(H)])
    bits = np.zeros((H, 64), np.uint8)
    bits[0, :24] = 8
    bits[1, 40:] = 8
    plan = bg.bgtq_plan_create(bits, energy, G, 384, 3, 0xBADC0DE)
    cap = -(-T // P) * P
    cont = bg.Cache(plan, 1, cap, recent=W)
    paged = bg.Cache(plan, 1, cap, recent=W, page_tokens=P, n_pages=cap // P + 2)
    perm = np.random.default_rng(8).permutation(paged.n_pages)[:cap // P].astype(np.int32)
    paged.page_table.copy_(dev(perm.reshape(1, -1)))
    k, v = dev(li.k[None]), dev(li.v[None])
    for c in (cont, paged):
        bg.bgtq_quantize_append(plan, k, v, dev(np.array([0], np.int32)), c)
    q = dev(li.q[None])
    seq = dev(np.array([T], np.int32))
    res = []
    for c in (cont, paged):
        a, st = decode(plan, c, q, seq, T)
        assert st == 0
        out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        bg.bgtq_decode_attn_noalloc(plan, q, c, seq, T, out, status=st2)
        mae = torch.empty((1, H * G), dtype=torch.float32, device="cuda")
        bg.bgtq_logit_mae(plan, q, k, c, T, mae)
        torch.cuda.synchronize()
        assert st2.item() == 0
        res.append((a, out.cpu().numpy().astype(np.float64), mae.cpu().numpy()))
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])
    assert np.array_equal(res[1][0], res[1][1])
    # the fidelity kernel sums per-block partials with float atomics, whose
    # order varies from run to run: equal up to that summation order
    assert np.allclose(res[0][2], res[1][2], rtol=1e-5, atol=0)
