"""GPU: the prefill-side calls at the sizes and in the launch configuration
the benchmark times, checked on samples the oracle computes one by one.

* bgtq_quantize_append of a 131072-token prompt of the Qwen2.5-3B-shaped
  layer (2 KV heads, K3V3) in one call (the bulk kernel's grid of the
  benchmark's append measurement): the records and norms of sampled position
  ranges (start, middle, end; even-aligned, so V pair records are whole) equal
  the oracle's encoder bit for bit.
* bgtq_prefill_chunk_attn of an 8192-token chunk onto 32768 cached tokens of
  the same layer (16 query heads, fp16 output, the workspace sized by
  bgtq_prefill_chunk_workspace): the first row of every warp of every query
  block and the last row, of one query head per KV head, against the oracle's float64
  attention over the dequantised prefix and the chunk's own keys 0 .. i, within
  the decode tolerance (an fp16 output may differ by half a binary16 ulp more);
  the chunk's own records equal one append of them.
"""

import numpy as np
import pytest

import rope_aware_quantized_gb300 as bg
from oracle import bgtq_oracle as O
from rope_aware_quantized_gb300 import synth

from tests.test_gpu_parity import cache_arrays, check_close, dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

H, G, BPK, VB = 2, 8, 384, 3


def layer(seed, T):
    li = synth.layer_inputs(seed, 0, H, G, T, 1e6, 1.2)
    be = [bg.bgtq_alloc_bits(li.calib[h], BPK) for h in range(H)]
    pseed = 0x51E0 + seed
    plan = bg.bgtq_plan_create(np.stack([b for b, _ in be]), np.stack([e for _, e in be]), G, BPK, VB, pseed)
    heads = [O.head_state(li.calib[h], BPK, VB, pseed, h) for h in range(H)]
    return li, plan, heads


def check_records(kc, vc, kn, vn, heads, li, ranges, base=0):
    """Records and norms at cache positions base + [a, b) equal the oracle's
    encoding of tokens [a, b) of li (a, b even)."""
    for h, hs in enumerate(heads):
        for a, b in ranges:
            enc = O.encode_head(hs, li.k[h][a:b], li.v[h][a:b])
            assert np.array_equal(kc[0, h, base + a:base + b], enc["krec"]), (h, a)
            assert np.array_equal(kn[0, h, base + a:base + b], enc["krho"]), (h, a)
            assert np.array_equal(vn[0, h, base + a:base + b], enc["vrho"]), (h, a)
            assert np.array_equal(vc[0, h, (base + a) // 2:(base + b) // 2], enc["vrec"]), (h, a)


def test_bulk_append_of_a_131072_token_prompt_sampled_bit_exact():
    T = 131072
    li, plan, heads = layer(3, T)
    cache = bg.Cache(plan, 1, T)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bgtq_quantize_append(plan, dev(li.k[None]), dev(li.v[None]), torch.zeros(1, dtype=torch.int32, device="cuda"),
                            cache, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    kc, vc, kn, vn = cache_arrays(plan, cache, H, BPK // 128, VB)
    check_records(kc, vc, kn, vn, heads, li, [(0, 256), (T // 2 - 128, T // 2 + 128), (T - 256, T)])


def test_chunk_of_8192_onto_32768_cached_sampled_rows():
    P0, C = 32768, 8192
    li, plan, heads = layer(4, P0 + C)
    cache = bg.Cache(plan, 1, P0 + C)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bgtq_quantize_append(plan, dev(li.k[None, :, :P0]), dev(li.v[None, :, :P0]),
                            torch.zeros(1, dtype=torch.int32, device="cuda"), cache, status=st)
    # queries: keys of other positions of the same KV head
    rng = np.random.default_rng(11)
    q = np.empty((1, H * G, C, 128), np.float16)
    for h in range(H):
        for g in range(G):
            q[0, h * G + g] = li.k[h][rng.integers(0, P0 + C, C)]
    out = torch.full((1, H * G, C, 128), float("nan"), dtype=torch.float16, device="cuda")
    ws = torch.empty(bg.bgtq_prefill_chunk_workspace(plan, 1, P0), dtype=torch.uint8, device="cuda")
    bg.bgtq_prefill_chunk_attn(plan, dev(q), dev(np.ascontiguousarray(li.k[None, :, P0:])),
                               dev(np.ascontiguousarray(li.v[None, :, P0:])), dev(np.array([P0], np.int32)), cache, out,
                               max_prefix=P0, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    # the first row of every warp of every query block (a fault confined to one
    # warp's tensor-memory lanes shows in it), and the last row
    rows = list(range(0, C, 32)) + [C - 1]
    for h, hs in enumerate(heads):
        enc = O.encode_head(hs, li.k[h][:P0], li.v[h][:P0])
        gq = h * G + h  # query head h of KV head h
        for i in rows:
            keys = np.concatenate([enc["khat"], li.k[h][P0:P0 + i + 1].astype(np.float64)])
            vals = np.concatenate([enc["vhat"], li.v[h][P0:P0 + i + 1].astype(np.float64)])
            want = O.attention(q[0, gq, i][None], keys, vals)
            check_close(got[0, gq, i][None], want, fp16_out=True)
    # the chunk's records: an append of the chunk's tokens at P0
    kc, vc, kn, vn = cache_arrays(plan, cache, H, BPK // 128, VB)
    for h, hs in enumerate(heads):
        for a, b in [(P0, P0 + 256), (P0 + C - 256, P0 + C)]:
            enc = O.encode_head(hs, li.k[h][a:b], li.v[h][a:b])
            assert np.array_equal(kc[0, h, a:b], enc["krec"]), (h, a)
            assert np.array_equal(kn[0, h, a:b], enc["krho"]), (h, a)
            assert np.array_equal(vc[0, h, a // 2:b // 2], enc["vrec"]), (h, a)
