"""bgtq_decode_step (append the new token, then attend, in one launch) against
the two-call path and the oracle.

The fused step must write exactly the codes, norms and V pair records that
bgtq_quantize_append writes for that token (bit-exact), and its attention
output must equal bgtq_decode_attn's on the same cache (bit for bit: the
kernels share the attention code and the merge order) and the oracle's
float64 attention within the usual tolerance.  Source: the packed-cache
serving path of "RoPE-Aware Bit Allocation for KV-Cache Quantization"
(English abstract; review §1 "Packed-Cache", Figure 2): each decode step
appends the new token's compressed K/V and attends on the compressed cache.
"""

import numpy as np
import pytest

import rope_aware_quantized_gb300 as bg
from rope_aware_quantized_gb300 import workloads

from tests.test_gpu_parity import build, cache_arrays, check_close, dev, oracle_out, oracle_layer

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def prefill(plan, cache, li, lens):
    """Append tokens [0, lens[b]) of every sequence (one call per sequence length group)."""
    for b, n in enumerate(lens):
        if n <= 0:
            continue
        view = cache.sequence_view(b)
        k = dev(li[b].k[None, :, :n])
        v = dev(li[b].v[None, :, :n])
        bg.bgtq_quantize_append(plan, k, v, dev(np.array([0], np.int32)), view)


def new_token(li, pos):
    k = np.stack([l.k[:, p] for l, p in zip(li, pos)])  # [B][H][128]
    v = np.stack([l.v[:, p] for l, p in zip(li, pos)])
    return k, v


def two_calls(plan, cache, q, k_new, v_new, pos, seq, max_len):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bgtq_quantize_append(plan, dev(k_new[:, :, None]), dev(v_new[:, :, None]), dev(pos), cache, status=st)
    ws = torch.zeros(bg.bgtq_decode_attn_workspace(plan, q.shape[0], max_len), dtype=torch.uint8, device="cuda")
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    bg.bgtq_decode_attn(plan, q, cache, dev(seq), max_len, out, ws, status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), int(st.item())


def fused(plan, cache, q, k_new, v_new, pos, seq, max_len, out_dtype=torch.float32):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(bg.bgtq_decode_attn_workspace(plan, q.shape[0], max_len), dtype=torch.uint8, device="cuda")
    out = torch.empty(q.shape, dtype=out_dtype, device="cuda")
    bg.bgtq_decode_step(plan, q, dev(k_new), dev(v_new), dev(pos), cache, dev(seq), max_len, out, ws, status=st)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), int(st.item())


@pytest.mark.parametrize("H,G,T,bits_per_key,v_bits,s_ln", [
    (2, 8, 3001, 384, 3, 1.2),   # new token at an even position
    (2, 8, 3000, 384, 3, 1.2),   # odd position: merges into the pair record of token 2998
    (3, 4, 2049, 256, 2, 1.2),
    (2, 1, 700, 128, 1, 1.2),
    (2, 3, 998, 256, 4, 1.5),
    (1, 8, 65, 384, 3, 1.0),     # the new token opens the second 64-token step
    (1, 2, 1, 384, 3, 1.0),      # the new token is the whole sequence
])
def test_fused_step_equals_append_then_attend(H, G, T, bits_per_key, v_bits, s_ln):
    li, plan, cache_a, heads = build(500 + T, H, G, T, bits_per_key, v_bits, s_ln=s_ln)
    cache_b = bg.Cache(plan, 1, cache_a.capacity)
    prefill(plan, cache_a, li, [T - 1])
    prefill(plan, cache_b, li, [T - 1])
    pos = np.array([T - 1], np.int32)
    seq = np.array([T], np.int32)
    k_new, v_new = new_token(li, pos)
    q = dev(li[0].q[None])
    want_two, st_a = two_calls(plan, cache_a, q, k_new, v_new, pos, seq, T)
    got, st_b = fused(plan, cache_b, q, k_new, v_new, pos, seq, T)
    assert st_a == 0 and st_b == 0
    bk, bv = bits_per_key // 128, v_bits
    for a, b in zip(cache_arrays(plan, cache_a, H, bk, bv), cache_arrays(plan, cache_b, H, bk, bv)):
        assert np.array_equal(a, b)
    assert np.array_equal(got, want_two)
    check_close(got[0], oracle_out(heads, li[0], li[0].q, T, G))


def test_fused_step_ragged_batch_rewrites_and_empty_sequences():
    """Per-sequence positions: the usual last position, a rewrite of an
    earlier position (the attention sees the new token there), a position
    beyond the attended length (appended, not attended) and an empty
    sequence whose new token is stored but the output is zero."""
    H, G, T = 2, 4, 1500
    li, plan, cache_a, heads = build(640, H, G, T, 256, 2, s_ln=1.2, batch=4, cap=1500)
    cache_b = bg.Cache(plan, 4, 1500)
    lens = [900, 1200, 400, 0]
    prefill(plan, cache_a, li, lens)
    prefill(plan, cache_b, li, lens)
    pos = np.array([900, 611, 1000, 0], np.int32)
    seq = np.array([901, 1200, 400, 0], np.int32)
    # the rewritten token of sequence 1 takes the key/value of token 1300
    k_new, v_new = new_token(li, [900, 1300, 1000, 0])
    q = dev(np.stack([l.q for l in li]))
    want_two, st_a = two_calls(plan, cache_a, q, k_new, v_new, pos, seq, 1500)
    got, st_b = fused(plan, cache_b, q, k_new, v_new, pos, seq, 1500)
    assert st_a == 0 and st_b == 0
    for a, b in zip(cache_arrays(plan, cache_a, H, 2, 2), cache_arrays(plan, cache_b, H, 2, 2)):
        assert np.array_equal(a, b)
    assert np.array_equal(got, want_two)
    assert np.all(got[3] == 0)
    # oracle: sequence 0 attends tokens 0..900, sequence 2 tokens 0..399
    check_close(got[0], oracle_out(heads, li[0], li[0].q, 901, G))
    check_close(got[2], oracle_out(heads, li[2], li[2].q, 400, G))


def test_fused_step_position_beyond_capacity_is_flagged_and_skipped():
    H, G, T = 1, 4, 128
    li, plan, cache, heads = build(7, H, G, T, 384, 3, cap=128)
    prefill(plan, cache, li, [T])
    before = [x.copy() for x in cache_arrays(plan, cache, H, 3, 3)]
    k_new, v_new = new_token(li, [5])
    got, st = fused(plan, cache, dev(li[0].q[None]), k_new, v_new, np.array([128], np.int32),
                    np.array([T], np.int32), T)
    assert st & bg.STATUS_APPEND_CAPACITY
    for a, b in zip(before, cache_arrays(plan, cache, H, 3, 3)):
        assert np.array_equal(a, b)
    check_close(got[0], oracle_out(heads, li[0], li[0].q, T, G))


def test_fused_step_full_size_qwen_layer_sampled():
    """The benchmark's per-layer step (131072 cached tokens, K3V3, 2 KV heads
    x 8 query heads) in the launch configuration the benchmark times."""
    w = workloads.WORKLOADS["qwen3b_36l_128k"]
    max_len = int(w.seq_lens().max())
    ls = workloads.build_layer(w, 3, keep_host=[(0, 0), (0, 1)])
    ws = torch.zeros(bg.bgtq_decode_attn_workspace(ls.plan, w.batch, max_len), dtype=torch.uint8, device="cuda")
    out = torch.empty(ls.q.shape, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bgtq_decode_step(ls.plan, ls.q, ls.new_k[:, :, 0].contiguous(), ls.new_v[:, :, 0].contiguous(), ls.pos_new,
                        ls.cache, ls.seq_lens, max_len, out, ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    got = out.cpu().numpy().astype(np.float64)
    for b, h in [(0, 0), (0, 1)]:
        check_close(got[b, h * w.group:(h + 1) * w.group], oracle_layer(w, 3, ls, b, h))
