"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Required agreement: allocation, packed codes, norms and dequantised values
bit-exact; attention within max-abs 2e-3 and relative L2 1e-3 of the
oracle's float64 attention over its own dequantised cache (the packed-cache
path must equal attention on the compressed cache: "RoPE-Aware Bit
Allocation for KV-Cache Quantization", English abstract, packed-cache serving
path).  Inputs are seeded synthetic tensors; the oracle encodes the same fp16
keys/values itself and never sees a CUDA result.
"""

import math

import numpy as np
import pytest

import rope_aware_quantized_gb300 as bg
from oracle import bgtq_oracle as O
from rope_aware_quantized_gb300 import synth, workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MAX_ABS = 2e-3
REL_L2 = 1e-3


def dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return t if dtype is None else t.to(dtype)


def build(seed, H, G, T, bits_per_key, v_bits, base=1e4, s_ln=1.0, layout=0, cap=None, batch=1):
    """Numpy inputs for `batch` sequences of T tokens, a plan and an empty cache."""
    li = [synth.layer_inputs(seed + 17 * b, 0, H, G, T, base, s_ln, rope_layout=layout) for b in range(batch)]
    bits, en = [], []
    for h in range(H):
        b, e = bg.bgtq_alloc_bits(li[0].calib[h], bits_per_key, 8, layout)
        bits.append(b)
        en.append(e)
    pseed = 0xABCDEF + seed
    plan = bg.bgtq_plan_create(np.stack(bits), np.stack(en), G, bits_per_key, v_bits, pseed, layout)
    cache = bg.Cache(plan, batch, cap or T + (T % 2))
    heads = [O.head_state(li[0].calib[h], bits_per_key, v_bits, pseed, h, rope_layout=layout) for h in range(H)]
    return li, plan, cache, heads


def append(plan, cache, li, t0, t1, batch=None):
    batch = batch or len(li)
    k = np.stack([l.k[:, t0:t1] for l in li[:batch]])
    v = np.stack([l.v[:, t0:t1] for l in li[:batch]])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bgtq_quantize_append(plan, dev(k), dev(v), dev(np.full(batch, t0, np.int32)), cache, status=status)
    return status


def cache_arrays(plan, cache, H, bk, bv):
    torch.cuda.synchronize()
    cap = cache.capacity
    kc = cache.k_codes.cpu().numpy().reshape(cache.batch, H, cap, 16 * bk)
    vc = cache.v_codes.cpu().numpy().reshape(cache.batch, H, cap // 2, 32 * bv)
    kn = cache.k_norm.cpu().numpy().reshape(cache.batch, H, cap)
    vn = cache.v_norm.cpu().numpy().reshape(cache.batch, H, cap)
    return kc, vc, kn, vn


def decode(plan, cache, q, seq_lens, max_len, out_dtype=torch.float32):
    ws = torch.zeros(bg.bgtq_decode_attn_workspace(plan, q.shape[0], max_len), dtype=torch.uint8, device="cuda")
    out = torch.empty(q.shape, dtype=out_dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bgtq_decode_attn(plan, q, cache, seq_lens, max_len, out, ws, status=status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), int(status.item())


def half_ulp16(x):
    """Half a binary16 ulp at |x|: the most that rounding an fp32 result to
    an fp16 output adds (round to nearest)."""
    return np.spacing(np.abs(np.asarray(x)).astype(np.float16)).astype(np.float64) / 2


def check_close(got, want, extra_abs=0.0, fp16_out=False):
    """The attention tolerance (max-abs MAX_ABS, relative L2 REL_L2); an fp16
    output may differ by half a binary16 ulp more, element by element."""
    err = np.abs(got - want)
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    bound = MAX_ABS + extra_abs + (half_ulp16(want) if fp16_out else 0.0)
    assert (err <= bound).all(), f"max abs {err.max():.3e}, worst excess {(err - bound).max():.3e}"
    assert rel <= REL_L2, f"rel l2 {rel:.3e}"


# ----------------------------------------------------------------------------- codec parity (bit-exact)

@pytest.mark.parametrize("bits_per_key,v_bits,layout,s_ln", [(384, 3, 0, 1.0), (256, 2, 0, 1.2), (128, 1, 0, 1.2),
                                                             (384, 2, 1, 1.2), (512, 4, 0, 0.8), (256, 5, 0, 1.5)])
def test_quantize_append_codes_norms_bit_exact(bits_per_key, v_bits, layout, s_ln):
    H, G, T = 2, 4, 1003
    li, plan, cache, heads = build(31 + bits_per_key + v_bits, H, G, T, bits_per_key, v_bits, s_ln=s_ln, layout=layout)
    st = append(plan, cache, li, 0, T)
    assert st.item() == 0
    bk = bits_per_key // 128
    kc, vc, kn, vn = cache_arrays(plan, cache, H, bk, v_bits)
    for h in range(H):
        enc = O.encode_head(heads[h], li[0].k[h], li[0].v[h])
        assert np.array_equal(kn[0, h, :T], enc["krho"])
        assert np.array_equal(vn[0, h, :T], enc["vrho"])
        assert np.array_equal(kc[0, h, :T], enc["krec"])
        # complete V pair records bit-exact; the trailing half record: even half
        full = T // 2
        assert np.array_equal(vc[0, h, :full], enc["vrec"][:full])
        got = O.unpack_v(vc[0, h, : (T + 1) // 2], v_bits, T)
        assert np.array_equal(got, enc["vcodes"])


def test_dequant_debug_bit_exact():
    H, G, T = 2, 4, 517
    li, plan, cache, heads = build(5, H, G, T, 384, 3, s_ln=1.2)
    append(plan, cache, li, 0, T)
    for h in range(H):
        enc = O.encode_head(heads[h], li[0].k[h], li[0].v[h])
        for cd in (False, True):
            ko = torch.empty((T, 128), dtype=torch.float32, device="cuda")
            vo = torch.empty_like(ko)
            bg.bgtq_dequant_debug(plan, cache, 0, h, 0, T, ko, vo, codec_domain=cd)
            torch.cuda.synchronize()
            if cd:
                want_k = O.dequant(enc["kcodes"], enc["krho"], heads[h].kc, codec_domain=True)
                want_v = O.dequant(enc["vcodes"], enc["vrho"], heads[h].vc, codec_domain=True)
            else:
                want_k, want_v = enc["khat"], enc["vhat"]
            assert np.array_equal(ko.cpu().numpy(), want_k)
            assert np.array_equal(vo.cpu().numpy(), want_v)


@pytest.mark.parametrize("cuts", [[0, 37, 38, 200, 301], [0, 1, 2, 3, 300, 301], [0, 150, 151, 301]])
def test_chunked_appends_with_odd_starts_equal_one_shot(cuts):
    H, G, T = 3, 2, 301
    li, plan, cache, heads = build(8, H, G, T, 256, 2, s_ln=1.2, cap=302)
    for a, b in zip(cuts[:-1], cuts[1:]):
        assert append(plan, cache, li, a, b).item() == 0
    kc, vc, kn, vn = cache_arrays(plan, cache, H, 2, 2)
    for h in range(H):
        enc = O.encode_head(heads[h], li[0].k[h], li[0].v[h])
        assert np.array_equal(kc[0, h, :T], enc["krec"])
        assert np.array_equal(O.unpack_v(vc[0, h, :151], 2, T), enc["vcodes"])
        assert np.array_equal(vn[0, h, :T], enc["vrho"])


def test_append_capacity_status_and_skip():
    H, G, T = 1, 4, 64
    li, plan, cache, heads = build(9, H, G, T, 384, 3, cap=64)
    append(plan, cache, li, 0, 60)
    before = cache.k_codes.clone()
    k = dev(li[0].k[None, :, :8])
    v = dev(li[0].v[None, :, :8])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bgtq_quantize_append(plan, k, v, dev(np.array([60], np.int32)), cache, status=st)
    torch.cuda.synchronize()
    assert st.item() & bg.STATUS_APPEND_CAPACITY
    assert torch.equal(before, cache.k_codes)


# ----------------------------------------------------------------------------- attention parity

def oracle_out(heads, li_b, q_b, seqlen, G, scale=1 / math.sqrt(128)):
    outs = []
    for h, hs in enumerate(heads):
        enc = O.encode_head(hs, li_b.k[h][:seqlen], li_b.v[h][:seqlen])
        outs.append(O.attention(q_b[h * G:(h + 1) * G], enc["khat"], enc["vhat"], scale))
    return np.concatenate(outs, axis=0)


@pytest.mark.parametrize("H,G,T,bits_per_key,v_bits,s_ln,qscale", [
    (1, 4, 4096, 384, 3, 1.0, 1.0),     # tiny workload shape, peaked (queries drawn like keys)
    (1, 4, 4096, 384, 3, 1.0, 0.05),    # same, non-peaked softmax
    (2, 8, 3000, 384, 3, 1.2, 1.0),     # Qwen-like group of 8
    (2, 8, 2500, 384, 2, 1.2, 0.1),
    (3, 4, 2049, 256, 2, 1.2, 1.0),     # Llama-like K2V2, ragged tail
    (2, 1, 700, 128, 1, 1.2, 0.3),      # K1V1, one query head per KV head
    (2, 3, 999, 256, 4, 1.5, 0.2),      # V4, odd group
    (1, 8, 64, 384, 3, 1.0, 1.0),       # exactly one CTA step
    (1, 2, 17, 384, 3, 1.0, 1.0),       # shorter than one warp tile
])
def test_decode_attention_matches_oracle(H, G, T, bits_per_key, v_bits, s_ln, qscale):
    li, plan, cache, heads = build(41 + T, H, G, T, bits_per_key, v_bits, s_ln=s_ln)
    append(plan, cache, li, 0, T)
    q = (li[0].q.astype(np.float32) * qscale).astype(np.float16)
    got, st = decode(plan, cache, dev(q[None]), dev(np.array([T], np.int32)), T)
    assert st == 0
    want = oracle_out(heads, li[0], q, T, G)
    check_close(got[0], want)


def test_decode_fp16_output_and_split_invariance():
    H, G, T = 2, 8, 5000
    li, plan, cache, heads = build(77, H, G, T, 384, 3, s_ln=1.2, cap=20000)
    append(plan, cache, li, 0, T)
    q = dev(li[0].q[None])
    lens = dev(np.array([T], np.int32))
    want = oracle_out(heads, li[0], li[0].q, T, G)
    outs = []
    for max_len in (T, 8192, 20000):     # different split counts
        got, _ = decode(plan, cache, q, lens, max_len)
        check_close(got[0], want)
        outs.append(got[0])
    assert np.abs(outs[0] - outs[2]).max() < 1e-4
    got16, _ = decode(plan, cache, q, lens, T, out_dtype=torch.float16)
    check_close(got16[0], want, fp16_out=True)


@pytest.mark.parametrize("qmul", [60.0, 1e-3])
def test_decode_extreme_query_magnitudes(qmul):
    """Whitening moves a block's scale into the query: sigma * q can leave the
    fp16 range; the kernel must stay finite and accurate at both extremes."""
    H, G, T = 1, 8, 900
    li, plan, cache, heads = build(123, H, G, T, 384, 3, s_ln=1.5)
    append(plan, cache, li, 0, T)
    q = np.clip(li[0].q.astype(np.float64) * qmul, -60000, 60000).astype(np.float16)
    got, _ = decode(plan, cache, dev(q[None]), dev(np.array([T], np.int32)), T)
    assert np.all(np.isfinite(got))
    check_close(got[0], oracle_out(heads, li[0], q, T, G))


@pytest.mark.parametrize("vmul", [0.01, 100.0])
def test_decode_value_magnitudes(vmul):
    """P' = p * rho_V enters the tensor cores as fp16 hi + lo: value norms two
    decades below and above unit scale must stay accurate (no fp16
    subnormals or overflow in the weights).  The bound is the stated
    absolute one even for values scaled by 100: the hi + lo weights carry
    about fp32 precision, so only float32 rounding is left."""
    H, G, T = 2, 8, 2000
    li, plan, cache, heads = build(321, H, G, T, 384, 3, s_ln=1.2)
    li = [synth.LayerInputs(li[0].k, (li[0].v.astype(np.float64) * vmul).astype(np.float16), li[0].q,
                            li[0].calib, li[0].sigma)]
    append(plan, cache, li, 0, T)
    for qmul in (1.0, 0.05):  # peaked and flat softmax
        q = (li[0].q.astype(np.float32) * qmul).astype(np.float16)
        got, st = decode(plan, cache, dev(q[None]), dev(np.array([T], np.int32)), T)
        assert st == 0 and np.all(np.isfinite(got))
        want = oracle_out(heads, li[0], q, T, G)
        err = np.abs(got[0] - want)
        rel = np.linalg.norm(got[0] - want) / np.linalg.norm(want)
        assert err.max() <= MAX_ABS, f"max abs {err.max():.3e}"
        assert rel <= REL_L2, f"rel l2 {rel:.3e}"


def test_decode_ragged_batch_with_empty_and_single_token_sequences():
    H, G, T = 2, 4, 1500
    li, plan, cache, heads = build(90, H, G, T, 256, 2, s_ln=1.2, batch=4, cap=1500)
    append(plan, cache, li, 0, T)
    lens = np.array([1, 0, 777, 1500], np.int32)
    q = np.stack([l.q for l in li])
    got, st = decode(plan, cache, dev(q), dev(lens), 1500)
    assert st == 0
    for b in range(4):
        if lens[b] == 0:
            assert np.all(got[b] == 0)
            continue
        check_close(got[b], oracle_out(heads, li[b], q[b], int(lens[b]), G))


def test_decode_capacity_not_multiple_of_four():
    """Per-head norm rows then start 8 bytes off a 16-byte boundary."""
    H, G, T = 3, 4, 1001
    li, plan, cache, heads = build(21, H, G, T, 384, 3, s_ln=1.2, cap=1002)
    append(plan, cache, li, 0, T)
    got, st = decode(plan, cache, dev(li[0].q[None]), dev(np.array([T], np.int32)), T)
    assert st == 0
    check_close(got[0], oracle_out(heads, li[0], li[0].q, T, G))


def test_decode_seq_len_beyond_capacity_is_clamped_and_flagged():
    H, G, T = 1, 4, 128
    li, plan, cache, heads = build(3, H, G, T, 384, 3, cap=128)
    append(plan, cache, li, 0, T)
    got, st = decode(plan, cache, dev(li[0].q[None]), dev(np.array([500], np.int32)), 128)
    assert st & bg.STATUS_SEQLEN_CAPACITY
    check_close(got[0], oracle_out(heads, li[0], li[0].q, T, G))


def test_decode_is_token_order_invariant():
    """Permuting cached tokens leaves the output unchanged (LogQuant summary, §4)."""
    H, G, T = 1, 4, 1024
    li, plan, cache, heads = build(12, H, G, T, 384, 3)
    perm = np.random.default_rng(0).permutation(T)
    li_p = [synth.LayerInputs(li[0].k[:, perm], li[0].v[:, perm], li[0].q, li[0].calib, li[0].sigma)]
    cache2 = bg.Cache(plan, 1, T)
    append(plan, cache, li, 0, T)
    append(plan, cache2, li_p, 0, T)
    a, _ = decode(plan, cache, dev(li[0].q[None]), dev(np.array([T], np.int32)), T)
    b, _ = decode(plan, cache2, dev(li[0].q[None]), dev(np.array([T], np.int32)), T)
    assert np.abs(a - b).max() < 1e-4


# ----------------------------------------------------------------------------- full-size workloads

def decode_step(ls, w, max_len):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bgtq_quantize_append(ls.plan, ls.new_k, ls.new_v, ls.pos_new, ls.cache, status=st)
    got, st2 = decode(ls.plan, ls.cache, ls.q, ls.seq_lens, max_len)
    assert st.item() == 0 and st2 == 0
    return got


def oracle_layer(w, layer, ls, b, h):
    hs = O.head_state(workloads.calib_keys(w, layer, h), w.bits_per_key, w.v_bits, workloads.plan_seed(w, layer), h)
    k, v = ls.host[(b, h)]
    enc = O.encode_head(hs, k, v)
    q = ls.q[b, h * w.group:(h + 1) * w.group].cpu().numpy()
    return O.attention(q, enc["khat"], enc["vhat"])


@pytest.mark.parametrize("name,layers,samples", [
    ("tiny", [0], [(0, 0)]),
    ("llama8b_layer", [0], [(0, 0), (0, 7)]),
    ("qwen3b_36l_128k", [0, 35], [(0, 0), (0, 1)]),
    ("qwen3b_36l_512k", [17], [(0, 1)]),
    ("llama8b_ragged_b32", [0], [(0, 3), (31, 0)]),
])
def test_full_size_workloads_sampled_against_oracle(name, layers, samples):
    w = workloads.WORKLOADS[name]
    lens = w.seq_lens()
    max_len = int(lens.max())
    for layer in layers:
        ls = workloads.build_layer(w, layer, keep_host=samples)
        got = decode_step(ls, w, max_len)
        assert np.all(np.isfinite(got))
        for b, h in samples:
            want = oracle_layer(w, layer, ls, b, h)
            check_close(got[b, h * w.group:(h + 1) * w.group], want)
        del ls
        torch.cuda.empty_cache()
