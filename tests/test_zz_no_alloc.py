"""bgtq_decode_attn_noalloc: decode attention for callers that cannot
allocate device memory (fixed memory budgets, pools that must not be
bypassed, host runtimes without a device allocator).  It must give the same
result as bgtq_decode_attn with a caller workspace, call after call, even
though every call reuses the library's one built-in scratch array.

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.  It builds everything it needs itself, so
it also passes alone in a fresh process.
"""

import numpy as np
import pytest

import rope_aware_quantized_gb300 as bg
from rope_aware_quantized_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MAX_ABS = 2e-3
REL_L2 = 1e-3


def _setup(seed, H, G, T, batch, bits_per_key=384, v_bits=3):
    li = [synth.layer_inputs(seed + 7 * b, 0, H, G, T, 1e6, 1.2) for b in range(batch)]
    bits, en = zip(*[bg.bgtq_alloc_bits(li[0].calib[h], bits_per_key) for h in range(H)])
    plan = bg.bgtq_plan_create(np.stack(bits), np.stack(en), G, bits_per_key, v_bits, 0x51A7 + seed)
    cache = bg.Cache(plan, batch, T + (T % 2))
    k = torch.from_numpy(np.stack([l.k for l in li])).cuda()
    v = torch.from_numpy(np.stack([l.v for l in li])).cuda()
    bg.bgtq_quantize_append(plan, k, v, torch.zeros(batch, dtype=torch.int32, device="cuda"), cache)
    q = torch.from_numpy(np.stack([l.q for l in li])).cuda()
    return plan, cache, q, li


def _oracle_close(out, li, q, lens, H, G, seed, bits_per_key=384, v_bits=3):
    """The required tolerance against the oracle's float64 attention over its
    own encoding of the same keys and values."""
    import math

    from oracle import bgtq_oracle as O
    got = out.double().cpu().numpy()
    for b, l in enumerate(li):
        n = int(lens[b])
        for h in range(H):
            # the plan's widths come from sequence 0's calibration keys
            hs = O.head_state(li[0].calib[h], bits_per_key, v_bits, 0x51A7 + seed, h)
            enc = O.encode_head(hs, l.k[h][:n], l.v[h][:n])
            want = O.attention(q[b, h * G:(h + 1) * G], enc["khat"], enc["vhat"], 1 / math.sqrt(128))
            g = got[b, h * G:(h + 1) * G]
            assert np.abs(g - want).max() <= MAX_ABS
            assert np.linalg.norm(g - want) / np.linalg.norm(want) <= REL_L2


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    # two different problems, each run through both entry points; the
    # built-in scratch is reused call after call.  Both entry points run the
    # same kernel with the same split plan and merge order, so the outputs
    # must be identical bit for bit.
    cases = [(1, 2, 8, 20000, 1, np.array([20000], np.int32)),
             (2, 3, 4, 3000, 3, np.array([3000, 1, 1777], np.int32))]
    for seed, H, G, T, batch, lens in cases:
        plan, cache, q, li = _setup(seed, H, G, T, batch)
        seq = torch.from_numpy(lens).cuda()
        ws = torch.zeros(bg.bgtq_decode_attn_workspace(plan, batch, T), dtype=torch.uint8, device="cuda")
        ref = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        bg.bgtq_decode_attn(plan, q, cache, seq, T, ref, ws)
        for _ in range(2):
            out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            bg.bgtq_decode_attn_noalloc(plan, q, cache, seq, T, out, status=st)
            torch.cuda.synchronize()
            assert st.item() == 0
            assert torch.equal(out, ref)
        if seed == 2:  # the small case: also against the oracle
            _oracle_close(out, li, q.cpu().numpy(), lens, H, G, seed)


def test_noalloc_rejects_problems_beyond_the_built_in_scratch():
    import ctypes
    plan, cache, q, _ = _setup(4, 8, 4, 64, 1, bits_per_key=256, v_bits=2)
    seq = torch.full((1,), 64, dtype=torch.int32, device="cuda")
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    batch = 4096  # 32768 (sequence, head) units: far more merge scratch than 2 MiB
    # rejected on the host before anything is launched or read
    rc = bg.lib().bgtq_decode_attn_noalloc(plan.handle, None, q.data_ptr(), ctypes.byref(cache.desc),
                                           seq.data_ptr(), 64, batch, out.data_ptr(), 1, 0.125, None)
    assert rc == -4
    assert b"scratch" in bg.lib().bgtq_last_error()
