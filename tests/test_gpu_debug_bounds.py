"""GPU: the BGTQ_DEBUG_BOUNDS build of the library, in which every record
index (sequence, head, position against the capacity, page-table entry,
final slot) and the table indices are range-checked; a failed check ORs
BGTQ_STATUS_BOUNDS into the call's status word and skips the access, with
no trap.

The build is chosen per process (BGTQ_DEBUG_BOUNDS=1 in the environment), so
each case runs in a child process.  Every bad index below is one that the
default build also catches before any access (it reads page 0 in place of a
bad page, clamps a sequence length to the capacity, skips an append past
it), so neither build touches memory outside the cache.
"""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

APPEND_CAPACITY, SEQLEN_CAPACITY, PAGE_RANGE, BOUNDS = 1, 2, 4, 16

CHILD = r'''
import hashlib, json
import numpy as np, torch
import rope_aware_quantized_gb300 as bg
from rope_aware_quantized_gb300 import synth

H, G, T, P = 2, 4, 256, 32
li = synth.layer_inputs(3, 0, H, G, T, 1e4, 1.0)
be = [bg.bgtq_alloc_bits(li.calib[h], 384) for h in range(H)]
plan = bg.bgtq_plan_create(np.stack([b for b, _ in be]), np.stack([e for _, e in be]), G, 384, 3, 0x77)
k = torch.from_numpy(li.k[None]).cuda()
v = torch.from_numpy(li.v[None]).cuda()
q = torch.from_numpy(li.q[None]).cuda()
i32 = lambda *x: torch.tensor(x, dtype=torch.int32, device="cuda")
res = {"lib": bg._native.library_path()}

def decode(cache, seq):
    ws = torch.zeros(bg.bgtq_decode_attn_workspace(plan, 1, T), dtype=torch.uint8, device="cuda")
    out = torch.zeros(q.shape, dtype=torch.float32, device="cuda")
    st = i32(0)
    bg.bgtq_decode_attn(plan, q, cache, i32(seq), T, out, ws, status=st)
    torch.cuda.synchronize()
    return int(st.item()), out

# a clean paged cache: append, decode
cache = bg.Cache(plan, 1, T, page_tokens=P)
st = i32(0)
bg.bgtq_quantize_append(plan, k, v, i32(0), cache, status=st)
torch.cuda.synchronize()
res["clean_append"] = int(st.item())
res["clean_decode"], out = decode(cache, T)
res["clean_out"] = hashlib.sha256(out.cpu().numpy().tobytes()).hexdigest()
# a page-table entry past the pool
cache.page_table[0, 3] = cache.n_pages + 5
res["bad_page"], _ = decode(cache, T)
# a sequence length past the capacity (contiguous cache)
flat = bg.Cache(plan, 1, T)
bg.bgtq_quantize_append(plan, k, v, i32(0), flat)
res["bad_seq"], _ = decode(flat, T + 100)
# appends that would run past the capacity: the bulk kernel (64 tokens) and
# the warp kernel (2 tokens)
for name, n in (("bad_append_bulk", 64), ("bad_append_warp", 2)):
    st = i32(0)
    bg.bgtq_quantize_append(plan, k[:, :, :n].contiguous(), v[:, :, :n].contiguous(), i32(T - 1), flat, status=st)
    torch.cuda.synchronize()
    res[name] = int(st.item())
print(json.dumps(res))
'''


def run_child(debug: bool) -> dict:
    env = dict(os.environ, BGTQ_DEBUG_BOUNDS="1" if debug else "0", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stderr[-4000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.fixture(scope="module")
def both():
    return run_child(True), run_child(False)


def test_debug_bounds_build_flags_a_bad_page_and_capacity(both):
    d, _ = both
    assert d["lib"].endswith("libbgtq_debug_bounds.so")
    assert d["clean_append"] == 0 and d["clean_decode"] == 0
    assert d["bad_page"] == PAGE_RANGE | BOUNDS
    assert d["bad_seq"] == SEQLEN_CAPACITY | BOUNDS
    assert d["bad_append_bulk"] == APPEND_CAPACITY | BOUNDS
    assert d["bad_append_warp"] == APPEND_CAPACITY | BOUNDS


def test_default_build_sets_no_bounds_bit_and_matches_the_debug_build(both):
    d, n = both
    assert n["lib"].endswith("libbgtq.so")
    assert n["clean_append"] == 0 and n["clean_decode"] == 0
    assert n["bad_page"] == PAGE_RANGE
    assert n["bad_seq"] == SEQLEN_CAPACITY
    assert n["bad_append_bulk"] == APPEND_CAPACITY and n["bad_append_warp"] == APPEND_CAPACITY
    # the checks change no result of a clean call
    assert d["clean_out"] == n["clean_out"]
