"""The C-ABI library on the host: it loads, exports every declared entry
point, and its host-side logic (Block-GTQ allocation, Lloyd-Max codebooks,
codec order, whitening, rotation signs, K-record lane layout) equals the
oracle bit for bit.  No GPU is needed: plans are built host-only.
"""

import ctypes
import os
import re

import numpy as np
import pytest

import rope_aware_quantized_gb300 as bg
from oracle import bgtq_oracle as O
from rope_aware_quantized_gb300 import _native, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    return _native.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "bgtq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bgtq_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
        assert isinstance(getattr(L, n), ctypes._CFuncPtr)


def test_error_reporting(L):
    calib = np.zeros((4, 128), np.float16)
    with pytest.raises(bg.BgtqError) as e:
        bg.bgtq_alloc_bits(calib, 383)
    assert e.value.code == -1 and "even" in str(e.value)
    with pytest.raises(bg.BgtqError):
        bg.bgtq_alloc_bits(calib, 384, b_max=9)
    bits = np.full((1, 64), 3, np.uint8)
    with pytest.raises(bg.BgtqError):
        bg.bgtq_plan_create(bits, np.ones((1, 64)), 4, 256, 3, 1, host_only=True)
    with pytest.raises(bg.BgtqError) as e:
        bg.bgtq_plan_create(bits, np.ones((1, 64)), 9, 384, 3, 1, host_only=True)
    assert e.value.code == -2
    assert L.bgtq_plan_destroy(None) == 0


def test_host_only_plan_rejects_device_work():
    bits = np.full((1, 64), 3, np.uint8)
    plan = bg.bgtq_plan_create(bits, np.ones((1, 64)), 4, 384, 3, 1, host_only=True)
    cache = bg._native.BgtqCache(1, 1, 1, 1, 16)
    rc = bg.lib().bgtq_decode_attn(plan.handle, None, 1, ctypes.byref(cache), 1, 16, 1, 1, 0, 0.1, 1, 1 << 20, None)
    assert rc == -1 and b"host-only" in bg.lib().bgtq_last_error()
    rc = bg.lib().bgtq_quantize_append(plan.handle, None, 1, 1, 1, 1, 1, ctypes.byref(cache), None)
    assert rc == -1


@pytest.mark.parametrize("seed,bits_per_key,layout,s_ln", [(1, 384, 0, 1.0), (2, 256, 0, 1.2), (3, 384, 1, 1.2),
                                                         (4, 128, 0, 2.0), (5, 512, 0, 0.5)])
def test_alloc_bits_matches_oracle(seed, bits_per_key, layout, s_ln):
    li = synth.layer_inputs(seed, 0, 1, 1, 8, 1e4, s_ln, rope_layout=layout)
    calib = li.calib[0]
    bits, energy = bg.bgtq_alloc_bits(calib, bits_per_key, 8, layout)
    obits, oenergy = O.alloc_bits(calib, bits_per_key, 8, layout)
    assert np.array_equal(energy, oenergy)          # float64 bit-exact
    assert np.array_equal(bits.astype(np.int64), obits)


def test_codebooks_match_oracle_bit_exactly():
    bits = np.full((1, 64), 3, np.uint8)
    plan = bg.bgtq_plan_create(bits, np.ones((1, 64)), 4, 384, 3, 1, host_only=True)
    for w in range(0, 9):
        cent, thr = plan.codebook(w)
        ocent, othr = O.codebooks()[w]
        assert np.array_equal(cent, ocent), w
        assert np.array_equal(thr, othr), w


def _ulp_walk(t, n):
    """float32 values t and the n neighbours on each side of t."""
    t = np.float32(t)
    out, a, b = [t], t, t
    for _ in range(n):
        a = np.nextafter(a, np.float32(-np.inf))
        b = np.nextafter(b, np.float32(np.inf))
        out += [a, b]
    return np.array(out, np.float32)


def test_code_search_cells_equal_threshold_count():
    """The bulk encoder takes each code from a cell table (one lookup and one
    comparison) instead of a search; its host copy must give the number of
    thresholds <= u (TQ-MSE's nearest-centroid rule with the oracle's tie
    rule) for every quotient: uniform draws over the whole quotient range
    [-sqrt(128), sqrt(128)] and past it, and every float within 300 ulps of
    every threshold, where a cell boundary or a tie would show."""
    bits = np.full((1, 64), 3, np.uint8)
    plan = bg.bgtq_plan_create(bits, np.ones((1, 64)), 4, 384, 3, 1, host_only=True)
    rng = np.random.default_rng(7)
    for w in range(0, 9):
        _, thr = O.codebooks()[w]
        u = [rng.uniform(-12.0, 12.0, 100000).astype(np.float32),
             np.array([0.0, -0.0, 11.3138, -11.3138, 1e30, -1e30, 3.4e38, -3.4e38, 1e-40, -1e-40], np.float32)]
        u += [_ulp_walk(t, 300) for t in thr]
        u = np.concatenate(u)
        want = np.searchsorted(thr, u, side="right")  # thresholds <= u
        assert np.array_equal(plan.code(w, u), want), w
    with pytest.raises(bg.BgtqError):
        plan.code(3, np.array([np.nan], np.float32))
    with pytest.raises(bg.BgtqError):
        plan.code(9, np.zeros(1, np.float32))


@pytest.mark.parametrize("seed,bits_per_key,v_bits,layout", [(11, 384, 3, 0), (12, 256, 2, 0), (13, 384, 2, 1),
                                                             (14, 128, 1, 0)])
def test_plan_tables_match_oracle(seed, bits_per_key, v_bits, layout):
    H = 3
    li = synth.layer_inputs(seed, 0, H, 2, 8, 5e5, 1.2, rope_layout=layout)
    bits, energy = [], []
    for h in range(H):
        b, e = bg.bgtq_alloc_bits(li.calib[h], bits_per_key, 8, layout)
        bits.append(b)
        energy.append(e)
    plan_seed = 0xC0FFEE + seed
    plan = bg.bgtq_plan_create(np.stack(bits), np.stack(energy), 2, bits_per_key, v_bits, plan_seed, layout,
                               host_only=True)
    for h in range(H):
        hs = O.head_state(li.calib[h], bits_per_key, v_bits, plan_seed, h, rope_layout=layout)
        kc, vc = hs.kc, hs.vc
        t = plan.head_tables(h)
        n = kc.n_coded
        assert t["n_coded"] == n
        assert np.array_equal(t["perm"][:n], kc.perm)
        assert np.array_equal(t["width"][:n], kc.width)
        assert np.array_equal(t["piece"][:n], kc.psize)
        assert np.array_equal(t["sign_k"][:n], kc.eps)
        assert np.array_equal(t["sign_v"], vc.eps)
        assert np.array_equal(t["whiten"][:n], kc.w)
        assert np.array_equal(t["dewhiten"][:n], kc.sig)
        sp, off, _ = O.k_lane_layout(kc, hs.bk)
        assert np.array_equal(t["slot_pair"], np.array(sp))
        assert np.array_equal(t["slot_offset"], np.array(off))


def test_lane_layout_hand_example_mixed_widths_in_the_library():
    """The library's K record layout for K2 with blocks 0-15 at 3 bits, 16-31
    at 1 and 32-63 at 2: the slots and offsets worked by hand from the rule
    (the oracle's test of the same example derives them step by step)."""
    bits = np.array([[3] * 16 + [1] * 16 + [2] * 32], np.uint8)
    plan = bg.bgtq_plan_create(bits, np.ones((1, 64)), 4, 256, 2, 1, host_only=True)
    t = plan.head_tables(0)
    for ln in range(4):
        assert list(t["slot_pair"][ln]) == [32 + ln, 40 + ln, ln, 8 + ln, 16 + ln, 24 + ln, 48 + ln, 56 + ln,
                                            36 + ln, 44 + ln, 4 + ln, 12 + ln, 20 + ln, 28 + ln, 52 + ln, 60 + ln]
        assert list(t["slot_offset"][ln]) == [0, 6, 12, 16, 20, 24, 28, 30, 32, 38, 44, 48, 52, 56, 60, 62]


def test_infeasible_lane_layout_is_reported_by_both():
    bits = np.zeros((1, 64), np.uint8)
    bits[0, :9] = 7
    bits[0, 9] = 1
    with pytest.raises(bg.BgtqError) as e:
        bg.bgtq_plan_create(bits, np.ones((1, 64)), 4, 128, 2, 1, host_only=True)
    assert e.value.code == -2
    kc = O.k_codec(bits[0], np.ones(64), 1, 0)
    with pytest.raises(ValueError):
        O.k_lane_layout(kc, 1)


def test_cache_bytes():
    bits = np.full((2, 64), 3, np.uint8)
    plan = bg.bgtq_plan_create(bits, np.ones((2, 64)), 8, 384, 3, 1, host_only=True)
    kb, vb, nb = bg.bgtq_cache_bytes(plan, 3, 1000)
    assert kb == 3 * 2 * 1000 * 48
    assert vb == 3 * 2 * 500 * 96
    assert nb == 3 * 2 * 1000 * 4
