"""Pins of the oracle's rotation, encoder, decoder and packing.

TQ-MSE "rotates then quantises" ("RoPE-Aware Bit Allocation for KV-Cache
Quantization" review, §1 Key Terms); its distortion falls at the 4^-b rate
the allocator assumes (review §3).  The build realises the rotation as a
randomized Walsh-Hadamard transform with SplitMix64 signs and packs codes
bit-exactly at the budget.  Pins: Vigna's published SplitMix64 outputs,
scipy's Hadamard matrix, orthogonality, dot-product preservation, the
Lloyd-Max distortion on Gaussian data, the per-block 4^-b law under
Block-GTQ, cell membership of every coordinate, and packing round trips.
"""

import math
import os

import numpy as np
import pytest
from scipy.linalg import hadamard

from oracle import bgtq_oracle as O
from rope_aware_quantized_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "splitmix64_seed0.txt")
GAMMA = 0x9E3779B97F4A7C15


def test_splitmix64_published_outputs():
    vals = [int(line, 16) for line in open(GOLDEN) if line.strip() and not line.startswith("#")]
    for k, v in enumerate(vals):
        assert O.splitmix64((k * GAMMA) & ((1 << 64) - 1)) == v


@pytest.mark.parametrize("n", [2, 4, 8, 16, 32, 64, 128])
def test_butterflies_are_sylvester_hadamard(n):
    eye = np.eye(n, dtype=np.float32)
    out = O._butterflies(eye, np.full(n, n))
    # row k of the output is H_n e_k, i.e. column k of Sylvester's H_n
    assert np.array_equal(out.T, hadamard(n).astype(np.float32))


def small_head(seed=1, bits_per_key=384, v_bits=3, s_ln=1.0, layout=0):
    li = synth.layer_inputs(seed, 0, 1, 4, 2048, 1e4, s_ln, rope_layout=layout)
    hs = O.head_state(li.calib[0], bits_per_key, v_bits, 77 + seed, 0, rope_layout=layout)
    return li, hs


def rotation_matrix(codec):
    """Codec-domain linear map (whitened coords -> y) as an explicit matrix."""
    n = codec.n_coded
    eye = np.eye(n, dtype=np.float32)
    v = O._butterflies(eye * codec.eps[None, :], codec.psize)
    return (v * codec.inv_sqrt[None, :]).astype(np.float64).T


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_rotation_is_orthogonal_and_blockwise(seed):
    _, hs = small_head(seed)
    r = rotation_matrix(hs.kc)
    assert np.allclose(r.T @ r, np.eye(hs.kc.n_coded), atol=2e-6)
    # never mixes different widths (Block-GTQ's per-block widths stay intact)
    nz = np.abs(r) > 0
    for i, j in zip(*np.nonzero(nz)):
        assert hs.kc.width[i] == hs.kc.width[j]
    h = O._butterflies(np.eye(128, dtype=np.float32)[:1], np.full(128, 128))
    assert np.all(h == 1.0)


def test_codec_logit_identity():
    """q . k_hat equals the codec-domain product (R sig q) . y_hat."""
    li, hs = small_head(2)
    codes, rho = O.encode(li.k[0][:64], hs.kc)
    khat = O.dequant(codes, rho, hs.kc)
    yhat = O.dequant(codes, rho, hs.kc, codec_domain=True)[:, : hs.kc.n_coded]
    q = li.q[:4].astype(np.float64)
    qc = (rotation_matrix(hs.kc) @ (q[:, hs.kc.perm] * hs.kc.sig[None, :].astype(np.float64)).T).T
    lhs = q @ khat.astype(np.float64).T
    rhs = qc @ yhat.astype(np.float64).T
    assert np.allclose(lhs, rhs, rtol=1e-5, atol=1e-5 * np.abs(lhs).max())


@pytest.mark.parametrize("bv", [1, 2, 3, 4, 5, 6])
def test_uniform_mse_equals_lloyd_max_distortion(bv):
    """On N(0,1) values the per-coordinate MSE is the Lloyd-Max distortion."""
    rng = np.random.default_rng(bv)
    x = rng.standard_normal((4000, 128)).astype(np.float16)
    vc = O.v_codec(bv, 5, 0)
    codes, rho = O.encode(x, vc)
    xh = O.dequant(codes, rho, vc)
    mse = np.mean((xh.astype(np.float64) - x.astype(np.float64)) ** 2)
    c, t = O.lloyd_max_fp64(bv)
    from tests.test_oracle_codebook import distortion
    d = distortion(c, t)
    assert abs(mse / d - 1) < 0.05


def test_mse_falls_about_4x_per_bit():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((3000, 128)).astype(np.float16)
    mses = []
    for bv in range(1, 7):
        vc = O.v_codec(bv, 3, 1)
        codes, rho = O.encode(x, vc)
        mses.append(np.mean((O.dequant(codes, rho, vc).astype(np.float64) - x) ** 2))
    for a, b in zip(mses[:-1], mses[1:]):
        assert 2.8 < a / b < 4.3


def test_block_gtq_error_follows_energy_and_width():
    """Under Block-GTQ the error of block i is ~ s_i * D(b_i) (the allocator's model)."""
    li = synth.layer_inputs(4, 0, 1, 4, 6000, 1e4, 1.0)
    hs = O.head_state(li.calib[0], 384, 3, 9, 0)
    codes, rho = O.encode(li.k[0], hs.kc)
    kh = O.dequant(codes, rho, hs.kc).astype(np.float64)
    k = li.k[0].astype(np.float64)
    dims = O.block_dims(0)
    dtab = {}
    from tests.test_oracle_codebook import distortion
    ratios = []
    for i, (a, b) in enumerate(dims):
        bi = int(hs.bits[i])
        err = np.mean((kh[:, a] - k[:, a]) ** 2 + (kh[:, b] - k[:, b]) ** 2)
        if bi == 0:
            assert np.all(kh[:, a] == 0) and np.all(kh[:, b] == 0)
            continue
        if bi not in dtab:
            c, t = O.lloyd_max_fp64(bi)
            dtab[bi] = distortion(c, t)
        ratios.append(err / (hs.s[i] * dtab[bi]))
    ratios = np.array(ratios)
    assert np.all(ratios > 0.5) and np.all(ratios < 2.0)
    assert abs(np.median(ratios) - 1) < 0.25


def test_every_coordinate_lands_in_its_cell():
    li, hs = small_head(3)
    for codec, x in ((hs.kc, li.k[0][:256]), (hs.vc, li.v[0][:256])):
        codes, rho = O.encode(x, codec)
        yhat = O.dequant(codes, rho, codec, codec_domain=True)[:, : codec.n_coded]
        # reconstruct y itself with the same float32 steps the encoder uses
        xf = x.astype(np.float32)
        z = xf[:, codec.perm] * codec.w[None, :] * codec.eps[None, :]
        y = O._butterflies(z, codec.psize) * codec.inv_sqrt[None, :]
        cbs = O.codebooks()
        for j in range(codec.n_coded):
            cent, thr = cbs[int(codec.width[j])]
            u = y[:, j] / rho
            lo = np.concatenate([[-np.inf], thr])[codes[:, j]]
            hi = np.concatenate([thr, [np.inf]])[codes[:, j]]
            assert np.all((u >= lo) & (u < hi))
        # the norm is the RMS of the rotated coordinates; rotation keeps energy
        s_y = np.sum(y.astype(np.float64) ** 2, axis=1)
        assert np.allclose(rho.astype(np.float64) ** 2 * codec.n_coded, s_y, rtol=1e-5)
        assert np.allclose(s_y, np.sum(z.astype(np.float64) ** 2, axis=1), rtol=1e-5)


@pytest.mark.parametrize("bits_per_key,bv", [(128, 1), (256, 2), (384, 3), (384, 2)])
def test_packing_round_trip_and_sizes(bits_per_key, bv):
    li, hs = small_head(5, bits_per_key, bv)
    x = li.k[0][:301]
    codes, rho = O.encode(x, hs.kc)
    rec = O.pack_k(codes, hs.kc, hs.bk)
    assert rec.shape == (301, 16 * hs.bk) and rec.dtype == np.uint8
    assert np.array_equal(O.unpack_k(rec, hs.kc, hs.bk), codes)
    vcodes, _ = O.encode(li.v[0][:301], hs.vc)
    vrec = O.pack_v(vcodes, bv)
    assert vrec.shape == (151, 32 * bv)
    assert np.array_equal(O.unpack_v(vrec, bv, 301), vcodes)
    # every budget bit is used: total field bits equal the budget exactly
    assert sum(2 * w for w in O.k_pairs(hs.kc)) == bits_per_key


@pytest.mark.parametrize("seed", range(10))
def test_lane_layout_invariants(seed):
    rng = np.random.default_rng(seed)
    for bk in (1, 2, 3):
        s = rng.lognormal(0.0, 1.5, O.NB)
        s[-4:] *= 64
        bits = O.greedy_bits(s, 128 * bk, 8)
        kc = O.k_codec(bits, s, 1, 0)
        sp, off, wd = O.k_lane_layout(kc, bk)
        assert sorted(m for lane in sp for m in lane) == list(range(O.NB))
        for t in range(4):
            total = sum(2 * wd[m] for m in sp[t])
            assert total == 32 * bk
            # the slot windows used by the decode kernel: slots 0-7 end inside
            # bits [0, 64) and slots 8-15 start at or after bit 32
            end8 = off[t][8]
            assert end8 <= 64
            if bk == 3:
                assert end8 >= 32
            # within a half the slots are in non-increasing width order
            w = [wd[m] for m in sp[t]]
            assert w[:8] == sorted(w[:8], reverse=True) and w[8:] == sorted(w[8:], reverse=True)


def test_lane_layout_reports_infeasible_allocations():
    bits = np.zeros(O.NB, dtype=np.int64)
    bits[:9] = 7
    bits[9] = 1
    s = np.ones(O.NB)
    kc = O.k_codec(bits, s, 1, 0)
    with pytest.raises(ValueError):
        O.k_lane_layout(kc, 1)


def test_v_pair_record_layout():
    codes = np.zeros((3, 128), dtype=np.int64)
    codes[0, 0] = 2
    codes[1, 0] = 1
    codes[2, 127] = 3
    rec = O.pack_v(codes, 2)
    words = rec.view("<u4")
    # dim 0 of pair 0: even token code 2 in bits 0-1, odd token code 1 in bits 2-3
    assert words[0, 0] == 2 | (1 << 2)
    # dim 127 of pair 1 (token 2 even, no odd token): bits 508-509 -> word 15, bits 28-29
    assert words[1, 15] == 3 << 28


def test_lane_layout_hand_example_uniform_widths():
    """Uniform K2 (every pair 4 bits): worked by hand from the rule.  Ranks
    equal pair indices; lane t first takes the pairs with rank = t (mod 4),
    which already sum to the 32-bit slice, so lane t = {t, t+4, ..., t+60};
    slots alternate even / odd positions of that list."""
    kc = O.k_codec(np.full(O.NB, 2), np.ones(O.NB), 1, 0)
    sp, off, wd = O.k_lane_layout(kc, 2)
    for t in range(4):
        lane = list(range(t, 64, 4))
        assert sp[t] == lane[0::2] + lane[1::2]
        assert off[t] == [4 * s for s in range(16)]
    # the K record of a token with code pattern code_j = j mod 4: pair m holds
    # (2m mod 4) | (2m+1 mod 4) << 2 = 0b1000 | ... computed field by field
    codes = (np.arange(128) % 4)[None, :]
    rec = O.pack_k(codes, kc, 2).view("<u4")[0]
    # lane 0, slot 0 = pair 0: codes (0, 1) -> field 0 | 1 << 2 = 4 at bits 0-3
    # lane 0, slot 1 = pair 8: codes (16 % 4, 17 % 4) = (0, 1) -> 4 at bits 4-7
    assert rec[0] & 0xFF == 0x44
    # every pair m has codes (2m % 4, (2m + 1) % 4) = (0|2, 1|3): field 4 or 14
    for t in range(4):
        word = int(rec[2 * t]) | (int(rec[2 * t + 1]) << 32)
        for s in range(16):
            m = sp[t][s]
            want = (2 * m % 4) | (((2 * m + 1) % 4) << 2)
            assert (word >> (4 * s)) & 0xF == want


def test_lane_layout_hand_example_mixed_widths():
    """K2 with three width classes, worked by hand from the rule.  Blocks 0-15
    get 3 bits, 16-31 get 1, 32-63 get 2.  Codec order (pieces by size, then
    width): the 64-piece of width 2 (blocks 32-63) is codec pairs 0-31, the
    32-piece of width 3 (blocks 0-15) pairs 32-47, the 32-piece of width 1
    (blocks 16-31) pairs 48-63.  Ranks by (width desc, index): pairs 32-47
    are ranks 0-15, pairs 0-31 ranks 16-47, pairs 48-63 ranks 48-63.  Lane t
    scans ranks = t (mod 4) first: 4 of width 3, 8 of width 2 and 4 of width 1,
    16 pairs whose widths sum to 32 = 16 bK, so it takes exactly those.  In
    the lane, sorted a_0..a_15 = 32+t, 36+t, 40+t, 44+t, t, 4+t, ..., 28+t,
    48+t, ..., 60+t; slots take a_0, a_2, ..., a_14 then a_1, ..., a_15, and
    the fields (2w bits) of slots 0-7 are 6, 6, 4, 4, 4, 4, 2, 2 bits long."""
    bits = np.array([3] * 16 + [1] * 16 + [2] * 32)
    kc = O.k_codec(bits, np.ones(O.NB), 1, 0)
    sp, off, wd = O.k_lane_layout(kc, 2)
    assert wd == [2] * 32 + [3] * 16 + [1] * 16
    for t in range(4):
        assert sp[t] == [32 + t, 40 + t, t, 8 + t, 16 + t, 24 + t, 48 + t, 56 + t,
                         36 + t, 44 + t, 4 + t, 12 + t, 20 + t, 28 + t, 52 + t, 60 + t]
        assert off[t] == [0, 6, 12, 16, 20, 24, 28, 30, 32, 38, 44, 48, 52, 56, 60, 62]
    # pair m's codes: (m >> 2) and (m >> 2) + 3, each mod 2^w.  Lane 0, slots
    # 0-7 (pairs 32, 40, 0, 8, 16, 24, 48, 56): fields 0 | 3 << 3 = 24,
    # 2 | 5 << 3 = 42, 0 | 3 << 2 = 12, 2 | 1 << 2 = 6, 12, 6, 0 | 1 << 1 = 2, 2
    # at bits 0, 6, 12, 16, 20, 24, 28, 30: 0xA6C6CA98 in the record's word 0
    codes = np.zeros((1, 128), dtype=np.int64)
    for m in range(64):
        mask = (1 << wd[m]) - 1
        codes[0, 2 * m] = (m >> 2) & mask
        codes[0, 2 * m + 1] = ((m >> 2) + 3) & mask
    rec = O.pack_k(codes, kc, 2).view("<u4")[0]
    assert int(rec[0]) == 0xA6C6CA98
    assert np.array_equal(O.unpack_k(O.pack_k(codes, kc, 2), kc, 2), codes)
