"""Block-GTQ packed-cache decode path: the CPU oracle.

TEST INFRASTRUCTURE.  This module is a plain, slow, deliberately literal
restatement of what the packed-cache decode path computes.  It exists to
check the CUDA library and is used only by the tests, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``.
The product path (the C-ABI library and its Python binding) never imports,
links or calls it, and it shares no code, table or constant generator with
the library: every table here (codebooks, thresholds, signs, permutations,
lane layouts) is derived independently from the definitions below.

Sources.  The method is described on two pages about one paper,
"RoPE-Aware Bit Allocation for KV-Cache Quantization":
  * the paper review (page title "[논문리뷰] RoPE-Aware Bit Allocation for
    KV-Cache Quantization"), §1 Key Terms and §3 Method & Key Results;
  * the abstract page (page title "RoPE를 고려한 KV-캐시 양자화 비트 할당"),
    English abstract.
They fix: RoPE splits a key into 2-D frequency blocks and the logit is a sum
over those blocks; TQ-MSE rotates then scalar-quantises with a near-optimal
distortion rate; Block-GTQ scores each (layer, KV head, block) with a
label-free energy from calibration data and greedily gives integer bit widths
by marginal gain under the TQ-MSE 4^-b rate; values use uniform TQ-MSE; the
packed-cache path attends directly on compressed K/V.  Everything the pages
leave open (energy formula, codebook, rotation, norm, packing) is settled by a
numbered reading (R1, R2, ...); each function below names and states the
reading it implements.

Floating point.  Allocation and codebook design are float64.  The encoder
and decoder are float32, one IEEE operation at a time in a fixed order
(numpy float32 arithmetic is correctly rounded and never contracted), so the
codes, norms and dequantised values are exact expectations for the CUDA
path.  Attention is float64 over the float32 dequantised cache.

Parity pins: every function here is pinned by tests in
``tests/test_oracle_*.py`` against closed forms, published constants
(tests/golden/), brute force or library routines.
"""

from __future__ import annotations

import math

import numpy as np
from scipy.linalg import solve_banded
from scipy.special import ndtr, ndtri

D = 128          # head dim
NB = 64          # RoPE 2-D blocks per key
WMAX = 8         # largest width any code may have (codes fit a byte)

# =============================================================================
# RoPE blocks (review §1 "RoPE": 2-D blocks; abstract: the logit is a sum over
# two-dimensional frequency blocks).  Reading R1: half-split pairing
# (i, i + 64) by default, interleaved (2i, 2i + 1) as an option.
# =============================================================================


def block_dims(rope_layout: int = 0):
    if rope_layout == 0:
        return [(i, i + NB) for i in range(NB)]
    if rope_layout == 1:
        return [(2 * i, 2 * i + 1) for i in range(NB)]
    raise ValueError("rope_layout must be 0 or 1")


# =============================================================================
# Allocation: energy score and greedy integer bit widths.
# Abstract: "computes a label-free energy score for each RoPE block and
# greedily allocates integer bit widths by marginal gain"; review §3: the
# gain uses the TQ-MSE 4^-b rate under a total budget.
# =============================================================================


def energy(calib_fp16: np.ndarray, rope_layout: int = 0) -> np.ndarray:
    """Reading R2: s_i = (1/n) sum_t (k_t[lo_i]^2 + k_t[hi_i]^2), float64.

    Accumulated in ascending t as acc = (acc + k[lo]^2) + k[hi]^2 (the
    squares of float16 values are exact in float64), divided by n last.
    """
    x = np.asarray(calib_fp16, dtype=np.float16).astype(np.float64)
    n = x.shape[0]
    if n <= 0 or x.shape[1] != D:
        raise ValueError("calibration keys must be [n>0][128]")
    dims = block_dims(rope_layout)
    lo = np.array([a for a, _ in dims])
    hi = np.array([b for _, b in dims])
    acc = np.zeros(NB, dtype=np.float64)
    for t in range(n):
        acc = (acc + x[t, lo] * x[t, lo]) + x[t, hi] * x[t, hi]
    return acc / float(n)


def greedy_bits(s: np.ndarray, bits_per_key: int, b_max: int = WMAX) -> np.ndarray:
    """Readings R3-R5: widths b_i in {0..b_max}, sum_i 2*b_i = bits_per_key.

    Each step gives one bit to both coordinates of the block with the largest
    marginal gain s_i*(4^-b_i - 4^-(b_i+1)) = (3/4) s_i 4^-b_i among blocks
    still below b_max; ties go to the smallest block index.  Comparisons are
    exact (scaling by a power of two).
    """
    if bits_per_key % 2 or bits_per_key < 0 or not (1 <= b_max <= WMAX):
        raise ValueError("bits_per_key must be even and >= 0, 1 <= b_max <= 8")
    steps = bits_per_key // 2
    if steps > NB * b_max:
        raise ValueError("budget exceeds 64 * b_max")
    b = [0] * NB
    for _ in range(steps):
        best, best_gain = -1, 0.0
        for i in range(NB):
            if b[i] >= b_max:
                continue
            gain = math.ldexp(float(s[i]), -2 * b[i])
            if best < 0 or gain > best_gain:
                best, best_gain = i, gain
        b[best] += 1
    return np.array(b, dtype=np.int64)


def alloc_bits(calib_fp16, bits_per_key: int, b_max: int = WMAX, rope_layout: int = 0):
    s = energy(calib_fp16, rope_layout)
    return greedy_bits(s, bits_per_key, b_max), s


# =============================================================================
# TQ-MSE scalar codebook (review §1 "TQ-MSE": rotate, then quantise with a
# near-optimal distortion rate).  Reading R9: Lloyd-Max quantiser for N(0,1)
# with 2^b levels, fixed point solved in float64, centroids rounded to fp16,
# thresholds = midpoints of adjacent rounded centroids.
# =============================================================================

_SQ2PI = math.sqrt(2.0 * math.pi)


def _pdf(x):
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    fin = np.isfinite(x)
    out[fin] = np.exp(-0.5 * x[fin] * x[fin]) / _SQ2PI
    return out


def _cells(t):
    a = np.concatenate([[-np.inf], t])
    b = np.concatenate([t, [np.inf]])
    mass = np.where(a > 0, ndtr(-a) - ndtr(-b), ndtr(b) - ndtr(a))
    c = (_pdf(a) - _pdf(b)) / mass
    return a, b, mass, c


def lloyd_max_fp64(bits: int):
    """Unrounded Lloyd-Max centroids and thresholds for N(0,1), 2^bits levels.

    The fixed point of "each threshold is the midpoint of its neighbouring
    centroids, each centroid is the conditional mean of its cell" is found by
    Newton's method on the thresholds (tridiagonal Jacobian), started from
    the high-rate (Panter-Dite) point density, until the step is below 1e-13.
    """
    n = 1 << bits
    if n == 2:
        c = math.sqrt(2.0 / math.pi)
        return np.array([-c, c]), np.array([0.0])
    t = math.sqrt(3.0) * ndtri(np.arange(1, n) / n)
    for _ in range(200):
        a, b, m, c = _cells(t)
        f = t - 0.5 * (c[:-1] + c[1:])
        pa, pb = _pdf(a), _pdf(b)
        fa = np.where(np.isfinite(a), a, 0.0)
        fb = np.where(np.isfinite(b), b, 0.0)
        dc_da = pa * (c - fa) / m          # d c_k / d (lower end of cell k)
        dc_db = pb * (fb - c) / m          # d c_k / d (upper end of cell k)
        k = n - 1
        ab = np.zeros((3, k))
        ab[1, :] = 1.0 - 0.5 * (dc_db[:-1] + dc_da[1:])
        ab[0, 1:] = -0.5 * dc_db[1:-1]      # dF_k / dt_{k+1}
        ab[2, :-1] = -0.5 * dc_da[1:-1]     # dF_{k+1} / dt_k
        step = solve_banded((1, 1), ab, -f)
        t = t + step
        t = 0.5 * (t - t[::-1])
        if np.max(np.abs(step)) < 1e-13:
            break
    _, _, _, c = _cells(t)
    return 0.5 * (c - c[::-1]), t


def codebook(bits: int):
    """(centroids, thresholds) as float32 arrays; centroids are fp16 values."""
    if bits == 0:
        return np.zeros(1, dtype=np.float32), np.zeros(0, dtype=np.float32)
    c, _ = lloyd_max_fp64(bits)
    ch = c.astype(np.float16).astype(np.float64)
    thr = (0.5 * (ch[:-1] + ch[1:])).astype(np.float32)
    return ch.astype(np.float32), thr


_CB_CACHE: dict = {}


def codebooks():
    """Codebooks for widths 0..8 (cached)."""
    if not _CB_CACHE:
        for b in range(WMAX + 1):
            _CB_CACHE[b] = codebook(b)
    return _CB_CACHE


# =============================================================================
# Random signs of the randomized Hadamard rotation (reading R8).  SplitMix64
# is Vigna's published generator; the sign is bit 63 of its output.
# =============================================================================

_M64 = (1 << 64) - 1


def splitmix64(x: int) -> int:
    z = (int(x) + 0x9E3779B97F4A7C15) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def sign(seed: int, head: int, tag: int, j: int) -> float:
    """-1 when bit 63 of splitmix64(seed ^ head<<16 ^ tag<<8 ^ j) is set."""
    key = (int(seed) ^ (int(head) << 16) ^ (int(tag) << 8) ^ int(j)) & _M64
    return -1.0 if (splitmix64(key) >> 63) & 1 else 1.0


# =============================================================================
# Codec domain of one head (readings R6-R8).
# =============================================================================


class Codec:
    """Codec-domain description of one head's K or V encoder."""

    def __init__(self, perm, width, psize, eps, w, sig, n_coded, blocks=None):
        self.perm = np.asarray(perm, dtype=np.int64)        # codec index -> original dim
        self.width = np.asarray(width, dtype=np.int64)      # code width per codec index
        self.psize = np.asarray(psize, dtype=np.int64)      # rotation piece size per codec index
        self.eps = np.asarray(eps, dtype=np.float32)        # +-1 per codec index
        self.w = np.asarray(w, dtype=np.float32)            # whitening multiplier per codec index
        self.sig = np.asarray(sig, dtype=np.float32)        # de-whitening multiplier per codec index
        self.n_coded = int(n_coded)
        self.blocks = blocks
        self.inv_sqrt = np.array([np.float32(1.0 / math.sqrt(float(p))) for p in self.psize], dtype=np.float32)


def k_codec(bits, s, seed: int, head: int, rope_layout: int = 0) -> Codec:
    """Reading R6 (codec order) and R7 (whitening) for one head's keys.

    Width classes in descending width; a class's coordinates are its blocks
    in ascending index, each contributing (lo_i, hi_i).  Each class is cut
    into power-of-two pieces by binary decomposition of its size, largest
    first.  All pieces are laid out sorted by (size desc, width desc).
    """
    bits = [int(b) for b in bits]
    dims = block_dims(rope_layout)
    pieces = []
    for wdt in range(WMAX, 0, -1):
        coords = []
        for i in range(NB):
            if bits[i] == wdt:
                coords += [dims[i][0], dims[i][1]]
        pos = 0
        for p in range(7, 0, -1):
            size = 1 << p
            if len(coords) & size:
                pieces.append((size, wdt, coords[pos:pos + size]))
                pos += size
    pieces.sort(key=lambda pc: (-pc[0], -pc[1]))
    dim_block = {}
    for i, (a, b) in enumerate(dims):
        dim_block[a] = i
        dim_block[b] = i
    perm, width, psize = [], [], []
    for size, wdt, coords in pieces:
        perm += coords
        width += [wdt] * size
        psize += [size] * size
    n = len(perm)
    wv, sv, ev = [], [], []
    for j in range(n):
        si = float(s[dim_block[perm[j]]])
        wv.append(np.float32(1.0) if si == 0.0 else np.float32(math.sqrt(2.0 / si)))
        sv.append(np.float32(math.sqrt(si / 2.0)))
        ev.append(sign(seed, head, 0, j))
    return Codec(perm, width, psize, ev, wv, sv, n, blocks=[dim_block[p] for p in perm])


def v_codec(v_bits: int, seed: int, head: int) -> Codec:
    """Values: uniform TQ-MSE (abstract: the uniform TQ-MSE baseline), one
    128-piece in natural order, no whitening, sign tag 1."""
    return Codec(np.arange(D), [v_bits] * D, [D] * D, [sign(seed, head, 1, j) for j in range(D)],
                 [1.0] * D, [1.0] * D, D)


# =============================================================================
# Encoder / decoder (readings R8, R10, R11, R13), float32, fixed order.
# =============================================================================

_F32 = np.float32


def _butterflies(v: np.ndarray, psize: np.ndarray) -> np.ndarray:
    """Unnormalised Walsh-Hadamard butterflies inside each aligned piece.

    Stages h = 1, 2, 4, ...; at each stage a pair (j, j+h) with bit h of j
    clear and both in a piece larger than h becomes (a + b, a - b).
    """
    v = v.astype(_F32, copy=True)
    n = v.shape[1]
    h = 1
    while h < D:
        new = v.copy()
        for j in range(n):
            if (j & h) == 0 and psize[j] > h:
                a = v[:, j]
                b = v[:, j + h]
                new[:, j] = a + b
                new[:, j + h] = a - b
        v = new
        h <<= 1
    return v


def encode(x_fp16: np.ndarray, codec: Codec, cbs=None):
    """Encode tokens x [T,128] fp16 -> (codes int [T, n_coded], rho f32 [T]).

    z_j = x[perm_j] * w_j; v = eps * z; butterflies; y = v * (1/sqrt(piece));
    rho = sqrt(sum y^2 / n_coded) summed by the fixed tree of reading R10;
    u = y / rho; code = number of thresholds <= u (ties go up).
    """
    cbs = cbs or codebooks()
    x = np.asarray(x_fp16, dtype=np.float16).astype(_F32)
    n = codec.n_coded
    z = x[:, codec.perm] * codec.w[None, :]
    v = z * codec.eps[None, :]
    v = _butterflies(v, codec.psize)
    y = v * codec.inv_sqrt[None, :]
    t = y.shape[0]
    sq = np.zeros((t, D), dtype=_F32)
    sq[:, :n] = y * y
    part = (sq[:, 0::4] + sq[:, 1::4]) + (sq[:, 2::4] + sq[:, 3::4])
    lanes = np.arange(32)
    for m in (16, 8, 4, 2, 1):
        part = part + part[:, lanes ^ m]
    total = part[:, 0]
    rho = np.sqrt(total / _F32(n))
    codes = np.zeros((t, n), dtype=np.int64)
    safe = np.where(rho > 0, rho, _F32(1.0))
    u = np.where(rho[:, None] > 0, y / safe[:, None], _F32(0.0)).astype(_F32)
    for j in range(n):
        thr = cbs[int(codec.width[j])][1]
        codes[:, j] = np.searchsorted(thr, u[:, j], side="right")
    return codes, rho.astype(_F32)


def dequant(codes: np.ndarray, rho: np.ndarray, codec: Codec, cbs=None, codec_domain: bool = False):
    """Decode -> float32 [T,128].  Codec domain: y_hat at codec index j.

    Original domain: y_hat_j = rho * c[code_j]; butterflies; * 1/sqrt(piece);
    * eps; * sig (keys); scattered to perm_j, uncoded dims are 0.
    """
    cbs = cbs or codebooks()
    t = codes.shape[0]
    n = codec.n_coded
    c = np.zeros((t, n), dtype=_F32)
    for j in range(n):
        c[:, j] = cbs[int(codec.width[j])][0][codes[:, j]]
    yh = np.asarray(rho, dtype=_F32)[:, None] * c
    out = np.zeros((t, D), dtype=_F32)
    if codec_domain:
        out[:, :n] = yh
        return out
    v = _butterflies(yh, codec.psize)
    v = v * codec.inv_sqrt[None, :]
    v = v * codec.eps[None, :]
    v = v * codec.sig[None, :]
    out[:, codec.perm] = v
    return out


# =============================================================================
# Packing (reading R12).
# K: one record of 16*bK bytes per token, split into four lane slices of bK
#    32-bit words; each slice holds 16 pair fields (code_{2m} | code_{2m+1} << w).
# V: one record of 32*bV bytes per token pair (2i, 2i+1): the field of dim j is
#    code_even | code_odd << bV at bit 2*bV*j.
# Bits are LSB-first inside little-endian 32-bit words.
# =============================================================================


def k_pairs(codec: Codec):
    """Widths of the 64 codec pairs; pairs past n_coded/2 are empty (width 0)."""
    npc = codec.n_coded // 2
    return [int(codec.width[2 * m]) for m in range(npc)] + [0] * (NB - npc)


def k_lane_layout(codec: Codec, bk: int):
    """Assign the 64 pairs to 4 lanes x 16 slots (reading R12).

    Rank pairs by (width desc, index asc).  Lanes 0, 1, 2 in turn take the
    first 16-subset, in the order ((rank - lane) mod 4, rank), whose widths
    sum to 16*bK (an item is taken when the remaining items can still
    complete the subset); lane 3 takes the rest.  Inside a lane the pairs
    sorted by (width desc, index asc) a_0..a_15 fill slots
    a_0, a_2, ..., a_14, a_1, a_3, ..., a_15.
    Returns slot_pair[4][16] and field offsets off[4][16] (bits into the
    lane's slice); raises ValueError when no balanced layout is found.
    """
    wd = k_pairs(codec)
    target = 16 * bk
    rank_order = sorted(range(NB), key=lambda m: (-wd[m], m))
    rank = {m: r for r, m in enumerate(rank_order)}
    remaining = list(range(NB))
    lanes = []
    for t in range(3):
        order = sorted(remaining, key=lambda m: ((rank[m] - t) % 4, rank[m]))
        n = len(order)
        # reach[i][k][s]: k items with width sum s can be chosen from order[i:]
        reach = np.zeros((n + 1, 17, target + 1), dtype=bool)
        reach[n, 0, 0] = True
        for i in range(n - 1, -1, -1):
            w = wd[order[i]]
            reach[i] = reach[i + 1]
            reach[i, 1:, w:] |= reach[i + 1, :-1, : target + 1 - w]
        if not reach[0][16][target]:
            raise ValueError("no balanced lane layout for this allocation")
        k, s, chosen = 16, target, []
        for i, m in enumerate(order):
            if k > 0 and wd[m] <= s and reach[i + 1][k - 1][s - wd[m]]:
                chosen.append(m)
                k -= 1
                s -= wd[m]
        lanes.append(chosen)
        remaining = [m for m in remaining if m not in chosen]
    lanes.append(remaining)
    slot_pair, off = [], []
    for t in range(4):
        a = sorted(lanes[t], key=lambda m: (-wd[m], m))
        slots = a[0::2] + a[1::2]
        o, offs = 0, []
        for m in slots:
            offs.append(o)
            o += 2 * wd[m]
        if o != 32 * bk:
            raise ValueError("lane slice does not fill its words")
        slot_pair.append(slots)
        off.append(offs)
    return slot_pair, off, wd


def _put_bits(words: np.ndarray, bitpos: int, value: np.ndarray, nbits: int):
    """OR `value` (nbits wide, per token) into uint64-held 32-bit words at bitpos."""
    if nbits == 0:
        return
    wi, sh = bitpos >> 5, bitpos & 31
    v = value.astype(np.uint64)
    words[:, wi] |= (v << np.uint64(sh)) & np.uint64(0xFFFFFFFF)
    if sh + nbits > 32:
        words[:, wi + 1] |= v >> np.uint64(32 - sh)


def _get_bits(words: np.ndarray, bitpos: int, nbits: int) -> np.ndarray:
    if nbits == 0:
        return np.zeros(words.shape[0], dtype=np.int64)
    wi, sh = bitpos >> 5, bitpos & 31
    v = words[:, wi] >> np.uint64(sh)
    if sh + nbits > 32:
        v = v | (words[:, wi + 1] << np.uint64(32 - sh))
    return (v & np.uint64((1 << nbits) - 1)).astype(np.int64)


def _words_to_bytes(words: np.ndarray) -> np.ndarray:
    return words.astype("<u4").view(np.uint8).reshape(words.shape[0], -1)


def _bytes_to_words(b: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(b).view("<u4").reshape(b.shape[0], -1).astype(np.uint64)


def pack_k(codes: np.ndarray, codec: Codec, bk: int) -> np.ndarray:
    """K records, uint8 [T, 16*bK]."""
    slot_pair, off, wd = k_lane_layout(codec, bk)
    t = codes.shape[0]
    npc = codec.n_coded // 2
    words = np.zeros((t, 4 * bk), dtype=np.uint64)
    for ln in range(4):
        for s in range(16):
            m = slot_pair[ln][s]
            w = wd[m]
            if w == 0 or m >= npc:
                continue
            field = codes[:, 2 * m] | (codes[:, 2 * m + 1] << w)
            _put_bits(words, 32 * bk * ln + off[ln][s], field, 2 * w)
    return _words_to_bytes(words)


def unpack_k(rec: np.ndarray, codec: Codec, bk: int) -> np.ndarray:
    slot_pair, off, wd = k_lane_layout(codec, bk)
    words = _bytes_to_words(rec)
    t = words.shape[0]
    npc = codec.n_coded // 2
    codes = np.zeros((t, codec.n_coded), dtype=np.int64)
    for ln in range(4):
        for s in range(16):
            m = slot_pair[ln][s]
            w = wd[m]
            if w == 0 or m >= npc:
                continue
            f = _get_bits(words, 32 * bk * ln + off[ln][s], 2 * w)
            codes[:, 2 * m] = f & ((1 << w) - 1)
            codes[:, 2 * m + 1] = f >> w
    return codes


def pack_v(codes: np.ndarray, bv: int) -> np.ndarray:
    """V pair records, uint8 [ceil(T/2), 32*bV]; a missing odd token is 0."""
    t = codes.shape[0]
    npairs = (t + 1) // 2
    ev = codes[0::2]
    od = np.zeros_like(ev)
    od[: t // 2] = codes[1::2]
    words = np.zeros((npairs, 8 * bv), dtype=np.uint64)
    for j in range(D):
        field = ev[:, j] | (od[:, j] << bv)
        _put_bits(words, 2 * bv * j, field, 2 * bv)
    return _words_to_bytes(words)


def unpack_v(rec: np.ndarray, bv: int, t: int) -> np.ndarray:
    words = _bytes_to_words(rec)
    codes = np.zeros((2 * words.shape[0], D), dtype=np.int64)
    for j in range(D):
        f = _get_bits(words, 2 * bv * j, 2 * bv)
        codes[0::2, j] = f & ((1 << bv) - 1)
        codes[1::2, j] = f >> bv
    return codes[:t]


# =============================================================================
# Attention over the dequantised cache (reading R14): float64 softmax.
# =============================================================================


def attention(q_fp16: np.ndarray, khat: np.ndarray, vhat: np.ndarray, scale: float = 1.0 / math.sqrt(D)):
    """o_g = sum_t softmax_t(scale * q_g . k_t) v_t, float64 [G,128]."""
    q = np.asarray(q_fp16, dtype=np.float16).astype(np.float64)
    k = np.asarray(khat, dtype=np.float64)
    v = np.asarray(vhat, dtype=np.float64)
    if k.shape[0] == 0:
        return np.zeros((q.shape[0], D))
    s = (q @ k.T) * scale
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    return (p @ v) / p.sum(axis=1, keepdims=True)


def attention_partial(q_fp16, khat, vhat, scale=1.0 / math.sqrt(D)):
    """(m, l, acc) of one token range, for the log-sum-exp merge."""
    q = np.asarray(q_fp16, dtype=np.float16).astype(np.float64)
    s = (q @ np.asarray(khat, dtype=np.float64).T) * scale
    m = s.max(axis=1)
    p = np.exp(s - m[:, None])
    return m, p.sum(axis=1), p @ np.asarray(vhat, dtype=np.float64)


def merge_partials(parts):
    """Log-sum-exp merge of (m, l, acc) partials -> normalised output."""
    m = np.max([p[0] for p in parts], axis=0)
    l_tot = sum(p[1] * np.exp(p[0] - m) for p in parts)
    acc = sum(p[2] * np.exp(p[0] - m)[:, None] for p in parts)
    return acc / l_tot[:, None]


# =============================================================================
# Convenience: a whole head and a whole layer.
# =============================================================================


class HeadState:
    def __init__(self, kc: Codec, vc: Codec, bits, s, bk: int, bv: int):
        self.kc, self.vc, self.bits, self.s, self.bk, self.bv = kc, vc, bits, s, bk, bv


def head_state(calib_fp16, bits_per_key: int, v_bits: int, seed: int, head: int,
               b_max: int = WMAX, rope_layout: int = 0) -> HeadState:
    bits, s = alloc_bits(calib_fp16, bits_per_key, b_max, rope_layout)
    return HeadState(k_codec(bits, s, seed, head, rope_layout), v_codec(v_bits, seed, head),
                     bits, s, bits_per_key // 128, v_bits)


def encode_head(hs: HeadState, k_fp16, v_fp16):
    """-> dict with codes, norms, packed records and dequantised K/V."""
    kcodes, krho = encode(k_fp16, hs.kc)
    vcodes, vrho = encode(v_fp16, hs.vc)
    out = {"kcodes": kcodes, "krho": krho, "vcodes": vcodes, "vrho": vrho}
    out["krec"] = pack_k(kcodes, hs.kc, hs.bk)
    out["vrec"] = pack_v(vcodes, hs.bv)
    out["khat"] = dequant(kcodes, krho, hs.kc)
    out["vhat"] = dequant(vcodes, vrho, hs.vc)
    return out


def decode_attention_head(hs: HeadState, q_fp16, khat, vhat, scale=1.0 / math.sqrt(D)):
    return attention(q_fp16, khat, vhat, scale)


# =============================================================================
# RoPE-logit fidelity diagnostic (review §3: Block-GTQ lowers the error of the
# RoPE logits against uniform TQ-MSE at matched bit budgets; abstract: the
# logit is a sum over 2-D frequency blocks, which is why per-block widths
# help).  Reading R19: the figure is the mean absolute error of the attention
# logits, scale * q.k_hat against scale * q.k over the cached tokens, per
# query head; the baseline is uniform TQ-MSE on the keys at the same budget.
# =============================================================================


def uniform_head_state(bits_per_key: int, v_bits: int, seed: int, head: int, rope_layout: int = 0) -> HeadState:
    """Uniform TQ-MSE keys at the budget of `bits_per_key`: every block gets
    bK = bits_per_key / 128 bits and all energies are equal (s_i = 2, so the
    whitening w_i = sqrt(2 / s_i) is the identity), which leaves a single
    rotation piece over all 128 coordinates, as for values (reading R17)."""
    bk = bits_per_key // 128
    bits = np.full(NB, bk, dtype=np.int64)
    s = np.full(NB, 2.0)
    return HeadState(k_codec(bits, s, seed, head, rope_layout), v_codec(v_bits, seed, head), bits, s, bk, v_bits)


def logit_mae(q_fp16: np.ndarray, k_fp16: np.ndarray, khat: np.ndarray, scale: float = 1.0 / math.sqrt(D)):
    """(1/T) sum_t |scale q.k_t - scale q.khat_t| for every query row, float64.
    q [G][128], k [T][128] (the keys as given), khat [T][128] (dequantised)."""
    q = q_fp16.astype(np.float64)
    exact = scale * (k_fp16.astype(np.float64) @ q.T)      # [T][G]
    approx = scale * (khat.astype(np.float64) @ q.T)
    return np.abs(exact - approx).mean(axis=0)


# =============================================================================
# fp16 recent-key buffer (abstract: the AIME result is stated "without an fp16
# recent-key buffer", so the option exists).  Reading R20: the last W cached
# keys of each (sequence, KV head) are also kept in fp16, and attention uses
# those exact keys for positions [T - W, T) and the dequantised keys before
# that; values stay packed.
# =============================================================================


def keys_with_recent(khat: np.ndarray, k_fp16: np.ndarray, w: int) -> np.ndarray:
    """khat [T][128] with rows max(0, T - w) .. T - 1 replaced by the fp16 keys."""
    t = khat.shape[0]
    out = khat.astype(np.float64).copy()
    lo = max(0, t - w)
    out[lo:] = k_fp16[lo:t].astype(np.float64)
    return out


def attention_recent(q_fp16, khat, vhat, k_fp16, w: int, scale: float = 1.0 / math.sqrt(D)):
    """Decode attention over the packed cache with an fp16 recent-key buffer of w keys."""
    return attention(q_fp16, keys_with_recent(khat, k_fp16, w), vhat, scale)


# =============================================================================
# Prefill attention fused with quantize (the method's next step before the
# decode path: attend over the prompt's fp16 tiles while its packed codes are
# written).  Reading R21: a prefill of T tokens into an empty cache writes the
# packed records of positions 0 .. T-1 with the encoder of readings R8-R13,
# unchanged, and returns causal attention over the tokens as given: query row
# i attends keys 0 .. i with the fp16 keys and values, float64 softmax, the
# query heads of a KV head sharing its keys (reading R15).
# =============================================================================


def prefill_attention(q_fp16, k_fp16, v_fp16, scale: float = 1.0 / math.sqrt(D), rows: int = 256):
    """q [G][T][128], k, v [T][128] (fp16) -> [G][T][128] float64:
    out[g][i] = sum_{j <= i} softmax_j(scale q[g][i] . k[j]) v[j]."""
    q = np.asarray(q_fp16, dtype=np.float16).astype(np.float64)
    k = np.asarray(k_fp16, dtype=np.float16).astype(np.float64)
    v = np.asarray(v_fp16, dtype=np.float16).astype(np.float64)
    G, T = q.shape[0], q.shape[1]
    out = np.zeros((G, T, D))
    for r0 in range(0, T, rows):
        r1 = min(T, r0 + rows)
        s = np.einsum("gid,jd->gij", q[:, r0:r1], k[:r1]) * scale
        causal = np.arange(r1)[None, :] <= np.arange(r0, r1)[:, None]
        s = np.where(causal[None], s, -np.inf)
        s = s - s.max(axis=2, keepdims=True)
        p = np.exp(s)
        out[:, r0:r1] = np.einsum("gij,jd->gid", p, v[:r1]) / p.sum(axis=2, keepdims=True)
    return out


# =============================================================================
# Chunked prefill onto a non-empty cache (the same next step, a later chunk of
# a long prompt).  Reading R22: a chunk of C tokens at positions P0 .. P0+C-1
# of a sequence whose cache already holds P0 packed tokens writes the packed
# records of its own positions (encoder unchanged: an append at pos_start =
# P0) and returns, for query row i, one softmax over the P0 cached keys as
# stored (dequantised, reading R13) and the chunk's keys 0 .. i as given
# (fp16), values likewise: the prefix is what the cache holds, the chunk is
# the prompt as given, exactly as a prefill into an empty cache (R21) treats
# its own tokens.  P0 = 0 is R21.
# =============================================================================


def chunk_prefill_attention(q_fp16, khat_prefix, vhat_prefix, k_fp16, v_fp16, scale: float = 1.0 / math.sqrt(D),
                            rows: int = 256):
    """q [G][C][128] (fp16), khat_prefix, vhat_prefix [P0][128] (the cache's
    dequantised prefix), k, v [C][128] (fp16, the chunk) -> [G][C][128]
    float64: out[g][i] = sum over keys j of softmax_j(scale q[g][i] . key_j)
    value_j, keys = the P0 prefix rows then the chunk rows 0 .. i."""
    q = np.asarray(q_fp16, dtype=np.float16).astype(np.float64)
    kp = np.asarray(khat_prefix, dtype=np.float64).reshape(-1, D)
    vp = np.asarray(vhat_prefix, dtype=np.float64).reshape(-1, D)
    keys = np.concatenate([kp, np.asarray(k_fp16, dtype=np.float16).astype(np.float64)])
    vals = np.concatenate([vp, np.asarray(v_fp16, dtype=np.float16).astype(np.float64)])
    p0 = kp.shape[0]
    G, C = q.shape[0], q.shape[1]
    out = np.zeros((G, C, D))
    for r0 in range(0, C, rows):
        r1 = min(C, r0 + rows)
        n = p0 + r1  # keys any of these rows can see
        s = np.einsum("gid,jd->gij", q[:, r0:r1], keys[:n]) * scale
        visible = np.arange(n)[None, :] <= p0 + np.arange(r0, r1)[:, None]
        s = np.where(visible[None], s, -np.inf)
        s = s - s.max(axis=2, keepdims=True)
        p = np.exp(s)
        out[:, r0:r1] = np.einsum("gij,jd->gid", p, vals[:n]) / p.sum(axis=2, keepdims=True)
    return out
