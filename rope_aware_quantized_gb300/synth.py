"""Seeded synthetic inputs for the packed-cache decode path.

This module holds none of the method's arithmetic: it only draws keys,
values, queries and calibration keys with the shapes and statistics of the
decode workloads the Block-GTQ abstract describes ("RoPE-Aware Bit
Allocation for KV-Cache Quantization", abstract: Llama-3.1-8B-, Qwen2.5-3B-
shaped decode at 32K-512K context).  Both the CUDA path and the CPU oracle
are fed from here; neither side generates its own inputs.

Recipe (the pages fix none of it; this is the build's stand-in for model
activations):

* Block energy model E(s_ln): for every (layer, KV head) and RoPE block
  i = 0..63 the per-coordinate standard deviation is sigma_i =
  exp(s_ln * N(0, 1)); the four lowest-frequency blocks i = 60..63 are scaled
  by 8 ("heavy low-frequency blocks").
* Keys before RoPE: both coordinates of block i are N(0, sigma_i^2).  RoPE is
  applied in float64 at the token's position with theta_i = base^(-2i/d)
  (half-split pairing: block i = dims (i, i + 64); the interleaved pairing
  (2i, 2i + 1) is available), then the key is rounded to float16.
* Queries: drawn like the keys of their KV head, at the decode position.
* Values: N(0, 1), float16.
* Calibration keys: a separate draw of n keys at positions 0..n-1.

Every stream is keyed by (config seed, layer, head, purpose) through numpy's
SeedSequence, so any subset can be regenerated independently.  The torch
variants draw the same distributions on a device for workloads too large for
numpy; they are seeded by torch generators and are not bit-identical to the
numpy draws (inputs are always handed to both sides as concrete tensors).
"""

from __future__ import annotations

import numpy as np

HEAD_DIM = 128
N_BLOCKS = HEAD_DIM // 2

PURPOSE_SIGMA = 0
PURPOSE_KEYS = 1
PURPOSE_VALUES = 2
PURPOSE_QUERIES = 3
PURPOSE_CALIB = 4
PURPOSE_NEW_TOKEN = 5


def rng_for(seed: int, layer: int, head: int, purpose: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(layer), int(head), int(purpose)])


def block_pairs(rope_layout: int = 0):
    """Dims of RoPE block i: (i, i+64) for half-split, (2i, 2i+1) interleaved."""
    if rope_layout == 0:
        return [(i, i + N_BLOCKS) for i in range(N_BLOCKS)]
    return [(2 * i, 2 * i + 1) for i in range(N_BLOCKS)]


def block_sigma(seed: int, layer: int, head: int, s_ln: float, heavy: bool = True) -> np.ndarray:
    """Per-block std sigma_i for one (layer, KV head), float64 [64]."""
    r = rng_for(seed, layer, head, PURPOSE_SIGMA)
    sig = np.exp(s_ln * r.standard_normal(N_BLOCKS))
    if heavy:
        sig[N_BLOCKS - 4:] *= 8.0
    return sig


def _rope_f64(x: np.ndarray, positions: np.ndarray, base: float, rope_layout: int) -> np.ndarray:
    """Rotate each 2-D block of x [T, 128] (float64) by position * theta_i."""
    pairs = block_pairs(rope_layout)
    lo = np.array([p[0] for p in pairs])
    hi = np.array([p[1] for p in pairs])
    theta = base ** (-2.0 * np.arange(N_BLOCKS, dtype=np.float64) / HEAD_DIM)
    ang = positions.astype(np.float64)[:, None] * theta[None, :]
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(x)
    out[:, lo] = x[:, lo] * c - x[:, hi] * s
    out[:, hi] = x[:, lo] * s + x[:, hi] * c
    return out


def draw_keys(rng: np.random.Generator, sigma: np.ndarray, positions: np.ndarray,
              base: float, rope_layout: int = 0) -> np.ndarray:
    """Keys [T, 128] float16, RoPE applied at `positions`."""
    t = len(positions)
    pairs = block_pairs(rope_layout)
    std = np.empty(HEAD_DIM)
    for i, (a, b) in enumerate(pairs):
        std[a] = sigma[i]
        std[b] = sigma[i]
    x = rng.standard_normal((t, HEAD_DIM)) * std[None, :]
    return _rope_f64(x, positions, base, rope_layout).astype(np.float16)


def draw_values(rng: np.random.Generator, t: int) -> np.ndarray:
    return rng.standard_normal((t, HEAD_DIM)).astype(np.float16)


class LayerInputs:
    """Inputs of one attention layer: K/V [H][T][128], q [Hq][128], calib [H][n][128]."""

    def __init__(self, k, v, q, calib, sigma):
        self.k = k
        self.v = v
        self.q = q
        self.calib = calib
        self.sigma = sigma


def layer_inputs(seed: int, layer: int, n_kv: int, group: int, t: int, base: float,
                 s_ln: float, n_calib: int = 512, rope_layout: int = 0,
                 heavy: bool = True, q_position: int | None = None) -> LayerInputs:
    """Numpy draw of one layer (small and medium workloads)."""
    qpos = t if q_position is None else q_position
    ks, vs, qs, cs, sg = [], [], [], [], []
    for h in range(n_kv):
        sig = block_sigma(seed, layer, h, s_ln, heavy)
        sg.append(sig)
        ks.append(draw_keys(rng_for(seed, layer, h, PURPOSE_KEYS), sig, np.arange(t), base, rope_layout))
        vs.append(draw_values(rng_for(seed, layer, h, PURPOSE_VALUES), t))
        rq = rng_for(seed, layer, h, PURPOSE_QUERIES)
        qs.append(draw_keys(rq, sig, np.full(group, qpos), base, rope_layout))
        cs.append(draw_keys(rng_for(seed, layer, h, PURPOSE_CALIB), sig, np.arange(n_calib), base, rope_layout))
    return LayerInputs(np.stack(ks), np.stack(vs), np.concatenate(qs, axis=0), np.stack(cs), np.stack(sg))


def calib_and_queries(seed: int, layer: int, n_kv: int, group: int, q_position: int, base: float,
                      s_ln: float, n_calib: int = 512, rope_layout: int = 0, heavy: bool = True):
    """Only the small parts of a layer (calibration keys, queries, sigma) for large workloads."""
    qs, cs, sg = [], [], []
    for h in range(n_kv):
        sig = block_sigma(seed, layer, h, s_ln, heavy)
        sg.append(sig)
        qs.append(draw_keys(rng_for(seed, layer, h, PURPOSE_QUERIES), sig, np.full(group, q_position), base, rope_layout))
        cs.append(draw_keys(rng_for(seed, layer, h, PURPOSE_CALIB), sig, np.arange(n_calib), base, rope_layout))
    return np.concatenate(qs, axis=0), np.stack(cs), np.stack(sg)


# --------------------------------------------------------------------------- torch (device) draws

def torch_keys(sigma: np.ndarray, positions, base: float, device, generator, rope_layout: int = 0):
    """Keys [T, 128] float16 drawn on `device` (float64 RoPE, like draw_keys)."""
    import torch
    pairs = block_pairs(rope_layout)
    lo = torch.tensor([p[0] for p in pairs], device=device)
    hi = torch.tensor([p[1] for p in pairs], device=device)
    sig = torch.tensor(sigma, dtype=torch.float64, device=device)
    pos = torch.as_tensor(positions, device=device).to(torch.float64)
    t = pos.numel()
    x = torch.randn((t, HEAD_DIM), dtype=torch.float32, device=device, generator=generator).to(torch.float64)
    xl = x[:, lo] * sig[None, :]
    xh = x[:, hi] * sig[None, :]
    theta = base ** (-2.0 * torch.arange(N_BLOCKS, dtype=torch.float64, device=device) / HEAD_DIM)
    ang = pos[:, None] * theta[None, :]
    c, s = torch.cos(ang), torch.sin(ang)
    out = torch.empty((t, HEAD_DIM), dtype=torch.float64, device=device)
    out[:, lo] = xl * c - xh * s
    out[:, hi] = xl * s + xh * c
    return out.to(torch.float16)


def torch_values(t: int, device, generator):
    import torch
    return torch.randn((t, HEAD_DIM), dtype=torch.float32, device=device, generator=generator).to(torch.float16)


def torch_generator(device, seed: int, layer: int, head: int, purpose: int):
    import torch
    g = torch.Generator(device=device)
    ss = np.random.SeedSequence([int(seed), int(layer), int(head), int(purpose)])
    g.manual_seed(int(ss.generate_state(1, dtype=np.uint64)[0] & ((1 << 63) - 1)))
    return g
