"""Named decode workloads and a builder that prepares them on the GPU.

The shapes are the decode settings the Block-GTQ abstract evaluates
("RoPE-Aware Bit Allocation for KV-Cache Quantization", English abstract:
Llama-3.1-8B K2V2, Qwen2.5-3B packed K3V3 at 128K, feasibility at 512K,
K3V2) with synthetic tensors of those shapes (see ``synth``).  Building a
workload uses only the library's public API: allocation from calibration
keys, plan creation, cache allocation and a prefill through
``bgtq_quantize_append``.
"""

from __future__ import annotations

import dataclasses

import numpy as np

from . import Cache, Plan, bgtq_alloc_bits, bgtq_plan_create, bgtq_quantize_append, synth


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    n_kv: int
    group: int
    context: int          # cached tokens per sequence after the decode append
    batch: int
    rope_base: float
    s_ln: float
    bits_per_key: int
    v_bits: int
    seed: int
    ragged: tuple = ()    # (lo, hi) of uniformly drawn per-sequence lengths

    @property
    def n_q(self):
        return self.n_kv * self.group

    def seq_lens(self) -> np.ndarray:
        if self.ragged:
            r = np.random.default_rng([self.seed, 999])
            return r.integers(self.ragged[0], self.ragged[1] + 1, self.batch).astype(np.int64)
        return np.full(self.batch, self.context, dtype=np.int64)

    def packed_bytes_per_token_head(self) -> int:
        return 16 * (self.bits_per_key // 128) + 16 * self.v_bits + 8


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 4, 4096, 1, 1e4, 1.0, 384, 3, 1),
    "llama8b_layer": Workload("llama8b_layer", 1, 8, 4, 32768, 1, 5e5, 1.2, 256, 2, 2),
    "qwen3b_36l_128k": Workload("qwen3b_36l_128k", 36, 2, 8, 131072, 1, 1e6, 1.2, 384, 3, 3),
    "qwen3b_36l_512k": Workload("qwen3b_36l_512k", 36, 2, 8, 524288, 1, 1e6, 1.2, 384, 2, 4),
    "llama8b_ragged_b32": Workload("llama8b_ragged_b32", 1, 8, 4, 65536, 32, 5e5, 1.2, 256, 2, 5, (4096, 65536)),
}


class LayerState:
    """Device state of one layer: plan, cache, query, new token and lengths."""

    def __init__(self, plan: Plan, cache: Cache, q, new_k, new_v, seq_lens, pos_new, host=None):
        self.plan = plan
        self.cache = cache
        self.q = q
        self.new_k = new_k
        self.new_v = new_v
        self.seq_lens = seq_lens
        self.pos_new = pos_new
        self.host = host or {}


def build_layer(w: Workload, layer: int, device="cuda", keep_host=(), capacity: int | None = None,
                prefill_chunk: int = 1 << 16, recent: int = 0, page_tokens: int = 0) -> LayerState:
    """Calibrate, plan, allocate and prefill one layer.

    Each sequence b holds tokens 0 .. len_b - 2 after the prefill; the decode
    step appends token len_b - 1 (the "new" token) and attends over len_b.
    `keep_host` lists (sequence, KV head) pairs whose full fp16 K/V are
    copied back to host memory, for checks against an independent model.
    page_tokens = P > 0 builds a paged cache whose page table is a seeded
    random permutation of the pool (no two neighbouring pages adjacent in
    memory by construction).
    """
    import torch
    lens = w.seq_lens()
    cap = capacity or int(((lens.max() + 1) // 2) * 2)
    if page_tokens:
        cap = -(-cap // page_tokens) * page_tokens
    qpos = lens - 1
    plan = build_plan(w, layer)
    cache = Cache(plan, w.batch, cap, device, recent=recent, page_tokens=page_tokens)
    if page_tokens:
        perm = np.random.default_rng([w.seed, layer, 0x9A6E]).permutation(cache.n_pages).astype(np.int32)
        cache.page_table.copy_(torch.from_numpy(perm.reshape(w.batch, cache.max_pages)).to(device))
    q = torch.empty((w.batch, w.n_q, 128), dtype=torch.float16, device=device)
    new_k = torch.empty((w.batch, w.n_kv, 1, 128), dtype=torch.float16, device=device)
    new_v = torch.empty_like(new_k)
    host = {}
    for bi in range(w.batch):
        n_pre = int(lens[bi]) - 1
        ks, vs = [], []
        for h in range(w.n_kv):
            sig = synth.block_sigma(w.seed, layer, h, w.s_ln)
            sub = h * 100000 + bi
            gk = synth.torch_generator(device, w.seed, layer, sub, synth.PURPOSE_KEYS)
            gv = synth.torch_generator(device, w.seed, layer, sub, synth.PURPOSE_VALUES)
            gq = synth.torch_generator(device, w.seed, layer, sub, synth.PURPOSE_QUERIES)
            k_all = synth.torch_keys(sig, torch.arange(n_pre + 1, device=device), w.rope_base, device, gk)
            v_all = synth.torch_values(n_pre + 1, device, gv)
            q[bi, h * w.group:(h + 1) * w.group] = synth.torch_keys(
                sig, torch.full((w.group,), int(qpos[bi]), device=device), w.rope_base, device, gq)
            new_k[bi, h, 0] = k_all[n_pre]
            new_v[bi, h, 0] = v_all[n_pre]
            if (bi, h) in set(keep_host):
                host[(bi, h)] = (k_all.cpu().numpy(), v_all.cpu().numpy())
            ks.append(k_all)
            vs.append(v_all)
        K = torch.stack(ks)
        V = torch.stack(vs)
        del ks, vs
        view = cache.sequence_view(bi)
        for c0 in range(0, n_pre, prefill_chunk):
            c1 = min(n_pre, c0 + prefill_chunk)
            pos = torch.tensor([c0], dtype=torch.int32, device=device)
            bgtq_quantize_append(plan, K[:, c0:c1].unsqueeze(0).contiguous(), V[:, c0:c1].unsqueeze(0).contiguous(),
                                 pos, view)
        del K, V
    seq_lens = torch.tensor(lens, dtype=torch.int32, device=device)
    pos_new = torch.tensor(lens - 1, dtype=torch.int32, device=device)
    torch.cuda.synchronize()
    return LayerState(plan, cache, q, new_k, new_v, seq_lens, pos_new, host)


def build_plan(w: Workload, layer: int) -> Plan:
    """Block-GTQ allocation of every KV head of (workload, layer) from its
    calibration keys, and the layer's plan."""
    bits, energy = [], []
    for h in range(w.n_kv):
        b, e = bgtq_alloc_bits(calib_keys(w, layer, h), w.bits_per_key, 8, 0)
        bits.append(b)
        energy.append(e)
    return bgtq_plan_create(np.stack(bits), np.stack(energy), w.group, w.bits_per_key, w.v_bits, plan_seed(w, layer))


def plan_seed(w: Workload, layer: int) -> int:
    """Seed of the rotation signs of (workload, layer)."""
    return ((w.seed << 32) ^ (layer * 0x9E37) ^ 0x5BD1E995) & ((1 << 64) - 1)


def calib_keys(w: Workload, layer: int, head: int) -> np.ndarray:
    """The 512 calibration keys of (workload, layer, KV head), float16."""
    sig = synth.block_sigma(w.seed, layer, head, w.s_ln)
    return synth.draw_keys(synth.rng_for(w.seed, layer, head, synth.PURPOSE_CALIB), sig, np.arange(512), w.rope_base)
