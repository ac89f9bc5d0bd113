"""RoPE-logit fidelity report: Block-GTQ against uniform TQ-MSE keys.

For every layer of a workload's layer stack, the keys of `--tokens`
positions are quantize-appended twice, once with the layer's Block-GTQ plan
(per-block widths from the calibration energies) and once with the uniform
TQ-MSE plan at the same key budget (every block at bK bits, equal energies),
and bgtq_logit_mae gives the mean absolute attention-logit error per query
head.  Prints one JSON line.  (Review §3 Method & Key Results: Block-GTQ
lowers the RoPE-logit error against uniform TQ-MSE at matched budgets.)

    python -m rope_aware_quantized_gb300.fidelity [--workload NAME] [--tokens T] [--layers N]
"""

from __future__ import annotations

import argparse
import json

import numpy as np


def layer_report(w, layer: int, tokens: int, torch):
    from . import Cache, bgtq_alloc_bits, bgtq_logit_mae, bgtq_plan_create, bgtq_quantize_append, synth, workloads

    bk = w.bits_per_key // 128
    bits, energy = zip(*[bgtq_alloc_bits(workloads.calib_keys(w, layer, h), w.bits_per_key) for h in range(w.n_kv)])
    seed = workloads.plan_seed(w, layer)
    plans = {
        "block_gtq": bgtq_plan_create(np.stack(bits), np.stack(energy), w.group, w.bits_per_key, w.v_bits, seed),
        "uniform": bgtq_plan_create(np.full((w.n_kv, 64), bk, np.uint8), np.full((w.n_kv, 64), 2.0), w.group,
                                    w.bits_per_key, w.v_bits, seed),
    }
    ks, vs, qs = [], [], []
    for h in range(w.n_kv):
        sig = synth.block_sigma(w.seed, layer, h, w.s_ln)
        gk = synth.torch_generator("cuda", w.seed, layer, h, synth.PURPOSE_KEYS)
        gv = synth.torch_generator("cuda", w.seed, layer, h, synth.PURPOSE_VALUES)
        gq = synth.torch_generator("cuda", w.seed, layer, h, synth.PURPOSE_QUERIES)
        ks.append(synth.torch_keys(sig, torch.arange(tokens, device="cuda"), w.rope_base, "cuda", gk))
        vs.append(synth.torch_values(tokens, "cuda", gv))
        qs.append(synth.torch_keys(sig, torch.full((w.group,), tokens, device="cuda"), w.rope_base, "cuda", gq))
    k = torch.stack(ks)[None].contiguous()
    v = torch.stack(vs)[None].contiguous()
    q = torch.cat(qs)[None].contiguous()
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = {}
    ms = None
    for name, plan in plans.items():
        cache = Cache(plan, 1, tokens + (tokens & 1))
        bgtq_quantize_append(plan, k, v, pos, cache)
        mae = torch.empty((1, w.n_q), dtype=torch.float32, device="cuda")
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        bgtq_logit_mae(plan, q, k, cache, tokens, mae)
        b.record()
        torch.cuda.synchronize()
        out[name] = float(mae.mean().item())
        ms = a.elapsed_time(b)
    return out, ms


def main():
    import torch

    from . import workloads

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="qwen3b_36l_128k")
    ap.add_argument("--tokens", type=int, default=8192)
    ap.add_argument("--layers", type=int, default=0)
    args = ap.parse_args()
    w = workloads.WORKLOADS[args.workload]
    n_layers = args.layers or w.layers
    rows, times = [], []
    for layer in range(n_layers):
        r, ms = layer_report(w, layer, args.tokens, torch)
        rows.append({"layer": layer, "block_gtq": r["block_gtq"], "uniform": r["uniform"],
                     "ratio": r["uniform"] / r["block_gtq"]})
        times.append(ms)
    ratios = [x["ratio"] for x in rows]
    print(json.dumps({
        "diagnostic": "rope_logit_mae (mean |scale q.k - scale q.khat| over cached tokens, per query head)",
        "workload": w.name, "layers": n_layers, "tokens": args.tokens, "kv_bits": f"K{w.bits_per_key // 128}",
        "data": "synthetic",
        "block_gtq_mean": float(np.mean([x["block_gtq"] for x in rows])),
        "uniform_mean": float(np.mean([x["uniform"] for x in rows])),
        "ratio_uniform_over_block_gtq": {"min": float(min(ratios)), "median": float(np.median(ratios)),
                                         "max": float(max(ratios))},
        "kernel_ms_median": float(np.median(times)),
        "per_layer": rows,
    }), flush=True)


if __name__ == "__main__":
    main()
