#!/usr/bin/env python
"""Benchmark of the Block-GTQ packed-cache decode path on GB300.

One step = one decode step of the whole workload: for every layer, append the
new token to the packed cache and run decode attention over the packed cache,
in one launch (bgtq_decode_step; --two-call: bgtq_quantize_append followed by
bgtq_decode_attn).  The default workload is the
Qwen2.5-3B-shaped 36-layer stack at 131072 cached tokens, K3V3 (2 KV heads,
16 query heads, batch 1).  The step's launches are captured once in a CUDA
graph and replayed.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gpu|reference]
                  [--workload NAME]

--impl reference times the CPU oracle (the plain restatement of the method)
on the host cores, on a bounded sample of the same workload.  Under torchrun
each rank runs an independent replica (the path shards by sequence/head with
no exchange); value = all ranks' tokens / max-over-ranks time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "packed-KV decode attn: tokens/s & achieved HBM GB/s (% of peak) at 128K ctx"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_step_qwen3b_128k.txt")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--workload", default="qwen3b_36l_128k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="build only the first N layers (profiling)")
    ap.add_argument("--eager", action="store_true", help="launch without a CUDA graph (profiling)")
    ap.add_argument("--recent", type=int, default=0,
                    help="keep the last W keys of every sequence in an fp16 recent-key buffer as well")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the fused prefill (bgtq_prefill_attn) of one layer and print its JSON line")
    ap.add_argument("--prefill-tokens", type=int, default=32768, help="prompt length of the fused-prefill measurement")
    ap.add_argument("--page-tokens", type=int, default=0,
                    help="paged cache: pages of P tokens in a shuffled pool instead of contiguous rows")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the measurements of the other workloads (profiling runs)")
    ap.add_argument("--two-call", action="store_true",
                    help="per layer bgtq_quantize_append + bgtq_decode_attn instead of the fused bgtq_decode_step")
    ap.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--sample-seconds", type=float, default=10.0, help=argparse.SUPPRESS)
    ap.add_argument("--sample-procs", type=int, default=1, help=argparse.SUPPRESS)
    return ap.parse_args()


def env_rank():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ----------------------------------------------------------------------------- CPU oracle sample

class OracleSample:
    """The oracle's decode step on one (layer, KV head) sample of the workload.

    One repetition unpacks and dequantises the sample's packed K/V cache,
    runs float64 attention for the head's G queries, and encodes + packs one
    new token.  Cost scales with the cached token-heads a step reads.
    """

    TOKENS = 8192

    def __init__(self, workload: str, layer: int = 0, head: int = 0):
        from oracle import bgtq_oracle as O
        from rope_aware_quantized_gb300 import synth, workloads
        self.O = O
        w = workloads.WORKLOADS[workload]
        layer %= w.layers
        head %= w.n_kv
        li = synth.layer_inputs(w.seed, layer, w.n_kv, w.group, self.TOKENS, w.rope_base, w.s_ln)
        self.q = li.q[head * w.group:(head + 1) * w.group]
        self.k, self.v = li.k[head], li.v[head]
        self.hs = O.head_state(workloads.calib_keys(w, layer, head), w.bits_per_key, w.v_bits,
                               workloads.plan_seed(w, layer), head)
        enc = O.encode_head(self.hs, self.k, self.v)
        self.krec, self.vrec, self.krho, self.vrho = enc["krec"], enc["vrec"], enc["krho"], enc["vrho"]

    def rep(self):
        O, hs = self.O, self.hs
        kcodes = O.unpack_k(self.krec, hs.kc, hs.bk)
        vcodes = O.unpack_v(self.vrec, hs.bv, self.TOKENS)
        khat = O.dequant(kcodes, self.krho, hs.kc)
        vhat = O.dequant(vcodes, self.vrho, hs.vc)
        O.attention(self.q, khat, vhat)
        nk, _ = O.encode(self.k[:1], hs.kc)
        O.pack_k(nk, hs.kc, hs.bk)
        nv, _ = O.encode(self.v[:1], hs.vc)
        O.pack_v(nv, hs.bv)


def single_thread_env():
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"


def host_cpu():
    """(logical cores, CPU model name) of this host."""
    model = None
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20)
        for line in r.stdout.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model and os.path.exists("/proc/cpuinfo"):
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                model = line.split(":", 1)[1].strip()
                break
    return os.cpu_count() or 1, model or "unknown"


# Worker state of the all-core oracle pool (spawned processes, one sample each).
_POOL_SAMPLE = None


def _pool_init(workload, counter, barrier):
    global _POOL_SAMPLE
    single_thread_env()
    with counter.get_lock():
        i = counter.value
        counter.value += 1
    from rope_aware_quantized_gb300 import workloads
    w = workloads.WORKLOADS[workload]
    _POOL_SAMPLE = OracleSample(workload, i % w.layers, (i // w.layers) % w.n_kv)
    _POOL_SAMPLE.rep()  # warm
    if barrier is not None:
        barrier.wait()


def _pool_run(seconds):
    """Repetitions of this worker's sample for about `seconds`."""
    reps, t0 = 0, time.perf_counter()
    while True:
        _POOL_SAMPLE.rep()
        reps += 1
        if time.perf_counter() - t0 >= seconds or reps >= 400:
            break
    return reps, time.perf_counter() - t0


def _pool_rep(_):
    t0 = time.perf_counter()
    _POOL_SAMPLE.rep()
    return time.perf_counter() - t0


def oracle_pool(workload: str, procs: int):
    """A spawned pool of `procs` single-threaded oracle workers, each holding
    the sample of a different (layer, KV head) of the workload."""
    import multiprocessing as mp
    single_thread_env()
    ctx = mp.get_context("spawn")
    counter = ctx.Value("i", 0)
    barrier = ctx.Barrier(procs)
    return ctx.Pool(procs, initializer=_pool_init, initargs=(workload, counter, barrier))


def oracle_sample(workload: str, seconds: float, procs: int):
    """Token-heads per second of the oracle's decode work: one process, or
    `procs` processes in parallel (each on its own sample)."""
    if procs <= 1:
        s = OracleSample(workload)
        s.rep()
        reps, t0 = 0, time.perf_counter()
        while True:
            s.rep()
            reps += 1
            el = time.perf_counter() - t0
            if el >= seconds or reps >= 400:
                break
        return {"token_heads_per_s": reps * s.TOKENS / el, "reps": reps, "tokens": s.TOKENS, "seconds": el,
                "procs": 1}
    pool = oracle_pool(workload, procs)
    try:
        res = pool.map(_pool_run, [seconds] * procs, chunksize=1)
    finally:
        pool.close()
        pool.join()
    reps = sum(r for r, _ in res)
    wall = max(e for _, e in res)
    return {"token_heads_per_s": reps * OracleSample.TOKENS / wall, "reps": reps, "tokens": OracleSample.TOKENS,
            "seconds": wall, "procs": procs}


def cpu_baseline(workload: str, seconds: float, procs: int):
    """Run the oracle sample in a child process (single-threaded numpy; a
    spawned pool of `procs` workers when procs > 1)."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    env.pop("LOCAL_RANK", None)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", "--workload", workload,
                        "--sample-seconds", str(seconds), "--sample-procs", str(procs)],
                       capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def step_token_heads(workload: str) -> int:
    from rope_aware_quantized_gb300 import workloads
    w = workloads.WORKLOADS[workload]
    return int(w.seq_lens().sum()) * w.n_kv * w.layers


def cpu_line_fields(workload: str, sample: dict):
    """Tokens/s of a whole decode step extrapolated from the sample rate."""
    from rope_aware_quantized_gb300 import workloads
    w = workloads.WORKLOADS[workload]
    token_heads = step_token_heads(workload)
    step_s = token_heads / sample["token_heads_per_s"]
    value = w.batch / step_s
    desc = (f"oracle decode work on {sample['procs']} process(es), each on its own (layer, KV head) sample of "
            f"{sample['tokens']} cached tokens ({sample['reps']} reps in {sample['seconds']:.1f} s): unpack + "
            f"dequantise K/V, float64 attention for {w.group} queries, encode + pack 1 token; the measured "
            f"token-head rate is extrapolated to the step's {token_heads} token-heads")
    return value, step_s, desc


def cpu_baseline_block(workload: str, seconds: float):
    """The line's cpu_baseline: the oracle on all host cores (value) and on
    one core, both extrapolated from bounded samples."""
    cores, model = host_cpu()
    procs = max(1, cores)
    one = cpu_baseline(workload, seconds, 1)
    allc = cpu_baseline(workload, seconds, procs) if procs > 1 else one
    v1, s1, d1 = cpu_line_fields(workload, one)
    va, sa, da = cpu_line_fields(workload, allc)
    token_heads = step_token_heads(workload)
    return {"value": va, "unit": UNIT, "cores": allc["procs"], "kind": "oracle", "sample": da,
            "extrapolated": True, "scale_factor": token_heads / (allc["procs"] * OracleSample.TOKENS),
            "ms_per_step": sa * 1000.0, "host_cores": cores, "cpu_model": model,
            "single_thread": {"value": v1, "unit": UNIT, "cores": 1, "ms_per_step": s1 * 1000.0,
                              "extrapolated": True, "scale_factor": token_heads / OracleSample.TOKENS,
                              "sample": d1}}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        load = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def code_digest(path: str) -> str:
    """sha256 prefix of a source file's code: // comments, surrounding
    whitespace and blank lines removed, so comment edits keep a profile valid."""
    import re
    lines = []
    for line in open(path, encoding="utf-8"):
        line = re.sub(r"//.*$", "", line).strip()
        if line:
            lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def traffic_from_profile():
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current decode kernel source."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    src = os.path.join(ROOT, "rope_aware_quantized_gb300", "csrc", "decode_kernel.cuh")
    sha = code_digest(src)
    vals = {}
    for line in open(PROFILE_SUMMARY):
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if (vals.get("decode_kernel.cuh code sha256 prefix", "").split() or [""])[0] != sha:
        return None
    try:
        return float(vals["dram bytes per launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(ms: float, dist=None, device="cpu") -> float:
    """The slowest rank's time: every rank ends with the same value."""
    if dist is None:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, batch: int, ms_per_step: float) -> float:
    """Whole-job tokens/s of `world` independent replicas (weak scaling): each
    replica decodes `batch` tokens per step; the job's step time is the
    slowest replica's."""
    return world * batch / (ms_per_step / 1000.0)


# ----------------------------------------------------------------------------- GPU arm

L2_BYTES = 129 * 2 ** 20  # GB300 L2


def decode_workload(wname: str, peaks: dict, stream, steps: int, warmup: int) -> dict:
    """Graph-timed fused decode steps (bgtq_decode_step per layer) of a named
    workload other than the headline one.  A workload whose step reads less
    than 4x L2 is run over enough replicas of its cache (separate buffers of
    the same content) that consecutive steps never find their bytes in L2;
    the graph then holds one step per replica."""
    import torch

    import rope_aware_quantized_gb300 as bg
    from rope_aware_quantized_gb300 import workloads

    w = workloads.WORKLOADS[wname]
    lens = w.seq_lens()
    max_len = int(lens.max())
    bpth = w.packed_bytes_per_token_head()
    layer_bytes = int(lens.sum()) * w.n_kv * bpth
    step_layers = w.layers
    replicas = 1
    if layer_bytes * w.layers < 4 * L2_BYTES:
        replicas = -(-4 * L2_BYTES // (layer_bytes * w.layers))
    layers = [workloads.build_layer(w, l % w.layers) for l in range(w.layers * replicas)]
    ws = torch.zeros(bg.bgtq_decode_attn_workspace(layers[0].plan, w.batch, max_len), dtype=torch.uint8, device="cuda")
    outs = [torch.empty((w.batch, w.n_q, 128), dtype=torch.float16, device="cuda") for _ in layers]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run_all():
        for ls, o in zip(layers, outs):
            bg.bgtq_decode_step(ls.plan, ls.q, ls.new_k[:, :, 0], ls.new_v[:, :, 0], ls.pos_new, ls.cache, ls.seq_lens,
                                max_len, o, ws, status=status)

    with torch.cuda.stream(stream):
        run_all()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        run_all()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    assert status.item() == 0, f"device status {status.item()}"
    ms = e0.elapsed_time(e1) / steps / replicas  # one decode step of the whole workload
    step_bytes = step_layers * (layer_bytes + w.batch * w.n_q * 128 * 2 * 2
                                + w.batch * w.n_kv * (2 * 256 + 16 * (w.bits_per_key // 128) + 16 * w.v_bits + 8))
    gbs = step_bytes / (ms / 1000.0) / 1e9
    r = {"tokens_per_s": w.batch / (ms / 1000.0), "ms_per_step": ms, "layers": w.layers, "batch": w.batch,
         "kv_heads": w.n_kv, "q_heads": w.n_q, "context_max": max_len, "context_mean": float(lens.mean()),
         "kv_bits": f"K{w.bits_per_key // 128}V{w.v_bits}", "packed_bytes_per_step": step_bytes,
         "fp16_kv_bytes_per_step": int(lens.sum()) * w.n_kv * 512 * w.layers,
         "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "bound": "hbm",
         "steps": steps, "warmup": warmup,
         "timing": "CUDA graph of per-layer bgtq_decode_step calls, events on the launching stream",
         "l2": (f"{replicas} cache replicas cycled ({replicas * layer_bytes * w.layers / 1e6:.0f} MB > 4x L2)"
                if replicas > 1 else "inputs larger than L2, no flush")}
    del layers, outs, ws
    torch.cuda.empty_cache()
    return r


def ragged_prefill(wname: str, peaks: dict, stream) -> dict:
    """The ragged workload's prefill pass: every sequence's full context of
    fp16 K and V rows (batch x KV heads x context tokens) encoded into an
    empty packed cache by one bgtq_quantize_append call."""
    import torch

    import rope_aware_quantized_gb300 as bg
    from rope_aware_quantized_gb300 import workloads

    w = workloads.WORKLOADS[wname]
    B, H, T = w.batch, w.n_kv, w.context
    plan = workloads.build_plan(w, 0)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(20262)
    k = torch.randn((B, H, T, 128), generator=gen, device="cuda").half()
    v = torch.randn((B, H, T, 128), generator=gen, device="cuda").half()
    cache = bg.Cache(plan, B, T)
    pos = torch.zeros(B, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    times = []
    with torch.cuda.stream(stream):
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            bg.bgtq_quantize_append(plan, k, v, pos, cache, status=status)
            b.record(stream)
            times.append((a, b))
    torch.cuda.synchronize()
    assert status.item() == 0, f"append status {status.item()}"
    ms = statistics.median(a.elapsed_time(b) for a, b in times[2:])
    rows = B * H * T
    nbytes = rows * 128 * 2 * 2 + rows * (16 * (w.bits_per_key // 128) + 16 * w.v_bits + 8)
    gbs = nbytes / (ms / 1000.0) / 1e9
    del k, v, cache
    torch.cuda.empty_cache()
    return {"tokens": B * T, "batch": B, "kv_heads": H, "tokens_per_sequence": T, "ms_per_launch": ms,
            "tokens_per_s": B * T / (ms / 1000.0), "bytes_per_launch": nbytes, "achieved": gbs, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "bound": "hbm",
            "bytes": "fp16 K and V rows read + packed K/V records and both norms written"}


def measure_prefill(w, plan, tokens: int, peaks: dict, stream) -> dict:
    """The quantize-append kernel alone on a prefill: `tokens` fp16 K/V rows
    per (sequence, KV head) of one layer encoded into an empty packed cache in
    one bgtq_quantize_append call (the inputs, 2 * batch * heads * tokens *
    256 bytes, are larger than L2 at the default workload; no flush)."""
    import torch

    import rope_aware_quantized_gb300 as bg

    B, H = w.batch, w.n_kv
    gen = torch.Generator(device="cuda")
    gen.manual_seed(20260)
    k = torch.randn((B, H, tokens, 128), generator=gen, device="cuda").half()
    v = torch.randn((B, H, tokens, 128), generator=gen, device="cuda").half()
    cache = bg.Cache(plan, B, tokens + (tokens & 1))
    pos = torch.zeros(B, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    times = []
    with torch.cuda.stream(stream):
        for i in range(8):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            bg.bgtq_quantize_append(plan, k, v, pos, cache, status=status)
            b.record(stream)
            times.append((a, b))
    torch.cuda.synchronize()
    assert status.item() == 0, f"append status {status.item()}"
    ms = statistics.median(a.elapsed_time(b) for a, b in times[3:])
    rows = B * H * tokens
    read = rows * 128 * 2 * 2
    written = rows * (16 * (w.bits_per_key // 128) + 16 * w.v_bits + 8)
    gbs = (read + written) / (ms / 1000.0) / 1e9
    del k, v, cache
    return {"tokens_per_s": B * tokens / (ms / 1000.0), "ms_per_launch": ms, "tokens": tokens, "batch": B,
            "kv_heads": H, "bytes_per_launch": read + written, "achieved": gbs, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "bound": "hbm",
            "bytes": "fp16 K and V rows read + packed K/V records and both norms written"}


def measure_prefill_attn(w, plan, tokens: int, peaks: dict, stream) -> dict:
    """The fused prefill (bgtq_prefill_attn: causal attention over the
    prompt's fp16 K/V plus the packed records of the prompt) on one layer of
    the workload's shape: `tokens` positions per sequence, fp16 output.
    Algorithmic work: 4 * 128 flops per (query head, query row, key) pair of
    the causal triangle (Q K^T and P V)."""
    import torch

    import rope_aware_quantized_gb300 as bg

    B, H, Hq = w.batch, w.n_kv, w.n_q
    gen = torch.Generator(device="cuda")
    gen.manual_seed(20261)
    q = torch.randn((B, Hq, tokens, 128), generator=gen, device="cuda").half()
    k = torch.randn((B, H, tokens, 128), generator=gen, device="cuda").half()
    v = torch.randn((B, H, tokens, 128), generator=gen, device="cuda").half()
    out = torch.empty_like(q)
    cache = bg.Cache(plan, B, tokens + (tokens & 1))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    times = []
    with torch.cuda.stream(stream):
        for i in range(6):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            bg.bgtq_prefill_attn(plan, q, k, v, cache, out, status=status)
            b.record(stream)
            times.append((a, b))
    torch.cuda.synchronize()
    assert status.item() == 0, f"prefill status {status.item()}"
    ms = statistics.median(a.elapsed_time(b) for a, b in times[2:])
    flops = 4.0 * 128 * B * Hq * tokens * (tokens + 1) / 2
    tf = flops / (ms / 1000.0) / 1e12
    del q, k, v, out, cache
    return {"tokens": tokens, "batch": B, "query_heads": Hq, "kv_heads": H, "ms_per_launch": ms,
            "tokens_per_s": B * tokens / (ms / 1000.0), "achieved": tf, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"], "bound": "tensor",
            "flops": "4 * 128 per (query head, row, key <= row): causal Q K^T and P V; fp16 tcgen05 MMAs, fp32 accumulators in tensor memory",
            "peak_note": "measured dense bf16 (burst); fp16 has the same nominal tensor rate"}


def measure_chunk_prefill(w, plan, prefix: int, chunk: int, peaks: dict, stream) -> dict:
    """Chunked prefill (bgtq_prefill_chunk_attn: the chunk's records by the
    append, then attention of every chunk row over the packed prefix and the
    chunk's own fp16 K/V) on one layer of the workload's shape: `prefix`
    cached tokens per sequence, a chunk of `chunk` tokens, fp16 output.
    Algorithmic work: 4 * 128 flops per (query head, chunk row, visible key),
    the prefix keys all visible, the chunk's causally."""
    import torch

    import rope_aware_quantized_gb300 as bg

    B, H, Hq = w.batch, w.n_kv, w.n_q
    gen = torch.Generator(device="cuda")
    gen.manual_seed(20262)
    cache = bg.Cache(plan, B, prefix + chunk + ((prefix + chunk) & 1))
    kp = torch.randn((B, H, prefix, 128), generator=gen, device="cuda").half()
    vp = torch.randn((B, H, prefix, 128), generator=gen, device="cuda").half()
    bg.bgtq_quantize_append(plan, kp, vp, torch.zeros(B, dtype=torch.int32, device="cuda"), cache)
    del kp, vp
    q = torch.randn((B, Hq, chunk, 128), generator=gen, device="cuda").half()
    k = torch.randn((B, H, chunk, 128), generator=gen, device="cuda").half()
    v = torch.randn((B, H, chunk, 128), generator=gen, device="cuda").half()
    pos = torch.full((B,), prefix, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    ws = torch.empty(bg.bgtq_prefill_chunk_workspace(plan, B, prefix), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    times = []
    with torch.cuda.stream(stream):
        for i in range(6):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            bg.bgtq_prefill_chunk_attn(plan, q, k, v, pos, cache, out, max_prefix=prefix, workspace=ws, status=status)
            b.record(stream)
            times.append((a, b))
    torch.cuda.synchronize()
    assert status.item() == 0, f"chunk prefill status {status.item()}"
    ms = statistics.median(a.elapsed_time(b) for a, b in times[2:])
    flops = 4.0 * 128 * B * Hq * chunk * (prefix + (chunk + 1) / 2)
    tf = flops / (ms / 1000.0) / 1e12
    del q, k, v, out, cache, ws
    return {"prefix_tokens": prefix, "chunk_tokens": chunk, "batch": B, "query_heads": Hq, "kv_heads": H,
            "ms_per_call": ms, "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": tf / peaks["bf16_tflops"], "bound": "tensor",
            "flops": "4 * 128 per (query head, chunk row, visible key); the prefix decoded once into the "
                     "workspace, then on tcgen05 with fp16 hi + lo query and probability splits (twice the MMAs "
                     "of the counted flops), the chunk as the fused prefill; the call includes the append",
            "peak_note": "measured dense bf16 (burst); fp16 has the same nominal tensor rate"}


def run_gpu(args):
    import numpy as np
    import torch

    import rope_aware_quantized_gb300 as bg
    from rope_aware_quantized_gb300 import workloads

    rank, local_rank, world = env_rank()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    bg._native.lib()
    w = workloads.WORKLOADS[args.workload]
    lens = w.seq_lens()
    max_len = int(lens.max())
    L, B = (args.layers or w.layers), w.batch
    if args.prefill_only:
        bits, energy = zip(*[bg.bgtq_alloc_bits(workloads.calib_keys(w, 0, h), w.bits_per_key) for h in range(w.n_kv)])
        plan = bg.bgtq_plan_create(np.stack(bits), np.stack(energy), w.group, w.bits_per_key, w.v_bits,
                                   workloads.plan_seed(w, 0))
        peaks, _ = load_peaks()
        r = measure_prefill_attn(w, plan, args.prefill_tokens, peaks, torch.cuda.Stream())
        rc = measure_chunk_prefill(w, plan, args.prefill_tokens, args.prefill_tokens // 4, peaks, torch.cuda.Stream())
        ra = measure_prefill(w, plan, max_len, peaks, torch.cuda.Stream())
        if rank == 0:
            print(json.dumps({"metric": "fused_prefill_tflops", "value": r["achieved"], "unit": "TFLOP/s",
                              "config": {"workload": w.name, "prompt_tokens": args.prefill_tokens},
                              "prefill_attn": r, "chunk_prefill": rc, "append_prefill": ra}), flush=True)
        return

    # device buffers of all layers' per-step inputs/outputs (views per layer)
    q_all = torch.empty((L, B, w.n_q, 128), dtype=torch.float16, device="cuda")
    nk_all = torch.empty((L, B, w.n_kv, 1, 128), dtype=torch.float16, device="cuda")
    nv_all = torch.empty_like(nk_all)
    out_all = torch.empty((L, B, w.n_q, 128), dtype=torch.float16, device="cuda")
    layers = []
    for l in range(L):
        ls = workloads.build_layer(w, l, recent=args.recent, page_tokens=args.page_tokens)
        q_all[l].copy_(ls.q)
        nk_all[l].copy_(ls.new_k)
        nv_all[l].copy_(ls.new_v)
        ls.q, ls.new_k, ls.new_v = q_all[l], nk_all[l], nv_all[l]
        layers.append(ls)
    torch.cuda.synchronize()
    ws = torch.zeros(bg.bgtq_decode_attn_workspace(layers[0].plan, B, max_len), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()

    fused = not args.two_call
    nk_tok = [nk_all[l][:, :, 0] for l in range(L)]  # [B][H][128] views of the new tokens
    nv_tok = [nv_all[l][:, :, 0] for l in range(L)]

    def layer_call(l, ls):
        if fused:
            bg.bgtq_decode_step(ls.plan, ls.q, nk_tok[l], nv_tok[l], ls.pos_new, ls.cache, ls.seq_lens, max_len,
                                out_all[l], ws, status=status)
        else:
            bg.bgtq_quantize_append(ls.plan, ls.new_k, ls.new_v, ls.pos_new, ls.cache, status=status)
            bg.bgtq_decode_attn(ls.plan, ls.q, ls.cache, ls.seq_lens, max_len, out_all[l], ws, status=status)

    def step():
        for l, ls in enumerate(layers):
            layer_call(l, ls)

    with torch.cuda.stream(stream):
        step()
        step()
    torch.cuda.synchronize()
    assert status.item() == 0, f"device status {status.item()}"
    if args.eager:
        class _Eager:
            def replay(self):
                step()
        graph = _Eager()
    else:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
    launches_per_step = L if fused else 2 * L

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    barrier()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    barrier()
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, "cuda")
    value = replica_throughput(world, B, ms)

    # dominant kernel alone: CUDA events around each decode launch on its stream
    durs = []
    with torch.cuda.stream(stream):
        for _ in range(3):
            for l, ls in enumerate(layers):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                if fused:
                    bg.bgtq_decode_step(ls.plan, ls.q, nk_tok[l], nv_tok[l], ls.pos_new, ls.cache, ls.seq_lens,
                                        max_len, out_all[l], ws, status=status)
                else:
                    bg.bgtq_decode_attn(ls.plan, ls.q, ls.cache, ls.seq_lens, max_len, out_all[l], ws, status=status)
                b.record(stream)
                durs.append((a, b))
    torch.cuda.synchronize()
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in durs)
    bpth = w.packed_bytes_per_token_head()
    # packed K/V codes + norms of every cached token, q read and out written;
    # the fused step also reads the new token and writes its records
    decode_bytes = int(lens.sum()) * w.n_kv * bpth + B * w.n_q * 128 * 2 * 2
    if fused:
        decode_bytes += B * w.n_kv * (2 * 256 + 16 * (w.bits_per_key // 128) + 16 * w.v_bits + 8)
    if args.recent:  # the fp16 keys of the window are read as well
        decode_bytes += int(np.minimum(lens, args.recent).sum()) * w.n_kv * 256
    peaks, peak_kind = load_peaks()
    iso_achieved = decode_bytes / (launch_ms / 1000.0) / 1e9
    traffic = traffic_from_profile()
    step_bytes = L * decode_bytes
    # the dominant kernel inside the timed step: every launch of the step is
    # this kernel (the fused step) or alternates with the 1-token append
    # (two-call), so its in-step time per launch is at most ms_per_step / L
    in_step_launch_ms = ms / L
    achieved = step_bytes / (ms / 1000.0) / 1e9

    prefill = measure_prefill(w, layers[0].plan, max_len, peaks, stream)
    prefill_attn = measure_prefill_attn(w, layers[0].plan, min(max_len, args.prefill_tokens), peaks, stream)
    chunk_prefill = measure_chunk_prefill(w, layers[0].plan, min(max_len, args.prefill_tokens),
                                          min(max_len, args.prefill_tokens) // 4, peaks, stream)

    # end to end: pinned host inputs -> device, graph replay, outputs -> host
    hq = torch.empty(q_all.shape, dtype=q_all.dtype, pin_memory=True)
    hk = torch.empty(nk_all.shape, dtype=nk_all.dtype, pin_memory=True)
    hv = torch.empty(nv_all.shape, dtype=nv_all.dtype, pin_memory=True)
    ho = torch.empty(out_all.shape, dtype=out_all.dtype, pin_memory=True)
    hq.copy_(q_all)
    hk.copy_(nk_all)
    hv.copy_(nv_all)
    torch.cuda.synchronize()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with torch.cuda.stream(stream):
        x0.record(stream)
        for _ in range(args.steps):
            q_all.copy_(hq, non_blocking=True)
            nk_all.copy_(hk, non_blocking=True)
            nv_all.copy_(hv, non_blocking=True)
            graph.replay()
            ho.copy_(out_all, non_blocking=True)
        x1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(x0.elapsed_time(x1) / args.steps, dist, "cuda")
    assert status.item() == 0, f"device status {status.item()}"

    # the other workloads of the path, each in its own measurement (rank 0 of
    # a single-GPU run; the headline workload's buffers are released first)
    others = {}
    if rank == 0 and world == 1 and not args.headline_only and args.workload == "qwen3b_36l_128k" and not args.layers:
        del graph, layers, q_all, nk_all, nv_all, out_all, nk_tok, nv_tok, hq, hk, hv, ho
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        k_other, w_other = max(5, args.steps // 2), max(3, args.warmup)
        for name in ("qwen3b_36l_512k", "llama8b_ragged_b32", "llama8b_layer", "tiny"):
            others[name] = decode_workload(name, peaks, stream, k_other, w_other)
        others["llama8b_ragged_b32"]["prefill"] = ragged_prefill("llama8b_ragged_b32", peaks, stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_block(args.workload, args.sample_seconds)

    if rank == 0:
        fp16_bytes = int(lens.sum()) * w.n_kv * 512 * L
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp16", "data": "synthetic",
            "config": {
                "workload": w.name if L == w.layers else f"{w.name}[first {L} layers]", "layers": L, "kv_heads": w.n_kv, "q_heads": w.n_q, "head_dim": 128,
                "context": int(max_len), "batch": B, "kv_bits": f"K{w.bits_per_key // 128}V{w.v_bits}",
                "step": ("per layer: bgtq_decode_step (quantize-append 1 token + decode attention, one launch)" if fused
                         else "per layer: bgtq_quantize_append 1 token + bgtq_decode_attn")
                        + (" (eager)" if args.eager else " (CUDA graph)"),
                "packed_bytes_per_step": step_bytes, "fp16_kv_bytes_per_step": fp16_bytes,
                "compute": "fp16 mma operands (hi+lo split of q and p), fp32 accumulate; fp32 encoder",
                "l2": "inputs larger than L2 (packed cache per step >> 129 MB L2), no flush",
                "parallelism": f"replicas x{world}",
                **({"recent_fp16_keys": args.recent} if args.recent else {}),
                **({"page_tokens": args.page_tokens} if args.page_tokens else {}),
            },
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                         "kernel": "decode_step" if fused else "decode_attn",
                         "launch_ms_in_step": in_step_launch_ms, "bytes_per_launch": decode_bytes,
                         "timing": "in-step: step bytes / ms_per_step of the graph-timed step "
                                   f"({launches_per_step} launches per step, dependent launches overlapping)",
                         "isolated": {"launch_ms": launch_ms, "achieved": iso_achieved,
                                      "frac": iso_achieved / peaks["hbm_gbs"],
                                      "timing": "CUDA events around each launch (breaks the launch overlap)"},
                         "peak_kind": f"{peak_kind} (copy, burst)"},
            "e2e": {"value": replica_throughput(world, B, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "path": "pinned H2D of q/new K/V, graph of the API calls, D2H of out"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "achieved_step_gbs": step_bytes / (ms / 1000.0) / 1e9,
        }
        line["append_prefill"] = prefill
        line["prefill_attn"] = prefill_attn
        line["chunk_prefill"] = chunk_prefill
        if others:
            line["workloads"] = others
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- reference arm (CPU oracle)

def run_reference(args):
    """The oracle as the reference arm: each step runs one repetition of the
    oracle's decode work on every host core (one (layer, KV head) sample per
    process) and is extrapolated to the whole step's token-heads."""
    rank, _, world = env_rank()
    if rank != 0:
        return
    single_thread_env()
    from rope_aware_quantized_gb300 import workloads
    w = workloads.WORKLOADS[args.workload]
    cores, model = host_cpu()
    procs = max(1, cores)
    pool = oracle_pool(args.workload, procs)
    try:
        times = []
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            pool.map(_pool_rep, range(procs), chunksize=1)
            dt = time.perf_counter() - t0
            if i >= args.warmup:
                times.append(dt)
    finally:
        pool.close()
        pool.join()
    th = procs * OracleSample.TOKENS
    s = {"token_heads_per_s": th * len(times) / sum(times), "reps": procs * len(times), "tokens": OracleSample.TOKENS,
         "seconds": sum(times), "procs": procs}
    value, step_s, desc = cpu_line_fields(args.workload, s)
    token_heads = step_token_heads(args.workload)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1000.0, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "layers": w.layers, "kv_heads": w.n_kv, "q_heads": w.n_q,
                   "context": int(w.seq_lens().max()), "batch": w.batch,
                   "kv_bits": f"K{w.bits_per_key // 128}V{w.v_bits}"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": procs, "kind": "oracle", "sample": desc,
                         "extrapolated": True, "scale_factor": token_heads / th, "host_cores": cores,
                         "cpu_model": model, "measured_ms_per_sample_step": 1000.0 * sum(times) / len(times)},
        "extrapolated": {"from_token_heads_per_step": th, "to_token_heads_per_step": token_heads,
                         "note": "each timed step runs the oracle on a bounded sample; ms_per_step and value are "
                                 "the sample's token-head rate scaled to the full step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.oracle_sample:
        single_thread_env()
        print(json.dumps(oracle_sample(args.workload, args.sample_seconds, args.sample_procs)), flush=True)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
