#!/usr/bin/env python3
"""Benchmark of the paged-KV decode step on GB300.

One step = the whole hot path for one decode iteration of the Qwen3-1.7B
attention shape (one layer): cache_write of the 34 sequences' new K/V rows,
then paged decode attention of 34 sequences x 640 tokens (16 q / 8 kv heads,
head_dim 128, 16-token blocks, 22,048-token pool, shuffled block tables).
Synthetic bf16 N(0,1) data from pkv_workloads (no weights, no dataset).

Timing: inputs resident in HBM; 8 replicas of the pool/tables/q (8 x 90 MB,
larger than the 129 MB L2) are rotated step by step, so every step reads its
K/V from HBM.  The steps are replayed from CUDA graphs (one graph per cycle
through the replicas) and timed with CUDA events on the launching stream,
synchronised on both sides.  The decode kernel's own average duration is
timed the same way over decode-only replays.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on
the host cores instead, on a bounded sample of the same workload.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention: achieved HBM GB/s vs GB300 peak; sequences/s per layer"
UNIT = "seqs/s"
CONFIG_ID = 2
WORKLOAD = "qwen3-1.7b paged decode: 34 seqs x 640 ctx, 16q/8kv heads, d128, block 16, pool 22048 tokens"

# DRAM traffic of one decode launch on this workload from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), and the hash of the kernel
# sources it was taken on; reported only while the sources still match.
NCU_TRAFFIC = {"bytes": None, "sources_sha": None, "capture": None}
KERNEL_SOURCES = ["paged_kv_cache_291_gb300/csrc/decode.cu", "paged_kv_cache_291_gb300/csrc/pkv_device.cuh"]


def sources_sha() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------- multi-rank host logic

def shard_sequences(num_seqs_per_rank: int, rank: int):
    """Weak scaling: every rank owns its own batch of sequences (its own pool
    and block tables); global sequence ids of rank r are r*B .. r*B+B-1."""
    return list(range(rank * num_seqs_per_rank, (rank + 1) * num_seqs_per_rank))


def reduce_max(value: float, dist=None) -> float:
    """Max over ranks of a host float (the slowest rank sets the job time)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    backend = dist.get_backend()
    dev = "cuda" if backend == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []
        self._thr = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self._thr = threading.Thread(target=self._read, daemon=True)
        self._thr.start()
        time.sleep(0.3)

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def stop(self):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._thr is not None:
                self._thr.join(timeout=2)

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, ln in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smmax=float(parts[2]), hw=parts[5], hwt=parts[6], swt=parts[7],
                                 swp=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smmax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def decode_bytes(w) -> int:
    """Algorithmic bytes of one decode launch: Q + gathered K/V (once per kv
    head) + block-table entries read + fp32 output."""
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    total = 0
    for n in w.context_lens.tolist():
        total += hq * d * 2                     # q
        total += n * hkv * d * 2 * 2            # K and V rows
        total += -(-n // 16) * 4                # block-table entries
        total += hq * d * 4                     # fp32 output
    return total


def cache_write_bytes(w) -> int:
    T = w.slot_mapping.shape[0]
    return T * (w.num_kv_heads * w.head_dim * 2 * 2 * 2 + 4)  # read + write of K and V rows, slot ids


_ORACLE_POOLS = {}


def oracle_step_seconds(w, seqs, threads):
    """Run the oracle's whole step (cache_write of the new rows, then
    attention) on the first `seqs` sequences; returns seconds.  The pools are
    copied once, outside the timing (cache_write is idempotent)."""
    import numpy as np
    import oracle
    if id(w) not in _ORACLE_POOLS:
        _ORACLE_POOLS[id(w)] = (w.k_pool.copy(), w.v_pool.copy())
    k, v = _ORACLE_POOLS[id(w)]
    sm = w.slot_mapping.copy()
    sm[seqs:] = -1
    t0 = time.perf_counter()
    oracle.cache_write(k, v, w.k_new, w.v_new, sm)
    qsl = np.arange(seqs + 1, dtype=np.int32)
    oracle.paged_attention(k, v, w.q[:seqs], qsl, w.context_lens[:seqs], w.block_tables[:seqs], w.scale,
                           threads=threads)
    return time.perf_counter() - t0


def cpu_baseline(w, budget_s=12.0):
    """The oracle on the host cores: whole steps repeated for about budget_s."""
    threads = os.cpu_count() or 1
    B = w.num_seqs
    oracle_step_seconds(w, B, threads)  # warm (compiles/loads the oracle)
    reps, spent = 0, 0.0
    while spent < budget_s and reps < 1000:
        spent += oracle_step_seconds(w, B, threads)
        reps += 1
    return {"value": reps * B / spent, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{reps} full steps (cache_write + attention of all {B} sequences), {spent:.1f} s, "
                      f"{threads} threads"}


# ----------------------------------------------------------- reference arm

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import pkv_workloads as W
    w = W.build_config(CONFIG_ID)
    threads = os.cpu_count() or 1
    B = w.num_seqs
    full = oracle_step_seconds(w, B, threads)
    # bounded per-step sample so that warmup + steps take about a minute
    per_step_budget = 60.0 / max(1, args.steps + args.warmup)
    seqs = max(1, min(B, int(B * per_step_budget / max(full, 1e-9))))
    for _ in range(args.warmup):
        oracle_step_seconds(w, seqs, threads)
    t = 0.0
    for _ in range(args.steps):
        t += oracle_step_seconds(w, seqs, threads)
    value = args.steps * seqs / t
    sample = f"first {seqs} of {B} sequences per step (cache_write + attention), {threads} threads"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------- our arm

def run_ours(args):
    import numpy as np
    import torch

    import paged_kv_cache_291_gb300 as pkv
    import pkv_workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    pkv.load()

    # Each rank builds its own batch (weak scaling); seed by rank.
    base = W.build_config(CONFIG_ID)
    w = base if rank == 0 else W.build_config(CONFIG_ID, seed=W.default_seed(CONFIG_ID) + 7919 * rank)
    R = args.replicas

    def td(a):
        x = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            x = x.view(torch.int16).view(torch.bfloat16)
        return x.to(dev)

    reps = []
    for r in range(R):
        reps.append(dict(k=td(w.k_pool), v=td(w.v_pool), q=td(w.q), kn=td(w.k_new), vn=td(w.v_new),
                         slots=td(w.slot_mapping), tables=td(w.block_tables), ctx=td(w.context_lens),
                         out=torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.float32, device=dev)))
    pb = args.partition_blocks
    need = pkv.decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_context_len, pb)
    for r in reps:
        r["ws"] = pkv.new_workspace(need, dev)
    stream = torch.cuda.Stream(device=dev)
    maxctx, scale = w.max_context_len, w.scale

    def step(r):
        pkv.cache_write(r["k"], r["v"], r["kn"], r["vn"], r["slots"], stream=stream)
        pkv.decode_attention(r["k"], r["v"], r["q"], r["tables"], r["ctx"], maxctx, scale, out=r["out"],
                             workspace=r["ws"], partition_blocks=pb, stream=stream)

    def decode_only(r):
        pkv.decode_attention(r["k"], r["v"], r["q"], r["tables"], r["ctx"], maxctx, scale, out=r["out"],
                             workspace=r["ws"], partition_blocks=pb, stream=stream)

    # Graphs: one cycle through the R replicas (2R launches / R launches).
    with torch.cuda.stream(stream):
        for r in reps:  # eager once (also loads kernels)
            step(r)
    stream.synchronize()
    status = pkv.get_error(stream)
    if status[0] != 0:
        raise RuntimeError(f"device error during eager step: {status}")

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in reps:
                fn(r)
        return g

    g_step = capture(step)
    g_dec = capture(decode_only)
    g_single = []
    for r in reps:
        g1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1, stream=stream):
            step(r)
        g_single.append(g1)

    def run_steps(n):
        cycles, rem = divmod(n, R)
        for _ in range(cycles):
            g_step.replay()
        for i in range(rem):
            g_single[i].replay()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # warmup
    with torch.cuda.stream(stream):
        run_steps(max(args.warmup, 3))
    barrier()

    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        run_steps(args.steps)
        e1.record(stream)
    barrier()
    t_wall1 = time.time()
    step_ms = e0.elapsed_time(e1) / args.steps
    step_ms_max = reduce_max(step_ms, dist)

    # The dominant kernel alone: decode launches replayed back to back.
    dec_cycles = max(1, args.steps // R)
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g_dec.replay()
        d0.record(stream)
        for _ in range(dec_cycles):
            g_dec.replay()
        d1.record(stream)
    barrier()
    if clocks:
        clocks.stop()
    dec_ms = d0.elapsed_time(d1) / (dec_cycles * R)
    st = pkv.get_error(stream)
    if st[0] != 0:
        raise RuntimeError(f"device error during timing: {st}")

    # End to end through the public API with pinned host buffers.
    e2e_steps = min(args.steps, args.e2e_steps)
    host_in = dict(q=torch.from_numpy(w.q.view(np.int16)).pin_memory(),
                   kn=torch.from_numpy(w.k_new.view(np.int16)).pin_memory(),
                   vn=torch.from_numpy(w.v_new.view(np.int16)).pin_memory(),
                   slots=torch.from_numpy(w.slot_mapping).pin_memory(),
                   tables=torch.from_numpy(w.block_tables).pin_memory(),
                   ctx=torch.from_numpy(w.context_lens).pin_memory())
    host_out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step(r):
        r["q"].view(torch.int16).copy_(host_in["q"], non_blocking=True)
        r["kn"].view(torch.int16).copy_(host_in["kn"], non_blocking=True)
        r["vn"].view(torch.int16).copy_(host_in["vn"], non_blocking=True)
        r["slots"].copy_(host_in["slots"], non_blocking=True)
        r["tables"].copy_(host_in["tables"], non_blocking=True)
        r["ctx"].copy_(host_in["ctx"], non_blocking=True)
        step(r)
        host_out.copy_(r["out"], non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(reps[i % R])
    barrier()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        x0.record(stream)
        for i in range(e2e_steps):
            e2e_step(reps[i % R])
        x1.record(stream)
    barrier()
    e2e_ms = reduce_max(x0.elapsed_time(x1) / e2e_steps, dist)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    B = w.num_seqs
    peak, peak_kind = measured_peaks()
    dbytes = decode_bytes(w)
    achieved = dbytes / (dec_ms * 1e-3) / 1e9
    traffic = NCU_TRAFFIC["bytes"] if NCU_TRAFFIC["sources_sha"] == sources_sha() else None
    step_bytes = dbytes + cache_write_bytes(w)
    ck = clocks.summary(t_wall0, t_wall1) if clocks else {}
    line = {
        "metric": METRIC,
        "value": world * B / (step_ms_max * 1e-3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": world * B, "seq_len": int(w.context_lens.max()),
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
                   "l2": f"{R} rotated input replicas of {step_bytes / 1e6:.0f} MB each (> 129 MB L2)",
                   "graph": "CUDA graph per cycle of replicas"},
        "step_gbs": step_bytes / (step_ms_max * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": "decode_kernel", "achieved": achieved, "peak": peak,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy)" if peak_kind == "measured"
                     else "fallback", "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes": dbytes, "avg_launch_us": dec_ms * 1e3},
        "gpu_launches": 2 * args.steps,
        "e2e": {"value": world * B / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": e2e_ms},
        "clocks": {"sm_mhz": ck.get("sm_mhz"), "sm_max_mhz": ck.get("sm_max_mhz"), "reasons": ck.get("reasons", []),
                   "samples": ck.get("samples", 0)},
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_budget)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--replicas", type=int, default=8)
    ap.add_argument("--e2e-steps", type=int, default=4000)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--partition-blocks", type=int, default=0, help="0 = automatic split-KV partitioning")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
