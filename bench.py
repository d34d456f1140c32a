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
CONFIG_ID = 2  # the Qwen3-1.7B decode step (34 sequences x 640 tokens)

# DRAM traffic of one decode launch on this workload from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), and the hash of the kernel
# sources it was taken on; reported only while the sources still match.
NCU_TRAFFIC = {"bytes": 91992576, "sources_sha": "ce493bad71d6d71f",
               "capture": "profiles/decode_kernel_qwen3_1p7b_decode.md"}
NCU_TRAFFIC_E4M3 = {"bytes": 44818432, "sources_sha": "ce493bad71d6d71f",
                    "capture": "profiles/decode_kernel_e4m3_qwen3_1p7b_decode.md"}
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


class NvmlClockSampler:
    """SM clock and clock-event reasons polled through NVML (read-only
    queries: nvmlDeviceGetClockInfo, nvmlDeviceGetMaxClockInfo,
    nvmlDeviceGetCurrentClocksEventReasons) every half millisecond while the
    timed region runs, so that even a region of a few milliseconds has
    samples.  The device is matched by PCI bus id.  Falls back to
    nvidia-smi sampling when NVML cannot be loaded."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, device: int):
        import ctypes

        import torch
        self.samples = []
        self._stop = threading.Event()
        self._thr = None
        self.fallback = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            pr = torch.cuda.get_device_properties(device)
            bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(h)) != 0:
                raise OSError("no NVML handle for " + bus.decode())
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self.lib, self.h, self.ct = lib, h, ctypes
            mx = ctypes.c_uint()
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))  # 1 = NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        except (OSError, AttributeError, RuntimeError):
            self.lib = None
            self.fallback = ClockSampler(device)

    def _poll(self):
        ct, lib, h = self.ct, self.lib, self.h
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self._stop.is_set():
            ok = lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk)) == 0 and self.reasons_fn(h, ct.byref(rs)) == 0
            if ok:
                self.samples.append((time.time(), float(clk.value), int(rs.value)))
            time.sleep(0.0005)

    def start(self):
        if self.lib is None:
            self.fallback.start()
            return
        self._thr = threading.Thread(target=self._poll, daemon=True)
        self._thr.start()
        time.sleep(0.01)

    def stop(self):
        if self.lib is None:
            self.fallback.stop()
            return
        self._stop.set()
        self._thr.join(timeout=2)

    def summary(self, t0: float, t1: float):
        if self.lib is None:
            return self.fallback.summary(t0, t1)
        rows = [(mhz, rs) for ts, mhz, rs in self.samples if t0 <= ts <= t1]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        reasons = sorted({name for _, rs in rows for bit, name in self.REASONS.items() if rs & bit})
        return {"sm_mhz": statistics.median(m for m, _ in rows), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense bf16 tensor peak: the measured burst figure (a kernel timed alone)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)"
    return 1900.0, "fallback"


def decode_rows(w):
    """Indices of the sequences that are decode rows (query_len == 1)."""
    import numpy as np
    return np.nonzero(w.query_lens == 1)[0]


def prefill_rows(w):
    import numpy as np
    return np.nonzero(w.query_lens > 1)[0]


def decode_bytes(w, kv_elem_bytes=2) -> int:
    """Algorithmic bytes of one decode launch: Q + gathered K/V (once per kv
    head) + block-table entries read + fp32 output, over the decode rows."""
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    total = 0
    for s in decode_rows(w).tolist():
        n = int(w.context_lens[s])
        total += hq * d * 2                     # q
        total += n * hkv * d * kv_elem_bytes * 2  # K and V rows
        total += -(-n // 16) * 4                # block-table entries
        total += hq * d * 4                     # fp32 output
    return total


def prefill_flops(w) -> int:
    """Algorithmic flops of the prefill rows: causal (query, key) pairs x
    4 d (q.k and p.v, multiply-add = 2) x q heads."""
    total = 0
    for s in prefill_rows(w).tolist():
        n, ql = int(w.context_lens[s]), int(w.query_lens[s])
        total += ql * (n - ql) + ql * (ql + 1) // 2
    return total * 4 * w.head_dim * w.num_q_heads


def cache_write_bytes(w) -> int:
    T = w.slot_mapping.shape[0]
    return T * (w.num_kv_heads * w.head_dim * 2 * 2 * 2 + 4)  # read + write of K and V rows, slot ids


def subset(w, seqs):
    """The same step restricted to the sequences `seqs` (their q rows, tables
    and contexts; the pools are shared)."""
    import numpy as np
    seqs = np.asarray(seqs, dtype=np.int64)
    qsl = w.query_start_loc
    rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in seqs]) if len(seqs) else np.zeros(0, np.int64)
    ql = (qsl[seqs + 1] - qsl[seqs]).astype(np.int32)
    nqsl = np.zeros(len(seqs) + 1, dtype=np.int32)
    nqsl[1:] = np.cumsum(ql)
    return dict(q=np.ascontiguousarray(w.q[rows]), tables=np.ascontiguousarray(w.block_tables[seqs]),
                ctx=np.ascontiguousarray(w.context_lens[seqs]), qsl=nqsl, decode=bool(np.all(ql == 1)),
                max_ctx=int(w.context_lens[seqs].max()) if len(seqs) else 0)


_ORACLE_POOLS = {}


def oracle_step_seconds(w, seqs, threads):
    """Run the oracle's whole step (copy-on-write copies, cache_write of the
    new rows, then attention) on the sequences `seqs`; returns seconds.  The
    pools are copied once, outside the timing (the step is idempotent)."""
    import numpy as np
    import oracle
    if id(w) not in _ORACLE_POOLS:
        _ORACLE_POOLS[id(w)] = (w.k_pool.copy(), w.v_pool.copy())
    k, v = _ORACLE_POOLS[id(w)]
    sub = subset(w, seqs)
    t0 = time.perf_counter()
    if w.copy_src is not None:
        oracle.copy_blocks(k, v, w.copy_src, w.copy_dst)
    oracle.cache_write(k, v, w.k_new, w.v_new, w.slot_mapping)
    oracle.paged_attention(k, v, sub["q"], sub["qsl"], sub["ctx"], sub["tables"], w.scale, threads=threads)
    return time.perf_counter() - t0


def oracle_sample(w, threads, budget_s):
    """Sequences per oracle step so that one step takes about budget_s."""
    B = w.num_seqs
    n = 1
    while True:
        t = oracle_step_seconds(w, list(range(n)), threads)
        if t > 0.2 * budget_s or n >= B:
            break
        n = min(B, n * 4)
    per_seq = t / n
    return max(1, min(B, int(budget_s / max(per_seq, 1e-9))))


def cpu_baseline(w, budget_s=12.0):
    """The oracle on the host cores, repeated steps for about budget_s."""
    threads = os.cpu_count() or 1
    B = w.num_seqs
    n = oracle_sample(w, threads, budget_s / 4)
    seqs = list(range(n))
    reps, spent = 0, 0.0
    while spent < budget_s and reps < 1000:
        spent += oracle_step_seconds(w, seqs, threads)
        reps += 1
    what = "all" if n == B else f"the first {n} of"
    return {"value": reps * n / spent, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{reps} steps over {what} {B} sequences (copy-on-write, cache_write and attention), "
                      f"{spent:.1f} s, {threads} threads"}


def build_workload(config, rank=0, threads=None):
    import pkv_workloads as W
    if rank == 0:
        return W.build_config(config, threads=threads)
    return W.build_config(config, seed=W.default_seed(config) + 7919 * rank, threads=threads)


# ----------------------------------------------------------- reference arm

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = build_workload(args.config)
    threads = os.cpu_count() or 1
    B = w.num_seqs
    per_step_budget = 60.0 / max(1, args.steps + args.warmup)
    n = oracle_sample(w, threads, per_step_budget)
    seqs = list(range(n))
    for _ in range(args.warmup):
        oracle_step_seconds(w, seqs, threads)
    t = 0.0
    for _ in range(args.steps):
        t += oracle_step_seconds(w, seqs, threads)
    value = args.steps * n / t
    sample = f"first {n} of {B} sequences per step (copy-on-write, cache_write and attention), {threads} threads"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------- our arm

def block_manager_timing(w, pkv, torch, dev, stream, iters=200, warm=10):
    """Device time of one pkv_blocks_append for this batch's rows: every row
    first holds its context minus this step's rows, then appends this step's
    rows again and again (the decode loop), replayed from a CUDA graph of
    `iters` appends and timed with events on the launching stream."""
    import numpy as np
    ql = np.diff(w.query_start_loc).astype(np.int64)
    prefix = w.context_lens.astype(np.int64) - ql
    S = w.num_seqs
    final = prefix + ql * (warm + iters)
    MB = int(-(-final.max() // 16)) + 1
    NB = int(np.sum(-(-final // 16))) + S
    blocks = pkv.Blocks(NB, S, MB, device=dev)
    torch.cuda.synchronize(dev)

    def i32(a):
        return torch.tensor(np.asarray(a, dtype=np.int32), device=dev)

    qsl0 = np.concatenate([[0], np.cumsum(prefix)])
    qsl = i32(w.query_start_loc)
    T = int(w.query_start_loc[-1])
    outs = [torch.empty((max(T, 1),), dtype=torch.int32, device=dev)] + \
           [torch.empty((max(S, 1),), dtype=torch.int32, device=dev) for _ in range(2)] + \
           [torch.empty((1,), dtype=torch.int32, device=dev)]
    with torch.cuda.stream(stream):
        blocks.append(i32(qsl0), int(qsl0[-1]), stream=stream)
        for _ in range(warm):
            blocks.append(qsl, T, *outs, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(iters):
            blocks.append(qsl, T, *outs, stream=stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    stream.synchronize()
    status = pkv.get_error(stream)
    if status[0] != 0:
        raise RuntimeError(f"device error in the block-manager timing: {status}")
    expect = int(np.sum(prefix + ql * (warm + iters)))
    if int(blocks.context_lens.sum().item()) != expect:
        raise RuntimeError("the timed appends did not all take effect")
    us = e0.elapsed_time(e1) * 1e3 / iters
    return {"call": "pkv_blocks_append", "workload": f"{S} rows, {T} new tokens per call, "
            f"{int(prefix.sum())} tokens held at the start", "us_per_call": us, "rows_per_s": S / (us * 1e-6),
            "launches_per_call": 1, "bound": "latency (one CTA of 1,024 threads)"}


def prefix_keys_timing(w, pkv, torch, dev, stream, iters=5):
    """Device time of pkv_prefix_keys over every row's whole context (one
    synthetic, seeded token id per cached token), as a prefix cache keys a
    batch of prompts: the SHA-256 chain over the rows' full blocks."""
    import numpy as np
    import pkv_workloads as W
    lens = w.context_lens.astype(np.int64)
    S = len(lens)
    qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    toks = (W.uniform_u64(w.seed, 77, int(qsl[-1])) % 151936).astype(np.int32)  # Qwen3 vocabulary size
    MB = max(1, int(lens.max()) // 16)
    tt = torch.tensor(toks, device=dev)
    qq = torch.tensor(qsl, device=dev)
    keys = torch.zeros((S, MB, 32), dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        pkv.prefix_keys(tt, qq, MB, keys=keys, stream=stream)
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(iters):
            pkv.prefix_keys(tt, qq, MB, keys=keys, stream=stream)
        e1.record(stream)
    stream.synchronize()
    status = pkv.get_error(stream)
    if status[0] != 0:
        raise RuntimeError(f"device error in the prefix-key timing: {status}")
    us = e0.elapsed_time(e1) * 1e3 / iters
    nkeys = int(np.sum(lens // 16))
    return {"call": "pkv_prefix_keys", "workload": f"{S} rows, {int(qsl[-1])} tokens, {nkeys} full blocks, "
            f"longest chain {int(lens.max()) // 16}", "us_per_call": us, "keys_per_s": nkeys / (us * 1e-6),
            "launches_per_call": 1, "bound": "latency (one thread per chain, SHA-256 rounds in sequence)"}


def prefix_cache_timing(w, pkv, torch, dev, stream):
    """Device time of pkv_blocks_register (every row's full blocks, all new
    keys) and of pkv_blocks_match (every row's full prefix cached, the blocks
    free again) for the workload's rows, one call each after a warm-up
    cycle, with keys from pkv_prefix_keys over seeded synthetic token ids."""
    import numpy as np
    import pkv_workloads as W
    lens = w.context_lens.astype(np.int64)
    S = len(lens)
    qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    toks = (W.uniform_u64(w.seed, 77, int(qsl[-1])) % 151936).astype(np.int32)
    MB = int(-(-lens.max() // 16))
    NB = int(np.sum(-(-lens // 16)))
    blocks = pkv.Blocks(NB, S, MB, device=dev, prefix_cache=True)
    keys = pkv.prefix_keys(torch.tensor(toks, device=dev), torch.tensor(qsl, device=dev), MB)
    nk = torch.tensor(lens // 16, dtype=torch.int32, device=dev)
    qsl_d = torch.tensor(qsl, device=dev)
    rows = torch.arange(S, dtype=torch.int32, device=dev)
    times = {}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for it in range(2):
            blocks.reset(stream=stream)
            blocks.append(qsl_d, int(qsl[-1]), stream=stream)
            e0.record(stream)
            blocks.register(keys, nk, stream=stream)
            e1.record(stream)
            stream.synchronize()
            times["register_us"] = e0.elapsed_time(e1) * 1e3
            blocks.release(rows, stream=stream)
            e0.record(stream)
            m = blocks.match(keys, nk, stream=stream)
            e1.record(stream)
            stream.synchronize()
            times["match_us"] = e0.elapsed_time(e1) * 1e3
    status = pkv.get_error(stream)
    if status[0] != 0 or int(m[:S].sum().item()) != int(np.sum(lens // 16)):
        raise RuntimeError(f"prefix-cache timing went wrong: {status}")
    return {"calls": "pkv_blocks_register, pkv_blocks_match",
            "workload": f"{S} rows, {int(np.sum(lens // 16))} full blocks, all new (register) / all hits (match)",
            **times, "launches_per_call": 1,
            "bound": "latency (one CTA per call)"}


def swap_timing(w, pkv, torch, dev, stream, reps):
    """Device time of swapping every block the workload's rows hold out to
    page-locked host memory and back in (pkv_swap_blocks), next to one
    contiguous copy of the same bytes by the copy engines (cudaMemcpyAsync
    through torch), in each direction."""
    import numpy as np
    blocks_np = np.unique(np.concatenate([w.block_tables[s, :-(-int(w.context_lens[s]) // 16)]
                                          for s in range(w.num_seqs)]))
    n = int(min(len(blocks_np), 65535))
    blocks_np = blocks_np[:n].astype(np.int32)
    r = reps[0]
    slab = 2 * w.num_kv_heads * 16 * w.head_dim * 2
    host = torch.empty((n * slab // 2,), dtype=torch.int16).pin_memory()
    dbuf = torch.empty_like(host, device=dev)
    blocks = torch.tensor(blocks_np, device=dev)
    slots = torch.arange(n, dtype=torch.int32, device=dev)
    out = {}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    legs = [("out_gbs", lambda: pkv.swap_out(r["k"], r["v"], blocks, slots, host, stream=stream)),
            ("in_gbs", lambda: pkv.swap_in(r["k"], r["v"], blocks, slots, host, stream=stream)),
            ("memcpy_d2h_gbs", lambda: host.copy_(dbuf, non_blocking=True)),
            ("memcpy_h2d_gbs", lambda: dbuf.copy_(host, non_blocking=True))]
    with torch.cuda.stream(stream):
        for key, fn in legs:
            fn()
            e0.record(stream)
            for _ in range(3):
                fn()
            e1.record(stream)
            stream.synchronize()
            out[key] = 3 * n * slab / (e0.elapsed_time(e1) * 1e-3) / 1e9
    status = pkv.get_error(stream)
    if status[0] != 0:
        raise RuntimeError(f"device error in the swap timing: {status}")
    return {"call": "pkv_swap_blocks", "workload": f"{n} blocks of {slab // 1024} KB ({n * slab / 1e6:.0f} MB) "
            "to and from page-locked host memory", **out, "launches_per_call": 1,
            "bound": "the host link (compared with the copy engines' contiguous copy)"}


def fp8_decode_timing(w, pkv, torch, dev, stream, reps, hbm, bf16_ms, traffic=None):
    """Decode of the same rows over e4m3 pools (one byte per element, one
    scale per pool): the pools are filled from the bf16 ones by the e4m3
    cache write, then the decode launches are replayed from a graph over
    enough pool replicas to exceed L2, like the bf16 timing."""
    import numpy as np
    seqs = decode_rows(w)
    if not len(seqs):
        return None
    sub = subset(w, seqs)
    nb, hkv, _, d = w.k_pool.shape
    pool8 = 2 * w.k_pool.size
    R8 = int(min(256, max(2, -(-512 * 2 ** 20 // pool8))))
    k_scale = v_scale = 1.0 / 64          # N(0, 1) values: +-7 reaches the e4m3 maximum of 448
    slots = torch.arange(nb * 16, dtype=torch.int32, device=dev)

    def td(a):
        x = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            x = x.view(torch.int16).view(torch.bfloat16)
        return x.to(dev)

    items = []
    with torch.cuda.stream(stream):
        for i in range(R8):
            r = reps[i % len(reps)]
            k8 = torch.empty(tuple(w.k_pool.shape), dtype=torch.uint8, device=dev)
            v8 = torch.empty_like(k8)
            rows_k = r["k"].permute(0, 2, 1, 3).reshape(nb * 16, hkv, d).contiguous()
            rows_v = r["v"].permute(0, 2, 1, 3).reshape(nb * 16, hkv, d).contiguous()
            pkv.cache_write(k8, v8, rows_k, rows_v, slots, stream=stream, k_scale=k_scale, v_scale=v_scale)
            n = pkv.decode_workspace_size(len(seqs), w.num_q_heads, hkv, d, sub["max_ctx"])
            items.append(dict(k=k8, v=v8, q=td(sub["q"]), tables=td(sub["tables"]), ctx=td(sub["ctx"]),
                              out=torch.empty((len(seqs), w.num_q_heads, d), dtype=torch.float32, device=dev),
                              ws=pkv.new_workspace(n, dev)))
    stream.synchronize()

    def f(it):
        pkv.decode_attention(it["k"], it["v"], it["q"], it["tables"], it["ctx"], sub["max_ctx"], w.scale,
                             out=it["out"], workspace=it["ws"], stream=stream, k_scale=k_scale, v_scale=v_scale)
    with torch.cuda.stream(stream):
        for it in items:
            f(it)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for it in items:
            f(it)
    cycles = max(3, 4096 // R8)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        for _ in range(cycles):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    st = pkv.get_error(stream)
    if st[0] != 0:
        raise RuntimeError(f"device error in the e4m3 decode timing: {st}")
    ms = e0.elapsed_time(e1) / (cycles * R8)
    nbytes = decode_bytes(w, kv_elem_bytes=1)
    achieved = nbytes / (ms * 1e-3) / 1e9
    out = {"call": "pkv_decode_attention on e4m3 pools", "kernel": "decode_kernel (e4m3)",
           "workload": f"the decode rows of this step, {len(seqs)} sequences, pools written by the e4m3 cache write "
                       f"(k_scale = v_scale = 1/64), {R8} rotated replicas of {pool8 / 1e6:.0f} MB",
           "avg_launch_us": ms * 1e3, "algorithmic_bytes": nbytes, "achieved_gbs": achieved, "peak": hbm,
           "frac": achieved / hbm, "traffic": traffic, "launches_per_call": 1}
    if bf16_ms:
        out["bf16_avg_launch_us"] = bf16_ms * 1e3
        out["speedup_vs_bf16"] = bf16_ms / ms
    return out


def run_ours(args):
    import numpy as np
    import torch

    import paged_kv_cache_291_gb300 as pkv

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

    # Each rank builds its own batch (weak scaling: sequences are independent
    # units, every rank owns its own pool, tables and sequences).
    w = build_workload(args.config, rank)
    pool_bytes = 2 * w.k_pool.nbytes
    R = args.replicas or int(min(256, max(2, -(-512 * 2 ** 20 // pool_bytes))))

    def td(a):
        x = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            x = x.view(torch.int16).view(torch.bfloat16)
        return x.to(dev)

    maxctx, scale = w.max_context_len, w.scale
    Tq = w.num_tokens
    # A step's inputs (everything but the pools) live in one staging buffer
    # per replica, 256-byte aligned views, so that the end-to-end leg moves
    # them from pinned host memory in a single copy.
    step_inputs = [("q", w.q), ("kn", w.k_new), ("vn", w.v_new), ("slots", w.slot_mapping),
                   ("tables", w.block_tables), ("ctx", w.context_lens), ("qsl", w.query_start_loc)]
    if w.copy_src is not None:
        step_inputs += [("src", w.copy_src), ("dst", w.copy_dst)]
    layout, off = {}, 0
    for key, a in step_inputs:
        off = (off + 255) // 256 * 256
        a = np.ascontiguousarray(a)
        layout[key] = (off, a)
        off += a.nbytes
    stage_bytes = (off + 255) // 256 * 256
    stage_np = np.zeros(stage_bytes, dtype=np.uint8)
    for key, (o, a) in layout.items():
        stage_np[o:o + a.nbytes] = a.view(np.uint8).ravel()
    torch_dtype = {np.dtype(np.uint16): torch.int16, np.dtype(np.int32): torch.int32, np.dtype(np.int64): torch.int64}

    def stage_views(stage):
        views = {}
        for key, (o, a) in layout.items():
            t = stage[o:o + a.nbytes].view(torch_dtype[a.dtype])
            if a.dtype == np.uint16:
                t = t.view(torch.bfloat16)
            views[key] = t.view(a.shape)
        return views

    reps = []
    for _ in range(R):
        stage = torch.from_numpy(stage_np).to(dev)
        r = dict(k=td(w.k_pool), v=td(w.v_pool), stage=stage,
                 out=torch.empty((Tq, w.num_q_heads, w.head_dim), dtype=torch.float32, device=dev))
        r.update(stage_views(stage))
        reps.append(r)
    pb = args.partition_blocks
    if w.is_decode:
        need = pkv.decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, maxctx, pb)
    else:
        need = pkv.prefill_workspace_size(w.num_seqs, Tq, w.num_q_heads, w.num_kv_heads, w.head_dim, maxctx)
    for r in reps:
        r["ws"] = pkv.new_workspace(need, dev)
    stream = torch.cuda.Stream(device=dev)
    qsl_host = w.query_start_loc

    def attention(r):
        if w.is_decode:
            pkv.decode_attention(r["k"], r["v"], r["q"], r["tables"], r["ctx"], maxctx, scale, out=r["out"],
                                 workspace=r["ws"], partition_blocks=pb, stream=stream)
        else:
            pkv.chunked_prefill_attention(r["k"], r["v"], r["q"], r["qsl"], r["ctx"], r["tables"], maxctx, scale,
                                          out=r["out"], workspace=r["ws"], query_start_loc_host=qsl_host,
                                          stream=stream)

    def step(r):
        if w.copy_src is not None:
            pkv.copy_blocks(r["k"], r["v"], r["src"], r["dst"], src_host=w.copy_src, dst_host=w.copy_dst,
                            stream=stream)
        pkv.cache_write(r["k"], r["v"], r["kn"], r["vn"], r["slots"], stream=stream)
        attention(r)

    launches_per_step = (1 if w.copy_src is not None else 0) + 1 + (1 if w.is_decode else 0)
    if not w.is_decode:
        launches_per_step += (1 if len(decode_rows(w)) else 0) + (1 if len(prefill_rows(w)) else 0)

    with torch.cuda.stream(stream):
        for r in reps:  # eager once (also loads kernels)
            step(r)
    stream.synchronize()
    status = pkv.get_error(stream)
    if status[0] != 0:
        raise RuntimeError(f"device error during eager step: {status}")

    def capture(fn, items):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for it in items:
                fn(it)
        return g

    g_step = capture(step, reps)
    g_single = [capture(step, [r]) for r in reps]

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

    with torch.cuda.stream(stream):
        run_steps(max(args.warmup, 3))
    barrier()

    clocks = NvmlClockSampler(torch.cuda.current_device()) if rank == 0 else None
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

    # Kernel-alone timings: decode rows and prefill rows as separate batches
    # over the same pools, replayed back to back from graphs.
    def kernel_time(seqs):
        sub = subset(w, seqs)
        items = []
        for r in reps:
            it = dict(k=r["k"], v=r["v"], q=td(sub["q"]), tables=td(sub["tables"]), ctx=td(sub["ctx"]),
                      qsl=td(sub["qsl"]), out=torch.empty((sub["q"].shape[0], w.num_q_heads, w.head_dim),
                                                           dtype=torch.float32, device=dev))
            if sub["decode"]:
                n = pkv.decode_workspace_size(len(seqs), w.num_q_heads, w.num_kv_heads, w.head_dim, sub["max_ctx"], pb)
            else:
                n = pkv.prefill_workspace_size(len(seqs), sub["q"].shape[0], w.num_q_heads, w.num_kv_heads,
                                               w.head_dim, sub["max_ctx"])
            it["ws"] = pkv.new_workspace(n, dev)
            items.append(it)

        def f(it):
            if sub["decode"]:
                pkv.decode_attention(it["k"], it["v"], it["q"], it["tables"], it["ctx"], sub["max_ctx"], scale,
                                     out=it["out"], workspace=it["ws"], partition_blocks=pb, stream=stream)
            else:
                pkv.chunked_prefill_attention(it["k"], it["v"], it["q"], it["qsl"], it["ctx"], it["tables"],
                                              sub["max_ctx"], scale, out=it["out"], workspace=it["ws"],
                                              query_start_loc_host=sub["qsl"], stream=stream)
        with torch.cuda.stream(stream):
            for it in items:
                f(it)
        stream.synchronize()
        g = capture(f, items)
        cycles = max(1, min(args.steps // R, 2000))
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            d0.record(stream)
            for _ in range(cycles):
                g.replay()
            d1.record(stream)
        barrier()
        return d0.elapsed_time(d1) / (cycles * R)

    dec_ms = kernel_time(decode_rows(w)) if len(decode_rows(w)) else None
    pre_ms = kernel_time(prefill_rows(w)) if len(prefill_rows(w)) else None
    if clocks:
        clocks.stop()
    st = pkv.get_error(stream)
    if st[0] != 0:
        raise RuntimeError(f"device error during timing: {st}")

    # End to end through the public API with pinned host buffers: every step
    # copies all its inputs (one staging buffer, one copy) to the device,
    # runs the calls and reads the output back.
    e2e_steps = min(args.steps, args.e2e_steps)
    host_stage = torch.from_numpy(stage_np).pin_memory()
    host_out = torch.empty((Tq, w.num_q_heads, w.head_dim), dtype=torch.float32).pin_memory()
    h2d = host_stage.numel()
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step(r):
        r["stage"].copy_(host_stage, non_blocking=True)
        step(r)
        host_out.copy_(r["out"], non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(reps[i % R])
    stream.synchronize()
    # As a serving loop does, the step (its input copy from pinned memory,
    # the calls, the output copy back) is captured through the same public
    # calls in CUDA graphs and replayed: one graph per cycle over the
    # replicas, as for the device-timed steps, and one per replica for the
    # remainder.
    g_e2e_cycle = capture(e2e_step, reps)
    g_e2e = [capture(e2e_step, [r]) for r in reps]

    def run_e2e(n):
        cycles, rem = divmod(n, R)
        for _ in range(cycles):
            g_e2e_cycle.replay()
        for i in range(rem):
            g_e2e[i].replay()

    with torch.cuda.stream(stream):
        run_e2e(min(3, e2e_steps))
    barrier()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        x0.record(stream)
        run_e2e(e2e_steps)
        x1.record(stream)
    barrier()
    e2e_ms = reduce_max(x0.elapsed_time(x1) / e2e_steps, dist)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    B = w.num_seqs
    hbm, hbm_kind = measured_peaks()
    tflops_peak, tf_kind = measured_tensor_peak()
    dbytes = decode_bytes(w)
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
        "config": {"workload": w.name, "global_batch": world * B, "seq_len": int(w.context_lens.max()),
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
                   "l2": f"{R} rotated input replicas of {pool_bytes / 1e6:.0f} MB pools (> 129 MB L2 in total)",
                   "graph": "CUDA graph per cycle of replicas"},
        "gpu_launches": launches_per_step * args.steps,
        # query rows (decode rows and prefill tokens) per second over the whole step
        "tokens_per_s": world * Tq / (step_ms_max * 1e-3),
        "e2e": {"value": world * B / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": e2e_ms},
    }
    decode_roof = None
    if dec_ms is not None:
        achieved = dbytes / (dec_ms * 1e-3) / 1e9
        traffic = (NCU_TRAFFIC["bytes"] if NCU_TRAFFIC["sources_sha"] == sources_sha() and args.config == CONFIG_ID
                   else None)
        decode_roof = {"bound": "hbm", "kernel": "decode_kernel", "achieved": achieved, "peak": hbm,
                       "peak_kind": f"{hbm_kind} (MEASURED_PEAKS.json hbm_gbs, copy)" if hbm_kind == "measured"
                       else "fallback", "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                       "algorithmic_bytes": dbytes, "avg_launch_us": dec_ms * 1e3}
    prefill_roof = None
    if pre_ms is not None:
        fl = prefill_flops(w)
        achieved = fl / (pre_ms * 1e-3) / 1e12
        prefill_roof = {"bound": "tensor", "kernel": "prefill_kernel", "achieved": achieved, "peak": tflops_peak,
                        "peak_kind": tf_kind, "unit": "TFLOP/s", "frac": achieved / tflops_peak, "traffic": None,
                        "algorithmic_flops": fl, "avg_launch_us": pre_ms * 1e3}
    if prefill_roof is not None and (decode_roof is None or pre_ms > dec_ms):
        line["roofline"] = prefill_roof
        if decode_roof is not None:
            line["decode_roofline"] = decode_roof
    else:
        line["roofline"] = decode_roof
        if prefill_roof is not None:
            line["prefill_roofline"] = prefill_roof
    ck = clocks.summary(t_wall0, t_wall1) if clocks else {}
    line["clocks"] = {"sm_mhz": ck.get("sm_mhz"), "sm_max_mhz": ck.get("sm_max_mhz"),
                      "reasons": ck.get("reasons", []), "samples": ck.get("samples", 0)}
    line["block_manager"] = block_manager_timing(w, pkv, torch, dev, stream)
    line["prefix_keys"] = prefix_keys_timing(w, pkv, torch, dev, stream)
    line["prefix_cache"] = prefix_cache_timing(w, pkv, torch, dev, stream)
    line["swap"] = swap_timing(w, pkv, torch, dev, stream, reps)
    line["fp8_decode"] = fp8_decode_timing(
        w, pkv, torch, dev, stream, reps, hbm, dec_ms,
        traffic=(NCU_TRAFFIC_E4M3["bytes"] if NCU_TRAFFIC_E4M3["sources_sha"] == sources_sha()
                 and args.config == CONFIG_ID else None))
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
    ap.add_argument("--replicas", type=int, default=0, help="0 = enough pool replicas to exceed 512 MB")
    ap.add_argument("--config", type=int, default=CONFIG_ID, choices=[1, 2, 3, 4, 5],
                    help="workload (default: the Qwen3-1.7B decode step the metric is quoted on)")
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
