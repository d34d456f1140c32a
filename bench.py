#!/usr/bin/env python3
"""Benchmark of the paged-KV hot path on GB300.

Headline: one step = the whole hot path for one decode iteration of the
Qwen3-1.7B attention shape (one layer): the store of the 34 sequences' new
K/V rows and paged decode attention of 34 sequences x 640 tokens (16 q / 8 kv
heads, head_dim 128, 16-token blocks, 22,048-token pool, shuffled block
tables).  Synthetic bf16 N(0,1) data from pkv_workloads (no weights, no
dataset).  `--config k` picks another workload for the headline.

Beside the headline, the `configs` object reports every workload (1..5) the
same way: the step rate, the decode kernel (and, for the mixed batch, the
tensor-core prefill kernel) timed alone against its roofline, the e4m3 decode
on the same rows, and the CPU oracle on the host cores (all of them and one
thread) on a bounded sample.

Timing: inputs resident in HBM; enough replicas of the pool, tables and q
(more than 512 MB in all, larger than the 129 MB L2) are rotated step by
step, so every step reads its K/V from HBM.  Steps are replayed from CUDA
graphs (one graph per cycle through the replicas) and timed with CUDA events
on the launching stream, synchronised on both sides.  Kernel-alone figures
are graph replays of that kernel over the replicas: the mean over all
launches, and the median and minimum of several trials; "warm" repeats one
replica, so its inputs stay in L2 where they fit.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on
the host cores instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
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
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal (the measured copy bandwidth is the roofline)
L2_ROTATE_BYTES = 512 << 20

# DRAM traffic of one launch of a kernel on a workload from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), with the hash of the
# kernel's sources it was taken on; reported only while they still match.
# Keys: (kernel entry, config).
NCU_TRAFFIC = {
    ("decode_step", 1): {"bytes": 1511680, "sources": "decode", "sources_sha": "9924469a8935d603"},
    ("decode_step", 2): {"bytes": 91181824, "sources": "decode", "sources_sha": "9924469a8935d603"},
    ("decode_step", 3): {"bytes": 4063371264, "sources": "decode", "sources_sha": "9924469a8935d603"},
    ("decode", 1): {"bytes": 1498880, "sources": "decode", "sources_sha": "9924469a8935d603"},
    ("decode", 2): {"bytes": 91179008, "sources": "decode", "sources_sha": "9924469a8935d603"},
    ("decode", 3): {"bytes": 4073321216, "sources": "decode", "sources_sha": "9924469a8935d603"},
    ("decode", 4): {"bytes": 18811392, "sources": "decode", "sources_sha": "9924469a8935d603"},
    ("decode", 5): {"bytes": 306025728, "sources": "decode", "sources_sha": "9924469a8935d603"},
    ("fp8_decode", 1): {"bytes": 814336, "sources": "decode", "sources_sha": "9924469a8935d603"},
    ("fp8_decode", 2): {"bytes": 44804608, "sources": "decode", "sources_sha": "9924469a8935d603"},
    ("fp8_decode", 3): {"bytes": 2038387456, "sources": "decode", "sources_sha": "9924469a8935d603"},
    ("fp8_decode", 4): {"bytes": 9532416, "sources": "decode", "sources_sha": "9924469a8935d603"},
    ("fp8_decode", 5): {"bytes": 154604544, "sources": "decode", "sources_sha": "9924469a8935d603"},
    # both kernels of the shared-prefix decode (shared_prefix_kernel, then decode_kernel)
    ("shared_prefix", 4): {"bytes": 19253248, "sources": "decode", "sources_sha": "9924469a8935d603"},
    # prefill tiles of the mixed batch (the K and V tiles are read by every row-tile CTA of a kv head)
    ("prefill", 5): {"bytes": 25325824, "sources": "prefill", "sources_sha": "334b56d190920b05"},
}
KERNEL_SOURCES = {
    "decode": ["paged_kv_cache_291_gb300/csrc/decode_kernel.cuh", "paged_kv_cache_291_gb300/csrc/decode.cu",
               "paged_kv_cache_291_gb300/csrc/decode_fused.cu", "paged_kv_cache_291_gb300/csrc/pkv_device.cuh",
               "paged_kv_cache_291_gb300/csrc/shared_prefix.cu"],
    "prefill": ["paged_kv_cache_291_gb300/csrc/prefill.cu", "paged_kv_cache_291_gb300/csrc/tcgen05.cuh",
                "paged_kv_cache_291_gb300/csrc/pkv_device.cuh"],
}


def sources_sha(group: str = "decode") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[group]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, config):
    rec = NCU_TRAFFIC.get((kernel, config))
    return rec["bytes"] if rec is not None and rec["sources_sha"] == sources_sha(rec["sources"]) else None


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


def _nvml_poll(bus, conn, dense, paused, stop):
    """Child process: poll the SM clock and the clock-event reasons of the
    GPU at PCI bus id `bus` through read-only NVML queries, every half
    millisecond (back to back while `dense` is set), until `stop`; then send
    the (time, MHz, reasons) samples back.  A process of its own, so that
    polling never competes with the benchmark's launches for the GIL."""
    import ctypes
    out = []
    try:
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        mx = ctypes.c_uint()
        lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))  # 1 = NVML_CLOCK_SM
        conn.send(("max", float(mx.value)))
        while not stop.is_set():
            if paused.is_set():
                time.sleep(0.01)
                continue
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and fn(h, ctypes.byref(rs)) == 0:
                out.append((time.time(), float(clk.value), int(rs.value)))
            if not dense.is_set():
                time.sleep(0.0005)
    except (OSError, AttributeError) as e:
        conn.send(("error", str(e)))
    conn.send(("samples", out))
    conn.close()


class NvmlClockSampler:
    """SM clock and clock-event reasons polled through NVML (read-only
    queries: nvmlDeviceGetClockInfo, nvmlDeviceGetMaxClockInfo,
    nvmlDeviceGetCurrentClocksEventReasons) in a child process, every half
    millisecond, back to back during the headline's timed region, so that
    even a region of a few hundred microseconds has samples.  The device is
    matched by PCI bus id.  Falls back to nvidia-smi sampling when NVML
    cannot be used."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, device: int):
        import multiprocessing as mp

        import torch
        self.samples = []
        self.max_mhz = None
        self.fallback = None
        pr = torch.cuda.get_device_properties(device)
        bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
        ctx = mp.get_context("spawn")  # CUDA is initialised in this process: never fork it
        self._dense, self._paused, self._stop = ctx.Event(), ctx.Event(), ctx.Event()
        self._conn, child = ctx.Pipe(duplex=False)
        self._proc = ctx.Process(target=_nvml_poll, args=(bus, child, self._dense, self._paused, self._stop),
                                 daemon=True)
        self.gpu_index = device

    def start(self):
        try:
            self._proc.start()
            if self._conn.poll(30):
                kind, val = self._conn.recv()
                if kind == "max":
                    self.max_mhz = val
                    return
        except (EOFError, OSError):
            pass
        self._stop.set()
        self._proc.join(timeout=5)
        self.fallback = ClockSampler(self.gpu_index)
        self.fallback.start()

    def dense(self, on: bool):
        """Poll back to back (on=True), for a timed region of a few hundred
        microseconds."""
        (self._dense.set if on else self._dense.clear)()
        time.sleep(0.002)

    def pause(self, on: bool):
        """Stop polling (on=True) while the host cores run something timed."""
        (self._paused.set if on else self._paused.clear)()

    def stop(self):
        if self.fallback is not None:
            self.fallback.stop()
            return
        self._stop.set()
        try:
            while self._conn.poll(30):
                kind, val = self._conn.recv()
                if kind == "samples":
                    self.samples = val
                    break
        except (EOFError, OSError):
            pass
        self._proc.join(timeout=10)

    def summary(self, t0: float, t1: float):
        if self.fallback is not None:
            return self.fallback.summary(t0, t1)
        rows = [(mhz, rs) for ts, mhz, rs in self.samples if t0 <= ts <= t1]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        reasons = sorted({name for _, rs in rows for bit, name in self.REASONS.items() if rs & bit})
        return {"sm_mhz": statistics.median(m for m, _ in rows), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------- peaks, bytes, flops

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


def decode_bytes(w, kv_elem_bytes=2, seqs=None) -> int:
    """Algorithmic bytes of one decode launch: Q + gathered K/V (once per kv
    head) + block-table entries read + fp32 output, over the decode rows (or
    the sequences `seqs`)."""
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    total = 0
    for s in (decode_rows(w) if seqs is None else seqs):
        n = int(w.context_lens[int(s)])
        total += hq * d * 2                     # q
        total += n * hkv * d * kv_elem_bytes * 2  # K and V rows
        total += -(-n // 16) * 4                # block-table entries
        total += hq * d * 4                     # fp32 output
    return total


def decode_unique_bytes(w, kv_elem_bytes=2) -> int:
    """The same launch with every distinct (physical block, kv head) slab
    counted once: what HBM must deliver when blocks shared by several
    sequences come from L2 after their first read (rows of the last,
    partly filled block counted up to the longest context that uses it)."""
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    rows = {}
    for s in decode_rows(w).tolist():
        n = int(w.context_lens[s])
        nb = -(-n // 16)
        for b in range(nb):
            phys = int(w.block_tables[s, b])
            rows[phys] = max(rows.get(phys, 0), min(16, n - 16 * b))
    kv = sum(rows.values()) * hkv * d * kv_elem_bytes * 2
    other = sum(hq * d * 2 + -(-int(w.context_lens[s]) // 16) * 4 + hq * d * 4 for s in decode_rows(w).tolist())
    return int(kv + other)


def prefill_flops(w) -> int:
    """Algorithmic flops of the prefill rows: causal (query, key) pairs x
    4 d (q.k and p.v, multiply-add = 2) x q heads."""
    total = 0
    for s in prefill_rows(w).tolist():
        n, ql = int(w.context_lens[s]), int(w.query_lens[s])
        total += ql * (n - ql) + ql * (ql + 1) // 2
    return total * 4 * w.head_dim * w.num_q_heads


def step_bytes(w) -> int:
    """Algorithmic bytes of a whole step: copy-on-write copies (read and
    write of whole blocks), the new rows' store (read and write), and the
    attention's Q, gathered K/V, table entries and output (prefill rows:
    their Q, the K/V of their keys once per kv head and their output)."""
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    total = decode_bytes(w)
    for s in prefill_rows(w).tolist():
        n, ql = int(w.context_lens[s]), int(w.query_lens[s])
        total += ql * hq * d * (2 + 4) + n * hkv * d * 2 * 2 + -(-n // 16) * 4
    T = w.slot_mapping.shape[0]
    total += T * (hkv * d * 2 * 2 * 2 + 4)
    if w.copy_src is not None:
        total += len(w.copy_src) * 2 * (2 * hkv * 16 * d * 2) + 8 * len(w.copy_src)
    return total


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


# ----------------------------------------------------------- the oracle on the host cores

def host_threads():
    """(threads the process may run on, CPUs in the machine)."""
    try:
        aff = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        aff = os.cpu_count() or 1
    return max(1, aff), os.cpu_count() or 1


_ORACLE_POOLS = {}


def oracle_step_seconds(w, seqs, threads):
    """Run the oracle's whole step (copy-on-write copies, the store of the new
    rows, then attention) with attention over the sequences `seqs`; returns
    seconds.  The pools are copied once, outside the timing (the step is
    idempotent)."""
    import oracle
    if _ORACLE_POOLS.get("w") is not w:  # the workload itself is kept, so a new one never matches
        _ORACLE_POOLS.clear()
        _ORACLE_POOLS.update(w=w, kv=(w.k_pool.copy(), w.v_pool.copy()))
    k, v = _ORACLE_POOLS["kv"]
    sub = subset(w, seqs)
    t0 = time.perf_counter()
    if w.copy_src is not None:
        oracle.copy_blocks(k, v, w.copy_src, w.copy_dst)
    oracle.cache_write(k, v, w.k_new, w.v_new, w.slot_mapping)
    oracle.paged_attention(k, v, sub["q"], sub["qsl"], sub["ctx"], sub["tables"], w.scale, threads=threads)
    return time.perf_counter() - t0


def spread(B, n):
    """n sequence indices spread evenly over 0..B-1 (first and last included)."""
    import numpy as np
    if n >= B:
        return list(range(B))
    return sorted(set(np.linspace(0, B - 1, n).round().astype(int).tolist()))


def seq_cost(w, s):
    """Relative oracle work of sequence s: the (query row, key) pairs of
    every q head (a dot product and a V update each) plus the gather of the
    context's K and V rows of every kv head."""
    n, ql = int(w.context_lens[s]), int(w.query_lens[s])
    pairs = ql * (n - ql) + ql * (ql + 1) // 2
    return max(1, (pairs * w.num_q_heads + n * w.num_kv_heads) * 2 * w.head_dim)


def predicted_cost(w, seqs, threads):
    """The oracle deals the sequences of a call to its threads round-robin:
    the step takes as long as the thread with the most work."""
    per = [0] * max(1, threads)
    for i, s in enumerate(seqs):
        per[i % len(per)] += seq_cost(w, s)
    return max(per)


def oracle_sample(w, threads, budget_s):
    """Sequences (spread over the batch) for an oracle step of about
    budget_s on `threads` threads: the oracle's rate is measured on the
    cheapest sequences, then the largest spread sample whose predicted time
    fits the budget is taken."""
    B = w.num_seqs
    order = sorted(range(B), key=lambda s: seq_cost(w, s))
    fixed = min(oracle_step_seconds(w, [], threads) for _ in range(3))  # the copies and the row store
    k = 1
    while True:
        cal = sorted(order[:k])
        t = oracle_step_seconds(w, cal, threads) - fixed
        if t > 0.05 or k >= B:
            break
        k = min(B, 2 * k)
    rate = predicted_cost(w, cal, threads) / max(t, 1e-6)
    best = [order[0]]
    for n in range(1, B + 1):
        seqs = spread(B, n)
        if fixed + predicted_cost(w, seqs, threads) / rate <= budget_s:
            best = seqs
    return best


def oracle_rate(w, seqs, threads, min_s=1.0, min_reps=3):
    """Median and minimum seconds of repeated oracle steps over `seqs`."""
    times = []
    while len(times) < min_reps or sum(times) < min_s:
        times.append(oracle_step_seconds(w, seqs, threads))
        if len(times) >= 50:
            break
    return statistics.median(times), min(times), len(times)


def oracle_leg(w, threads, budget_s, min_reps):
    """The oracle's step over a sample of sequences sized for about budget_s
    on `threads` threads: sequences, query rows and decode K/V bytes per
    second from the median of repeated steps."""
    seqs = oracle_sample(w, threads, budget_s)
    med, mn, reps = oracle_rate(w, seqs, threads, min_s=budget_s, min_reps=min_reps)
    rows = int(sum(int(w.query_lens[s]) for s in seqs))
    dec = [s for s in seqs if int(w.query_lens[s]) == 1]
    nbytes = decode_bytes(w, seqs=dec)
    B = w.num_seqs
    what = "all" if len(seqs) == B else f"{len(seqs)} (spread over the batch) of"
    return {"value": len(seqs) / med, "unit": UNIT, "cores": threads, "median_s": med, "min_s": mn, "reps": reps,
            "tokens_per_s": rows / med, "decode_gbs": nbytes / med / 1e9 if nbytes else None,
            "sample": f"copy-on-write, the store of the new rows and attention over {what} {B} sequences "
                      f"({rows} query rows) per step, {threads} thread{'s' if threads > 1 else ''}"}


def cpu_baseline(w, budget_s=3.0, one_thread=True):
    """The oracle as it stands (threaded over sequences), on all the host
    cores the process may use and on one thread, each over a bounded sample
    of sequences spread over the batch and sized for about budget_s, each
    the median of repeated steps."""
    threads, ncpu = host_threads()
    out = {"kind": "oracle", "cpus": ncpu, "affinity_cpus": threads}
    out.update(oracle_leg(w, threads, budget_s, 3))
    if one_thread:
        out["one_thread"] = oracle_leg(w, 1, budget_s, 1)
    return out


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
    threads, _ = host_threads()
    B = w.num_seqs
    per_step_budget = 60.0 / max(1, args.steps + args.warmup)
    seqs = oracle_sample(w, threads, per_step_budget)
    for _ in range(args.warmup):
        oracle_step_seconds(w, seqs, threads)
    t = 0.0
    for _ in range(args.steps):
        t += oracle_step_seconds(w, seqs, threads)
    n = len(seqs)
    value = args.steps * n / t
    what = "all" if n == B else f"{n} (spread over the batch) of"
    sample = (f"{what} {B} sequences per step (copy-on-write, the store of the new rows and attention), "
              f"{threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------- one workload on the device

class ConfigRun:
    """One workload on the device: R rotated replicas of its inputs (more
    than 512 MB in all), the step through the public calls (copy-on-write if
    the workload has it, the store of the new rows, attention), and CUDA
    graphs over the replicas."""

    def __init__(self, config, w, pkv, torch, dev, stream, replicas=0, partition_blocks=0):
        import numpy as np
        self.config, self.w, self.pkv, self.torch, self.dev, self.stream = config, w, pkv, torch, dev, stream
        self.pb = partition_blocks
        pool_bytes = 2 * w.k_pool.nbytes
        self.pool_bytes = pool_bytes
        self.R = R = replicas or int(min(256, max(2, -(-L2_ROTATE_BYTES // pool_bytes))))
        self.maxctx, self.scale, self.Tq = w.max_context_len, w.scale, w.num_tokens
        # A step's inputs (everything but the pools) live in one staging
        # buffer per replica, 256-byte aligned views, so that the end-to-end
        # leg moves them from pinned host memory in a single copy.
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
        self.stage_np = stage_np = np.zeros(stage_bytes, dtype=np.uint8)
        for key, (o, a) in layout.items():
            stage_np[o:o + a.nbytes] = a.view(np.uint8).ravel()
        tdt = {np.dtype(np.uint16): torch.int16, np.dtype(np.int32): torch.int32, np.dtype(np.int64): torch.int64}

        def stage_views(stage):
            views = {}
            for key, (o, a) in layout.items():
                t = stage[o:o + a.nbytes].view(tdt[a.dtype])
                if a.dtype == np.uint16:
                    t = t.view(torch.bfloat16)
                views[key] = t.view(a.shape)
            return views

        k0, v0 = self.td(w.k_pool), self.td(w.v_pool)
        self.reps = []
        for i in range(R):
            stage = torch.from_numpy(stage_np).to(dev)
            r = dict(k=k0 if i == 0 else k0.clone(), v=v0 if i == 0 else v0.clone(), stage=stage,
                     out=torch.empty((self.Tq, w.num_q_heads, w.head_dim), dtype=torch.float32, device=dev))
            r.update(stage_views(stage))
            self.reps.append(r)
        # Sequences whose tables all start with the same full blocks (a shared
        # prefix): decode reads those once per kv head for all of them.
        self.shared_blocks = 0
        if w.is_decode and w.num_seqs > 1 and self.pb == 0:
            self.shared_blocks = pkv.common_prefix_blocks(w.block_tables, w.context_lens)
        if self.shared_blocks > 0:
            need = pkv.decode_shared_prefix_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                                           self.maxctx, self.shared_blocks)
        elif w.is_decode:
            need = pkv.decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, self.maxctx,
                                             self.pb)
        else:
            need = pkv.prefill_workspace_size(w.num_seqs, self.Tq, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                              self.maxctx)
        for r in self.reps:
            r["ws"] = pkv.new_workspace(need, dev)
        # One new row per sequence at its last position (a plain decode step):
        # the store and the attention run as one launch (pkv_decode_step).
        self.fused = bool(w.is_decode and w.copy_src is None and w.slot_mapping.shape[0] == w.num_seqs)
        if self.fused:
            self.launches_per_step = 1
        else:
            self.launches_per_step = ((1 if w.copy_src is not None else 0) + 1 + (1 if w.is_decode else 0) +
                                      (1 if self.shared_blocks > 0 else 0))
            if not w.is_decode:
                self.launches_per_step += (1 if len(decode_rows(w)) else 0) + (1 if len(prefill_rows(w)) else 0)
        with torch.cuda.stream(stream):
            for r in self.reps:  # eager once (also loads kernels)
                self.step(r)
        stream.synchronize()
        self.check("eager step")
        self.g_step = self.capture(self.step, self.reps)
        self.g_single = [self.capture(self.step, [r]) for r in self.reps]

    def td(self, a):
        import numpy as np
        torch = self.torch
        x = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            x = x.view(torch.int16).view(torch.bfloat16)
        return x.to(self.dev)

    def check(self, what):
        st = self.pkv.get_error(self.stream)
        if st[0] != 0:
            raise RuntimeError(f"device error during {what} ({self.w.name}): {st}")

    def attention(self, r):
        w, pkv, s = self.w, self.pkv, self.stream
        if self.shared_blocks > 0:
            pkv.decode_attention_shared_prefix(r["k"], r["v"], r["q"], r["tables"], r["ctx"], self.maxctx,
                                               self.shared_blocks, self.scale, out=r["out"], workspace=r["ws"],
                                               stream=s)
        elif w.is_decode:
            pkv.decode_attention(r["k"], r["v"], r["q"], r["tables"], r["ctx"], self.maxctx, self.scale,
                                 out=r["out"], workspace=r["ws"], partition_blocks=self.pb, stream=s)
        else:
            pkv.chunked_prefill_attention(r["k"], r["v"], r["q"], r["qsl"], r["ctx"], r["tables"], self.maxctx,
                                          self.scale, out=r["out"], workspace=r["ws"],
                                          query_start_loc_host=w.query_start_loc, stream=s)

    def step(self, r):
        w, pkv, s = self.w, self.pkv, self.stream
        if self.fused:
            pkv.decode_step(r["k"], r["v"], r["kn"], r["vn"], r["slots"], r["q"], r["tables"], r["ctx"], self.maxctx,
                            self.scale, out=r["out"], workspace=r["ws"], partition_blocks=self.pb, stream=s)
            return
        if w.copy_src is not None:
            pkv.copy_blocks(r["k"], r["v"], r["src"], r["dst"], src_host=w.copy_src, dst_host=w.copy_dst, stream=s)
        pkv.cache_write(r["k"], r["v"], r["kn"], r["vn"], r["slots"], stream=s)
        self.attention(r)

    def capture(self, fn, items):
        g = self.torch.cuda.CUDAGraph()
        with self.torch.cuda.graph(g, stream=self.stream):
            for it in items:
                fn(it)
        return g

    def run_steps(self, n):
        cycles, rem = divmod(n, self.R)
        for _ in range(cycles):
            self.g_step.replay()
        for i in range(rem):
            self.g_single[i].replay()

    def timed(self, fn, sync):
        """Device milliseconds of fn() between events on the stream."""
        torch = self.torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sync()
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            fn()
            e1.record(self.stream)
        sync()
        return e0.elapsed_time(e1)

    def sync(self):
        self.torch.cuda.synchronize(self.dev)

    def step_trials(self, min_steps=200, min_ms=20.0, trials=5):
        """Steps timed in `trials` trials of equal length (whole cycles)."""
        with self.torch.cuda.stream(self.stream):
            self.run_steps(2 * self.R)
        self.sync()
        per = self.timed(lambda: self.run_steps(self.R), self.sync) / self.R
        n = max(min_steps, int(min_ms / max(per, 1e-6)))
        cyc = max(1, -(-n // (self.R * trials)))
        ms = [self.timed(lambda: self.run_steps(cyc * self.R), self.sync) / (cyc * self.R) for _ in range(trials)]
        self.check("timed steps")
        total = cyc * self.R * trials
        return {"mean_ms": statistics.fmean(ms), "median_ms": statistics.median(ms), "min_ms": min(ms),
                "steps": total, "trials": trials}

    def kernel_alone(self, seqs, kv_e4m3=False, fused=False, shared=0, min_launches=200, min_ms=20.0, trials=5,
                     warm_launches=50):
        """One attention launch over the sequences `seqs` (decode rows or
        prefill rows; fused: the whole decode step, the new rows' store
        included; shared > 0: the shared-prefix decode over that many shared
        blocks, its two launches), replayed from graphs over the replicas
        (bf16 pools) or over e4m3 copies of them (kv_e4m3, pools written by
        the e4m3 store); mean over all launches, median and minimum of the
        trials, and a warm figure repeating one replica."""
        import numpy as np
        torch, pkv, w, dev = self.torch, self.pkv, self.w, self.dev
        sub = subset(w, seqs)
        nb, hkv, _, d = w.k_pool.shape
        ks = vs = None
        if kv_e4m3:
            ks = vs = 1.0 / 64  # N(0, 1) values: +-7 reaches the e4m3 maximum of 448
            pool8 = 2 * w.k_pool.size
            R = int(min(256, max(2, -(-L2_ROTATE_BYTES // pool8))))
            slots = torch.arange(nb * 16, dtype=torch.int32, device=dev)
        else:
            R = self.R
        items = []
        with torch.cuda.stream(self.stream):
            for i in range(R):
                r = self.reps[i % self.R]
                if kv_e4m3:
                    k = torch.empty(tuple(w.k_pool.shape), dtype=torch.uint8, device=dev)
                    v = torch.empty_like(k)
                    rk = r["k"].permute(0, 2, 1, 3).reshape(nb * 16, hkv, d).contiguous()
                    rv = r["v"].permute(0, 2, 1, 3).reshape(nb * 16, hkv, d).contiguous()
                    pkv.cache_write(k, v, rk, rv, slots, stream=self.stream, k_scale=ks, v_scale=vs)
                    del rk, rv
                else:
                    k, v = r["k"], r["v"]
                it = dict(k=k, v=v, q=self.td(sub["q"]), tables=self.td(sub["tables"]), ctx=self.td(sub["ctx"]),
                          qsl=self.td(sub["qsl"]), out=torch.empty((sub["q"].shape[0], w.num_q_heads, d),
                                                                   dtype=torch.float32, device=dev))
                if fused:
                    it.update(kn=r["kn"], vn=r["vn"], slots=r["slots"])
                if shared > 0:
                    n = pkv.decode_shared_prefix_workspace_size(len(seqs), w.num_q_heads, hkv, d, sub["max_ctx"],
                                                                shared)
                elif sub["decode"]:
                    n = pkv.decode_workspace_size(len(seqs), w.num_q_heads, hkv, d, sub["max_ctx"], self.pb)
                else:
                    n = pkv.prefill_workspace_size(len(seqs), sub["q"].shape[0], w.num_q_heads, hkv, d,
                                                   sub["max_ctx"])
                it["ws"] = pkv.new_workspace(n, dev)
                items.append(it)
        self.stream.synchronize()

        def f(it):
            if fused:
                pkv.decode_step(it["k"], it["v"], it["kn"], it["vn"], it["slots"], it["q"], it["tables"], it["ctx"],
                                sub["max_ctx"], self.scale, out=it["out"], workspace=it["ws"],
                                partition_blocks=self.pb, stream=self.stream, k_scale=ks, v_scale=vs)
            elif shared > 0:
                pkv.decode_attention_shared_prefix(it["k"], it["v"], it["q"], it["tables"], it["ctx"], sub["max_ctx"],
                                                   shared, self.scale, out=it["out"], workspace=it["ws"],
                                                   stream=self.stream)
            elif sub["decode"]:
                pkv.decode_attention(it["k"], it["v"], it["q"], it["tables"], it["ctx"], sub["max_ctx"], self.scale,
                                     out=it["out"], workspace=it["ws"], partition_blocks=self.pb, stream=self.stream,
                                     k_scale=ks, v_scale=vs)
            else:
                pkv.chunked_prefill_attention(it["k"], it["v"], it["q"], it["qsl"], it["ctx"], it["tables"],
                                              sub["max_ctx"], self.scale, out=it["out"], workspace=it["ws"],
                                              query_start_loc_host=sub["qsl"], stream=self.stream)
        with torch.cuda.stream(self.stream):
            for it in items:
                f(it)
        self.stream.synchronize()
        g = self.capture(f, items)
        g_warm = self.capture(f, [items[0]] * warm_launches)
        with torch.cuda.stream(self.stream):
            g.replay()
        per = self.timed(g.replay, self.sync) / R
        n = max(min_launches, int(min_ms / max(per, 1e-6)))
        cyc = max(1, -(-n // (R * trials)))

        def run():
            for _ in range(cyc):
                g.replay()
        ms = [self.timed(run, self.sync) / (cyc * R) for _ in range(trials)]
        with torch.cuda.stream(self.stream):
            g_warm.replay()
        warm = self.timed(g_warm.replay, self.sync) / warm_launches
        self.check("kernel-alone timing")
        del items, g, g_warm
        return {"mean_us": 1e3 * statistics.fmean(ms), "median_us": 1e3 * statistics.median(ms),
                "min_us": 1e3 * min(ms), "warm_us": 1e3 * warm, "launches": cyc * R * trials, "trials": trials,
                "replicas": R}

    def free(self):
        self.reps = []
        self.g_step = None
        self.g_single = []
        self.torch.cuda.synchronize(self.dev)
        self.torch.cuda.empty_cache()


def new_row_bytes(w, kv_elem_bytes=2) -> int:
    """Bytes of a step's new-row store: rows read (bf16), rows written
    (pool elements) and slot ids."""
    T = w.slot_mapping.shape[0]
    return T * (w.num_kv_heads * w.head_dim * 2 * (2 + kv_elem_bytes) + 4)


def decode_entry(w, t, hbm, hbm_kind, kv_elem_bytes=2, traffic=None, fused=False, shared=0):
    """Roofline record of the decode kernel from a kernel_alone timing
    (fused: the decode step's kernel, the new rows' store included; shared:
    the shared-prefix kernel and the decode kernel, timed together)."""
    nbytes = decode_bytes(w, kv_elem_bytes=kv_elem_bytes) + (new_row_bytes(w, kv_elem_bytes) if fused else 0)
    achieved = nbytes / (t["mean_us"] * 1e-6) / 1e9
    name = "decode_kernel" + (" (fused step: new rows' store + attention)" if fused else "")
    if shared:
        name = f"shared_prefix_kernel + decode_kernel ({shared} shared blocks read once per kv head)"
    rec = {"bound": "hbm", "kernel": name + (" (e4m3 pools)" if kv_elem_bytes == 1 else ""),
           "achieved": achieved, "peak": hbm,
           "peak_kind": f"{hbm_kind} (MEASURED_PEAKS.json hbm_gbs, copy)" if hbm_kind == "measured" else "fallback",
           "unit": "GB/s", "frac": achieved / hbm, "frac_nominal": achieved / NOMINAL_HBM_GBS,
           "nominal_peak": NOMINAL_HBM_GBS, "traffic": traffic, "algorithmic_bytes": nbytes,
           "avg_launch_us": t["mean_us"], "median_us": t["median_us"], "min_us": t["min_us"],
           "warm_us": t["warm_us"], "launches": t["launches"], "replicas": t["replicas"],
           "seqs_per_s": len(decode_rows(w)) / (t["mean_us"] * 1e-6)}
    ub = decode_unique_bytes(w, kv_elem_bytes) + (new_row_bytes(w, kv_elem_bytes) if fused else 0)
    if ub != nbytes:  # blocks shared between sequences
        rec["unique_bytes"] = ub
        rec["achieved_unique_gbs"] = ub / (t["mean_us"] * 1e-6) / 1e9
        rec["frac_unique"] = rec["achieved_unique_gbs"] / hbm
    return rec


def prefill_entry(w, t, peak, kind, traffic=None):
    fl = prefill_flops(w)
    achieved = fl / (t["mean_us"] * 1e-6) / 1e12
    return {"bound": "tensor", "kernel": "prefill_kernel", "achieved": achieved, "peak": peak, "peak_kind": kind,
            "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic, "algorithmic_flops": fl,
            "avg_launch_us": t["mean_us"], "median_us": t["median_us"], "min_us": t["min_us"],
            "warm_us": t["warm_us"], "launches": t["launches"], "replicas": t["replicas"],
            "tokens_per_s": int(sum(int(w.query_lens[s]) for s in prefill_rows(w))) / (t["mean_us"] * 1e-6)}


# ----------------------------------------------------------- other calls of the library

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


def config_entry(run, hbm, hbm_kind, tpeak, tkind, clocks=None, cpu=True, cpu_budget=3.0, step=None):
    """Everything reported for one workload: step rate, kernel-alone
    rooflines (decode, prefill), the e4m3 decode and the oracle's rates."""
    w = run.w
    t0 = time.time()
    st = step or run.step_trials()
    sb = step_bytes(w)
    entry = {"workload": w.name, "config": run.config, "seqs": w.num_seqs, "query_rows": w.num_tokens,
             "step": {**st, "seqs_per_s": w.num_seqs / (st["mean_ms"] * 1e-3),
                      "tokens_per_s": w.num_tokens / (st["mean_ms"] * 1e-3),
                      "launches_per_step": run.launches_per_step, "algorithmic_bytes": sb,
                      "achieved_gbs": sb / (st["mean_ms"] * 1e-3) / 1e9,
                      "frac": sb / (st["mean_ms"] * 1e-3) / 1e9 / hbm},
             "l2": f"{run.R} rotated input replicas of {run.pool_bytes / 1e6:.0f} MB pools"}
    dec, pre = decode_rows(w), prefill_rows(w)
    dec_t = None
    if run.fused:
        entry["decode_step"] = decode_entry(w, run.kernel_alone(dec, fused=True), hbm, hbm_kind,
                                            traffic=ncu_traffic("decode_step", run.config), fused=True)
    if len(dec):
        dec_t = run.kernel_alone(dec)
        if run.shared_blocks > 0:
            entry["decode_per_sequence"] = decode_entry(w, dec_t, hbm, hbm_kind,
                                                        traffic=ncu_traffic("decode", run.config))
            entry["decode"] = decode_entry(w, run.kernel_alone(dec, shared=run.shared_blocks), hbm, hbm_kind,
                                           traffic=ncu_traffic("shared_prefix", run.config), shared=run.shared_blocks)
        else:
            entry["decode"] = decode_entry(w, dec_t, hbm, hbm_kind, traffic=ncu_traffic("decode", run.config))
    if len(pre):
        entry["prefill"] = prefill_entry(w, run.kernel_alone(pre), tpeak, tkind,
                                         traffic=ncu_traffic("prefill", run.config))
    if len(dec):
        t8 = run.kernel_alone(dec, kv_e4m3=True)
        e8 = decode_entry(w, t8, hbm, hbm_kind, kv_elem_bytes=1, traffic=ncu_traffic("fp8_decode", run.config))
        e8["speedup_vs_bf16"] = dec_t["mean_us"] / t8["mean_us"]
        e8["scales"] = "k_scale = v_scale = 1/64, pools written by the e4m3 store"
        entry["fp8_decode"] = e8
    if clocks is not None:
        entry["clocks"] = (t0, time.time())  # summarised once the sampler has stopped
    if cpu:
        if clocks is not None:
            clocks.pause(True)
        entry["cpu_baseline"] = cpu_baseline(w, cpu_budget)
        if clocks is not None:
            clocks.pause(False)
    return entry


def run_ours(args):
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
    stream = torch.cuda.Stream(device=dev)
    hbm, hbm_kind = measured_peaks()
    tpeak, tkind = measured_tensor_peak()

    # Each rank builds its own batch (weak scaling: sequences are independent
    # units, every rank owns its own pool, tables and sequences).
    w = build_workload(args.config, rank)
    run = ConfigRun(args.config, w, pkv, torch, dev, stream, args.replicas, args.partition_blocks)
    R, Tq, B = run.R, run.Tq, w.num_seqs

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        run.run_steps(max(args.warmup, 3))
    barrier()

    clocks = NvmlClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
        clocks.dense(True)
        time.sleep(0.005)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        run.run_steps(args.steps)
        e1.record(stream)
    barrier()
    t_wall1 = time.time()
    if clocks:
        clocks.dense(False)
    step_ms = e0.elapsed_time(e1) / args.steps
    step_ms_max = reduce_max(step_ms, dist)
    run.check("timed steps")

    # End to end through the public API with pinned host buffers: every step
    # copies all its inputs (one staging buffer, one copy) to the device,
    # runs the calls and brings the output back.  The input copy is a
    # pkv_copy launch (the GPU reads the pinned buffer directly), which
    # chains with the step's kernels where a copy-engine transfer would cost
    # an engine switch (about 10 us a step on this machine); the output goes
    # back without a copy: the step's kernels write its rows straight into
    # the pinned host buffer.
    # As a serving loop does, the step (its input copy from pinned memory,
    # the calls writing the pinned output) is captured through the same public
    # calls in CUDA graphs and replayed: one graph per cycle over the
    # replicas, and one per replica for the remainder.
    e2e_steps = min(args.steps, args.e2e_steps)
    host_stage = torch.from_numpy(run.stage_np).pin_memory()
    host_out = torch.empty((Tq, w.num_q_heads, w.head_dim), dtype=torch.float32).pin_memory()
    h2d = host_stage.numel()
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step(r):
        pkv.copy(r["stage"], host_stage, stream=stream)
        run.step(dict(r, out=host_out))

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(run.reps[i % R])
    stream.synchronize()
    g_e2e_cycle = run.capture(e2e_step, run.reps)
    g_e2e = [run.capture(e2e_step, [r]) for r in run.reps]

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
    run.check("end-to-end steps")
    del g_e2e_cycle, g_e2e

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

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
                   "l2": f"{R} rotated input replicas of {run.pool_bytes / 1e6:.0f} MB pools (> 129 MB L2 in total)",
                   "graph": "CUDA graph per cycle of replicas"},
        "gpu_launches": run.launches_per_step * args.steps,
        # query rows (decode rows and prefill tokens) per second over the whole step
        "tokens_per_s": world * Tq / (step_ms_max * 1e-3),
        "e2e": {"value": world * B / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": e2e_ms},
    }

    # The headline workload's own entry: kernel-alone rooflines, e4m3 decode.
    head = config_entry(run, hbm, hbm_kind, tpeak, tkind, clocks, cpu=False)
    dec, pre = head.get("decode_step") or head.get("decode"), head.get("prefill")
    if pre is not None and (dec is None or pre["avg_launch_us"] > dec["avg_launch_us"]):
        line["roofline"] = pre
        if dec is not None:
            line["decode_roofline"] = dec
    else:
        line["roofline"] = dec
        if pre is not None:
            line["prefill_roofline"] = pre
    line["fp8_decode"] = head.get("fp8_decode")
    line["block_manager"] = block_manager_timing(w, pkv, torch, dev, stream)
    line["prefix_keys"] = prefix_keys_timing(w, pkv, torch, dev, stream)
    line["prefix_cache"] = prefix_cache_timing(w, pkv, torch, dev, stream)
    line["swap"] = swap_timing(w, pkv, torch, dev, stream, run.reps)
    run.free()
    del run

    # Every workload (the headline's entry is the one above).
    configs = {}
    sweep = [] if args.sweep == "none" else [int(x) for x in args.sweep.split(",") if x]
    cpu_on = world == 1 and not args.no_cpu_baseline
    for k in sweep:
        if k == args.config:
            configs[str(k)] = head
            if cpu_on:
                clocks.pause(True)
                head["cpu_baseline"] = cpu_baseline(w, args.cpu_budget)
                clocks.pause(False)
            continue
        wk = build_workload(k)
        rk = ConfigRun(k, wk, pkv, torch, dev, stream, 0, args.partition_blocks)
        with torch.cuda.stream(stream):
            rk.run_steps(max(3, rk.R))
        stream.synchronize()
        configs[str(k)] = config_entry(rk, hbm, hbm_kind, tpeak, tkind, clocks, cpu=cpu_on,
                                       cpu_budget=args.cpu_budget)
        rk.free()
        del rk, wk
    if clocks:
        clocks.stop()
        ck = clocks.summary(t_wall0, t_wall1)
        line["clocks"] = {"sm_mhz": ck.get("sm_mhz"), "sm_max_mhz": ck.get("sm_max_mhz"),
                          "reasons": ck.get("reasons", []), "samples": ck.get("samples", 0)}
        for entry in configs.values():
            if isinstance(entry.get("clocks"), tuple):
                entry["clocks"] = clocks.summary(*entry["clocks"])
    if configs:
        line["configs"] = configs
    if cpu_on:
        own = configs.get(str(args.config))
        line["cpu_baseline"] = own["cpu_baseline"] if own else cpu_baseline(w, args.cpu_budget)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_ncu_case(args):
    """A short run for a profiler: the workload's step once, then
    `--ncu-launches` launches of one kernel (decode, decode_step, prefill,
    fp8_decode or shared_prefix: the shared-prefix decode's two kernels) over
    one copy of the inputs, no timing loops."""
    import torch

    import paged_kv_cache_291_gb300 as pkv
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    pkv.load()
    stream = torch.cuda.Stream(device=dev)
    w = build_workload(args.config)
    run = ConfigRun(args.config, w, pkv, torch, dev, stream, 1, args.partition_blocks)
    dec, pre = decode_rows(w), prefill_rows(w)
    which = args.ncu_case
    if which == "decode_step" and not run.fused:
        raise SystemExit(f"{w.name}: its step is not a plain decode step")
    if which == "shared_prefix" and run.shared_blocks == 0:
        raise SystemExit(f"{w.name}: its sequences share no prefix blocks")
    seqs = pre if which == "prefill" else dec
    if not len(seqs):
        raise SystemExit(f"{w.name} has no rows for {which}")
    t = run.kernel_alone(seqs, kv_e4m3=which == "fp8_decode", fused=which == "decode_step",
                         shared=run.shared_blocks if which == "shared_prefix" else 0,
                         min_launches=args.ncu_launches, min_ms=0.0, trials=1, warm_launches=1)
    print(json.dumps({"ncu_case": which, "workload": w.name, "launches": t["launches"] + 3,
                      "mean_us": t["mean_us"]}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--replicas", type=int, default=0, help="0 = enough pool replicas to exceed 512 MB")
    ap.add_argument("--config", type=int, default=CONFIG_ID, choices=[1, 2, 3, 4, 5],
                    help="headline workload (default: the Qwen3-1.7B decode step the metric is quoted on)")
    ap.add_argument("--sweep", default="1,2,3,4,5",
                    help="workloads reported in the `configs` object (comma list, or 'none')")
    ap.add_argument("--e2e-steps", type=int, default=4000)
    ap.add_argument("--cpu-budget", type=float, default=3.0,
                    help="seconds of one-thread oracle work per sampled step of each workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--partition-blocks", type=int, default=0, help="0 = automatic split-KV partitioning")
    ap.add_argument("--ncu-case", choices=["decode", "decode_step", "prefill", "fp8_decode", "shared_prefix"],
                    default=None,
                    help="a short run of one kernel for a profiler (no timing, no JSON bench line)")
    ap.add_argument("--ncu-launches", type=int, default=3)
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.ncu_case:
        return run_ncu_case(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
