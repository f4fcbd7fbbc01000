"""Benchmark of the paged-attention hot path on GB300.

A step is one pass of the hot path over one batch: copy-on-write block
copies, slot derivation, cache write of the new tokens, and paged attention
(split-KV with merge). The default workload is the Llama-3-70B layer shape
with prefix sharing: 256 sequences, 64 query / 8 KV heads, head_dim 128,
block size 16, lengths log-uniform in [512, 8192], groups of 16 sharing a
1024-token prefix, one copy-on-write per sequence, bf16.

Metric: algorithmic HBM GB/s of the step (each distinct live KV tile read
once per KV head, plus q, out, tables, the cache write and the block copies),
with seq-steps/s alongside. The roofline entry reports the attention call
(all its kernels) against the measured HBM copy bandwidth. `per_config`
holds the same measurement, in the same run, for the other workloads (8B,
long context, mixed chunked prefill against the tensor peak) and for the
e4m3 cache.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

Timing: W warm-up steps; then timed blocks of exactly K steps, each block
bracketed by a barrier, a device synchronisation and CUDA events on the
launching stream, repeated until about one second of device time has been
timed; ms_per_step is the median block over K (max over ranks). nvidia-smi
samples the clocks from the first warm-up step to the end of the run, and the
line reports the samples taken inside the timed blocks.

Under torchrun each rank runs its own replica of the batch on its own GPU
(weak scaling, no data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention HBM GB/s (% of GB300 peak) & seq-steps/s at 70B layer"
DEFAULT_CONFIG = "llama3_70b_prefix_bf16"
PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "paged_kv_cache_14_gb300", "csrc")

# Workloads measured beside the headline in one run: (workload, KV cache).
PER_CONFIG = (
    ("llama3_8b_bf16", "native"),
    ("long_splitkv_bf16", "native"),
    ("mixed_prefill_fp16", "native"),
    ("llama3_8b_bf16", "e4m3"),
    ("llama3_70b_prefix_bf16", "e4m3"),
    ("long_splitkv_bf16", "e4m3"),
    ("mixed_prefill_fp16", "e4m3"),
    ("llama3_70b_prefix_bf16", "e5m2"),
)


# ---------------------------------------------------------------------------
# Algorithmic bytes and FLOPs (metric bookkeeping on host arrays).
# ---------------------------------------------------------------------------

def decode_algorithmic_bytes(batch, kv_esize: int | None = None) -> dict:
    """Bytes decode must move: every distinct live (physical block, KV head)
    tile once, counting its valid tokens (the largest count any sequence
    reading it uses), for K and V; plus q, out, the block-table entries read
    and seq_lens. kv_esize = 1 for an e4m3 cache, which adds the (K, V)
    scale pair (8 bytes) of every distinct live tile. Only rows with
    q_len == 1 count (the decode rows of a mixed batch)."""
    B = batch.block_size
    esize = batch.q.element_size()
    kv_es = esize if kv_esize is None else kv_esize
    valid = {}
    whole = set()
    entries = 0
    rows = 0
    logical_tok = 0
    for i in range(batch.num_seqs):
        if int(batch.q_lens[i]) != 1:
            continue
        rows += 1
        L = int(batch.kv_lens[i])
        logical_tok += L
        nb = -(-L // B)
        entries += nb
        row = batch.block_tables[i]
        for j in range(nb):
            phys = int(row[j])
            v = min(B, L - j * B)
            if valid.get(phys, 0) < v:
                valid[phys] = v
            whole.add(phys)
    kv_tok = sum(valid.values())
    per_tok = 2 * batch.num_kv_heads * batch.head_dim * kv_es
    q_bytes = rows * batch.num_q_heads * batch.head_dim * esize
    out_bytes = q_bytes
    meta = entries * 4 + rows * 4
    if kv_esize is not None and kv_esize == 1:
        meta += len(valid) * batch.num_kv_heads * 8
    return {
        "kv_bytes": kv_tok * per_tok,
        "kv_bytes_whole_blocks": len(whole) * B * per_tok,
        "kv_bytes_logical": logical_tok * per_tok,
        "total": kv_tok * per_tok + q_bytes + out_bytes + meta,
    }


def prefill_flops(batch) -> float:
    """Tensor FLOPs of the chunk rows (q_len > 1): for every query row and
    query head, 2*D for q.k and 2*D for p.v per key it attends to."""
    f = 0.0
    for i in range(batch.num_seqs):
        ql = int(batch.q_lens[i])
        if ql <= 1:
            continue
        ctx = int(batch.kv_lens[i]) - ql
        keys = ql * ctx + ql * (ql + 1) // 2
        f += 4.0 * batch.head_dim * batch.num_q_heads * keys
    return f


def step_extra_bytes(batch, kv_esize: int | None = None) -> int:
    """Bytes of the non-attention rows of a step: block copies (read + write
    of both pools), slot derivation and the cache write (new rows read in the
    I/O dtype, written in the cache's; an e4m3 cache adds its scales)."""
    esize = batch.q.element_size()
    kv_es = esize if kv_esize is None else kv_esize
    block_bytes = batch.num_kv_heads * batch.block_size * batch.head_dim * kv_es
    scales = 8 * batch.num_kv_heads if kv_es == 1 else 0
    copies = len(batch.cow_pairs) * 2 * (2 * block_bytes + scales)
    t = len(batch.new_positions)
    slots = t * (4 + 4 + 4 + 8)
    row = batch.num_kv_heads * batch.head_dim
    write = t * (8 + 2 * row * (esize + kv_es) + 2 * scales)
    return copies + slots + write


# ---------------------------------------------------------------------------
# Clocks sampled during the run.
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi polled every 50 ms from a reader thread; every line is
    stamped with the host's monotonic clock on arrival, so the samples of a
    time window (the timed blocks) can be picked out afterwards."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id):
        # An index or a PCI bus id ("00000000:1B:00.0") as nvidia-smi --id takes.
        self.gpu_index = gpu_id
        self.proc = None
        self.samples: list[tuple[float, str]] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)
            self.proc = None

    @classmethod
    def parse(cls, line: str):
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 7:
            return None
        try:
            sm, mx = float(parts[0]), float(parts[1])
        except ValueError:
            return None
        reasons = {n for n, flag in zip(cls.NAMES, parts[3:7]) if flag.lower().startswith("active")}
        return sm, mx, reasons

    def summary(self, t0: float | None = None, t1: float | None = None) -> dict:
        """Median SM clock, max clock and throttle reasons of the samples
        taken in [t0, t1] (all samples when no window is given)."""
        sm, mx, reasons = [], [], set()
        for t, line in list(self.samples):
            if t0 is not None and not (t0 <= t <= t1):
                continue
            p = self.parse(line)
            if p is None:
                continue
            sm.append(p[0])
            mx.append(p[1])
            reasons |= p[2]
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# Helpers.
# ---------------------------------------------------------------------------

def measured_peak_hbm() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def measured_peak_tensor() -> tuple[float, str]:
    """Dense 16-bit tensor peak (TFLOP/s): the measured cuBLAS bf16 burst
    figure (fp16 has the same nominal rate, ratio 1)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst; fp16 nominal ratio 1)"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def source_sha256() -> str:
    """Hash of every CUDA source of the library (names and contents): a
    committed ncu summary applies only to the sources it was captured on."""
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            h.update(name.encode())
            with open(os.path.join(CSRC, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def profile_summary(config: str, kv_cache: str = "native") -> str:
    """The committed ncu summary of the attention call on this workload."""
    kind = "prefill" if config.startswith("mixed_prefill") else "decode"
    if kv_cache in ("e4m3", "e5m2"):
        return os.path.join(PROFILES, f"{kind}_{kv_cache}_{config}.md")
    if kind == "prefill":
        return os.path.join(PROFILES, f"prefill_{config}.md")
    return os.path.join(PROFILES, f"decode_{config}.md")


def profiled_traffic(summary: str) -> dict | None:
    """DRAM read + write bytes of one attention call (every kernel of the
    call) and of its dominant kernel, from a committed ncu summary, if the
    library's CUDA sources have not changed since it was captured."""
    try:
        text = open(summary).read()
    except OSError:
        return None
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_call = re.search(r"call_dram_bytes:\s*([0-9.eE+]+)", text)
    m_kern = re.search(r"kernel_dram_bytes:\s*([0-9.eE+]+)", text)
    m_name = re.search(r"dominant_kernel:\s*(\S+)", text)
    if not m_sha or not m_call or m_sha.group(1) != source_sha256():
        return None
    return {"call": float(m_call.group(1)), "kernel": float(m_kern.group(1)) if m_kern else None,
            "kernel_name": m_name.group(1) if m_name else None}


def reduce_max_over_ranks(values, world: int, device="cpu") -> list[float]:
    """Elementwise max of per-rank timings (the slowest rank sets the step
    time); a no-op for one rank. The only collective of the bench: timing
    bookkeeping, not data."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def weak_scaling_value(world: int, bytes_per_step: float, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank moves bytes_per_step per step (replicas)."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def timed_block_count(first_block_ms: float, min_total_ms: float, lo: int = 3, hi: int = 1000) -> int:
    """Number of K-step blocks to time so that about min_total_ms of device
    time is covered (at least lo, at most hi)."""
    if first_block_ms <= 0:
        return hi
    return int(min(hi, max(lo, math.ceil(min_total_ms / first_block_ms))))


def nvsmi_gpu_id(torch, device: int):
    """This process's GPU as nvidia-smi names it: its PCI bus id when torch
    reports one (CUDA_VISIBLE_DEVICES may renumber devices), else the index."""
    p = torch.cuda.get_device_properties(device)
    try:
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except AttributeError:
        return device


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


# ---------------------------------------------------------------------------
# CPU oracle timing (the reported baseline and the reference arm).
# ---------------------------------------------------------------------------

# Runs in a subprocess without any GPU (CUDA_VISIBLE_DEVICES=""), so its
# worker pool is forked before any GPU use in that process. Each worker runs
# the unchanged oracle on one sequence at a time, with one BLAS thread.
ORACLE_SNIPPET = r"""
import concurrent.futures as cf, json, multiprocessing as mp, os, sys, time
import numpy as np
sys.path.insert(0, {root!r})
import oracle
import oracle.fp8_kv as f8
from workloads import make_config, e4m3_pool, e5m2_pool
b = make_config({config!r})
fmt = {fmt!r}  # "native", "e4m3" or "e5m2"
fp8 = fmt != "native"
if fp8:
    pool_of = e5m2_pool if fmt == "e5m2" else e4m3_pool
    write8 = f8.reshape_and_cache_e5m2 if fmt == "e5m2" else f8.reshape_and_cache_fp8
    deq = f8.dequantize_e5m2 if fmt == "e5m2" else f8.dequantize
    kc, vc, sc = (x.numpy() for x in pool_of(b.meta.get("seed", 0), b.num_blocks, b.num_kv_heads,
                                             b.block_size, b.head_dim))
    f8.copy_blocks_fp8(kc, vc, sc, b.cow_pairs)
    slots = oracle.slot_mapping(b.block_tables, b.new_seq_ids, b.new_positions, b.block_size)
    write8(b.k_new.float().numpy(), b.v_new.float().numpy(), slots, kc, vc, sc, b.block_size)
else:
    kc = b.k_cache.clone(); vc = b.v_cache.clone()
    oracle.copy_blocks(kc, vc, b.cow_pairs)
    slots = oracle.slot_mapping(b.block_tables, b.new_seq_ids, b.new_positions, b.block_size)
    oracle.reshape_and_cache(b.k_new, b.v_new, slots, kc, vc, b.block_size)


def decode_one(i):
    if not fp8:
        oracle.decode(b.q, kc, vc, b.block_tables, b.kv_lens, b.scale, b.block_size, seqs=[i])
        return i
    # 8-bit pools: dequantise the sequence's blocks, then the same decode.
    nb = -(-int(b.kv_lens[i]) // b.block_size)
    blocks = b.block_tables[i][:nb]
    kd = deq(kc[blocks], sc[blocks, :, 0])
    vd = deq(vc[blocks], sc[blocks, :, 1])
    tables = np.zeros_like(b.block_tables)
    tables[i, :nb] = np.arange(nb)
    oracle.decode(b.q, kd, vd, tables, b.kv_lens, b.scale, b.block_size, seqs=[i])
    return i


order = [int(i) for i in np.random.default_rng(123).permutation(b.num_seqs)]
workers = max(1, min({workers!r}, b.num_seqs))
budget = {budget!r}
total_budget = {total!r}
results = []
with cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("fork")) as ex:
    list(ex.map(abs, range(workers)))  # start every worker before timing
    for rep in range({reps!r}):
        # One pass over the batch in a seeded order, cut short once the
        # budget is spent (what is in flight then is finished and counted).
        t0 = time.perf_counter(); done = []; inflight = set(); nxt = 0
        while nxt < len(order) and len(inflight) < 2 * workers:
            inflight.add(ex.submit(decode_one, order[nxt])); nxt += 1
        while inflight:
            fin, inflight = cf.wait(inflight, return_when=cf.FIRST_COMPLETED)
            done += [f.result() for f in fin]
            while nxt < len(order) and len(inflight) < 2 * workers and time.perf_counter() - t0 < budget:
                inflight.add(ex.submit(decode_one, order[nxt])); nxt += 1
        dt = time.perf_counter() - t0
        order = order[len(done):] + order[:len(done)]
        results.append(dict(seconds=dt, seqs=done, tokens=int(sum(int(b.kv_lens[i]) for i in done)),
                            workers=workers))
        if sum(r["seconds"] for r in results) > total_budget:
            break
print("ORACLE_JSON " + json.dumps(results))
"""


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_oracle_sample(config: str, budget_s: float, reps: int, fmt: str = "native",
                      workers: int | None = None, total_s: float = 1e9) -> list[dict]:
    """Up to `reps` timed passes of the oracle over the workload's sequences
    (each cut at budget_s), stopping once total_s seconds have been timed."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = ORACLE_SNIPPET.format(root=ROOT, config=config, budget=budget_s, reps=reps, fmt=fmt,
                                 workers=workers or host_cores(), total=total_s)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    for line in r.stdout.splitlines():
        if line.startswith("ORACLE_JSON "):
            return json.loads(line[len("ORACLE_JSON "):])
    raise RuntimeError("oracle sample failed:\n" + r.stdout[-2000:] + r.stderr[-4000:])


def oracle_rate(res: dict, per_seq_bytes: np.ndarray) -> tuple[float, float]:
    """(GB/s, seq-steps/s) of the oracle over its sample: the algorithmic
    decode bytes of the sampled sequences over the time it took."""
    seqs = res["seqs"]
    byts = float(per_seq_bytes[seqs].sum())
    return byts / res["seconds"] / 1e9, len(seqs) / res["seconds"]


def per_seq_decode_bytes(batch, kv_esize: int | None = None) -> np.ndarray:
    esize = batch.q.element_size()
    per_tok = 2 * batch.num_kv_heads * batch.head_dim * (esize if kv_esize is None else kv_esize)
    qo = 2 * batch.num_q_heads * batch.head_dim * esize
    return batch.kv_lens.astype(np.float64) * per_tok + qo


def cpu_baseline_entry(res: dict, value: float, unit: str, fmt: str, num_seqs: int) -> dict:
    return {"value": round(value, 6), "unit": unit, "cores": res["workers"], "kind": "oracle",
            "host_cores": host_cores(), "blas_threads_per_worker": 1,
            "sample": f"decode of {len(res['seqs'])} of {num_seqs} sequences ({res['tokens']} keys) in "
                      f"{res['seconds']:.2f} s, fp64 numpy, {res['workers']} worker processes x 1 thread, "
                      "one sequence per task" + (f" ({fmt} pools dequantised per sequence)" if fmt != "native" else "")}


# ---------------------------------------------------------------------------
# Arms.
# ---------------------------------------------------------------------------

def reference_arm(args) -> None:
    from workloads import make_config
    rank, world, _ = dist_info()
    if rank != 0:
        return
    batch = make_config(args.config, with_values=False)
    per_seq = per_seq_decode_bytes(batch)
    steps = args.warmup + args.steps
    budget = max(0.5, min(20.0, 150.0 / max(1, steps)))
    res = run_oracle_sample(args.config, budget, steps)
    timed = res[args.warmup:]
    secs = sum(r["seconds"] for r in timed)
    byts = sum(float(per_seq[r["seqs"]].sum()) for r in timed)
    nseq = sum(len(r["seqs"]) for r in timed)
    value = byts / secs / 1e9
    merged = {"seconds": secs, "seqs": [i for r in timed for i in r["seqs"]],
              "tokens": sum(r["tokens"] for r in timed), "workers": timed[0]["workers"]}
    cpu = cpu_baseline_entry(merged, value, "GB/s", "native", batch.num_seqs * len(timed))
    cpu["sample"] = (f"{len(timed)} steps, each one pass over the {batch.num_seqs} sequences in a seeded order "
                     f"(cut at ~{budget:.1f} s): " + cpu["sample"])
    line = {
        "impl": "reference", "metric": METRIC,
        "value": round(value, 6), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000.0 * secs / len(timed), 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "seq_steps_per_s": round(nseq / secs, 4),
        "config": {"workload": args.config,
                   "sample": "one pass over the batch's sequences per step, cut at ~%.1f s" % budget},
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


class Timer:
    """CUDA-event timing on the launching stream."""

    def __init__(self, torch, stream, barrier):
        self.torch, self.stream, self.barrier = torch, stream, barrier

    def block(self, fn, n: int) -> tuple[float, float, float]:
        """Runs fn n times between two events, bracketed by barrier + device
        synchronisation. Returns (ms, host start, host end)."""
        ev = self.torch.cuda.Event
        a, b = ev(enable_timing=True), ev(enable_timing=True)
        self.barrier()
        t0 = time.monotonic()
        a.record(self.stream)
        for _ in range(n):
            fn()
        b.record(self.stream)
        self.barrier()
        return a.elapsed_time(b), t0, time.monotonic()

    def each(self, before, fn, n: int) -> list[float]:
        """n calls of fn, each between its own pair of events, with `before`
        run (untimed) ahead of each."""
        ev = self.torch.cuda.Event
        pairs = [(ev(enable_timing=True), ev(enable_timing=True)) for _ in range(n)]
        self.barrier()
        for a, b in pairs:
            before()
            a.record(self.stream)
            fn()
            b.record(self.stream)
        self.barrier()
        return [a.elapsed_time(b) for a, b in pairs]


def attention_entry(pa, st, batch, kv_es, timer, calls: int, config: str, kv_cache: str) -> dict:
    """Roofline entry of the step's attention call alone: `calls` calls, each
    after the step's cache side, timed one by one; median call."""
    ms = timer.each(st.prepare, st.attend, calls)
    med = statistics.median(ms)
    prof = profiled_traffic(profile_summary(config, kv_cache))
    if st.is_decode:
        byts = decode_algorithmic_bytes(batch, kv_es)
        peak, kind = measured_peak_hbm()
        gbs = byts["total"] / (med * 1e-3) / 1e9
        return {"kernel": st.attention_kernels, "bound": "hbm", "achieved": round(gbs, 2), "peak": peak,
                "peak_kind": kind, "unit": "GB/s", "frac": round(gbs / peak, 4),
                "traffic": prof["call"] if prof else None,
                "traffic_scope": "DRAM read + write of one whole attention call (all its kernels), ncu",
                "dominant_kernel_traffic": prof["kernel"] if prof else None,
                "algorithmic_bytes": byts["total"], "ms_per_launch": round(med, 5),
                "ms_per_launch_mean": round(statistics.mean(ms), 5), "calls": calls}
    flops = prefill_flops(batch)
    tpeak, tkind = measured_peak_tensor()
    hpeak, _ = measured_peak_hbm()
    rows = decode_algorithmic_bytes(batch)["total"]
    tf = flops / (med * 1e-3) / 1e12
    return {"kernel": st.attention_kernels, "bound": "tensor", "achieved": round(tf, 2), "peak": tpeak,
            "peak_kind": tkind, "unit": "TFLOP/s", "frac": round(tf / tpeak, 4),
            "traffic": prof["call"] if prof else None,
            "traffic_scope": "DRAM read + write of one whole attention call (all its kernels), ncu",
            "algorithmic_flops": flops, "decode_rows_algorithmic_bytes": rows,
            "bound_ms": {"chunk_flops_at_tensor_peak": round(flops / (tpeak * 1e12) * 1e3, 5),
                         "decode_rows_bytes_at_hbm_peak": round(rows / (hpeak * 1e9) * 1e3, 5)},
            "ms_per_launch": round(med, 5), "ms_per_launch_mean": round(statistics.mean(ms), 5), "calls": calls}


def chunk_only_entry(pa, torch, st, batch, timer, calls: int) -> dict:
    """The chunk rows (q_len > 1) of a mixed batch alone, as one
    pa_chunked_prefill call: the tensor-core chunk kernel and its plan."""
    idx = [i for i in range(batch.num_seqs) if int(batch.q_lens[i]) > 1]
    cu = batch.cu_q_lens
    q = torch.cat([st.q[int(cu[i]):int(cu[i + 1])] for i in idx]).contiguous()
    ql = np.array([int(batch.q_lens[i]) for i in idx], np.int64)
    cuq = torch.tensor(np.concatenate([[0], np.cumsum(ql)]), dtype=torch.int32, device=q.device)
    sel = torch.tensor(idx, dtype=torch.long, device=q.device)
    tables = st.block_tables.index_select(0, sel).contiguous()
    ctx = st.ctx_lens.index_select(0, sel).contiguous()
    out = torch.empty_like(q)
    ws = torch.empty(max(16, pa.pa_chunked_prefill_workspace_size(
        len(idx), q.shape[1], st.num_kv_heads, st.head_dim, st.block_size, q.shape[0], st.max_seq_len)),
        dtype=torch.uint8, device=q.device)
    max_q = int(ql.max())

    def call():
        if st.kv_scales is not None:
            chunked_8bit = st.call_8bit("pa_chunked_prefill")  # e4m3 (_fp8) or e5m2 codes
            chunked_8bit(q, cuq, st.k_cache, st.v_cache, st.kv_scales, tables, ctx, max_q, st.max_seq_len,
                         batch.scale, out=out, workspace=ws)
        else:
            pa.pa_chunked_prefill(q, cuq, st.k_cache, st.v_cache, tables, ctx, max_q, st.max_seq_len, batch.scale,
                                  out=out, workspace=ws)
    for _ in range(3):
        call()
    ms = timer.each(lambda: None, call, calls)
    med = statistics.median(ms)
    flops = prefill_flops(batch)
    tpeak, tkind = measured_peak_tensor()
    tf = flops / (med * 1e-3) / 1e12
    return {"kernel": "prefill plan + tcgen05 chunk kernel (the batch's chunks only, no decode rows)",
            "bound": "tensor", "achieved": round(tf, 2), "peak": tpeak, "peak_kind": tkind, "unit": "TFLOP/s",
            "frac": round(tf / tpeak, 4), "algorithmic_flops": flops, "ms_per_launch": round(med, 5),
            "calls": calls}


def per_config_entry(pa, torch, batch, kv_cache: str, timer, steps: int, warmup: int) -> dict:
    """Step and attention-call measurements of one more workload."""
    from paged_kv_cache_14_gb300.step import step_from_host
    from workloads import e4m3_pool, e5m2_pool
    fp8 = kv_cache in ("e4m3", "e5m2")
    pool = (e5m2_pool if kv_cache == "e5m2" else e4m3_pool)(
        batch.meta["seed"], batch.num_blocks, batch.num_kv_heads, batch.block_size, batch.head_dim) if fp8 else None
    shared = batch.is_decode and batch.prefix_lens is not None and bool(batch.prefix_lens.any())
    st = step_from_host(batch, shared_prefix=shared, fp8_pool=pool, kv_format=kv_cache if fp8 else "e4m3")
    kv_es = 1 if fp8 else None
    for _ in range(warmup):
        st.run()
    n = max(steps, 50)
    ms_block, _, _ = timer.block(st.run, n)
    step_bytes = decode_algorithmic_bytes(batch, kv_es)["total"] + step_extra_bytes(batch, kv_es)
    entry = {"workload": batch.name, "kv_cache": f"{kv_cache} codes + fp32 (K, V) scale per (block, KV head)"
             if fp8 else batch.dtype, "step": st.step_calls, "steps": n,
             "ms_per_step": round(ms_block / n, 5),
             "roofline": attention_entry(pa, st, batch, kv_es, timer, n, batch.name, kv_cache)}
    if st.is_decode:
        entry["step_gbs"] = round(step_bytes / (ms_block / n * 1e-3) / 1e9, 2)
        entry["seq_steps_per_s"] = round(batch.num_seqs / (ms_block / n * 1e-3), 1)
    else:
        entry["chunks_only"] = chunk_only_entry(pa, torch, st, batch, timer, n)
    status = pa.pa_get_status()
    if status != 0:
        raise RuntimeError(f"device status after {batch.name}/{kv_cache}: {pa.pa_strerror(status)}")
    del st
    torch.cuda.empty_cache()
    return entry


def native_arm(args) -> None:
    import torch
    import torch.distributed as dist

    import paged_kv_cache_14_gb300 as pa
    from paged_kv_cache_14_gb300.step import HostPipeline, step_from_host
    from workloads import e4m3_pool, e5m2_pool, make_config

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    pa.load()
    batch = make_config(args.config)
    fp8 = args.kv_cache in ("e4m3", "e5m2")
    shared = batch.is_decode and (args.decode == "shared_prefix" or (
        args.decode == "auto" and batch.prefix_lens is not None and bool(batch.prefix_lens.any())))
    pool = (e5m2_pool if args.kv_cache == "e5m2" else e4m3_pool)(
        batch.meta["seed"], batch.num_blocks, batch.num_kv_heads, batch.block_size, batch.head_dim) if fp8 else None
    st = step_from_host(batch, partition_size=args.partition, shared_prefix=shared, fp8_pool=pool,
                        kv_format=args.kv_cache if fp8 else "e4m3")
    if args.attention_once:
        # One attention call after warm-up steps, nothing timed: the command
        # the committed ncu summaries capture (its last launches are one
        # cache side and one attention call).
        for _ in range(args.warmup):
            st.run()
        torch.cuda.synchronize()
        st.prepare()
        st.attend()
        torch.cuda.synchronize()
        status = pa.pa_get_status()
        print(json.dumps({"attention_once": args.config, "kv_cache": args.kv_cache, "kernels": st.attention_kernels,
                          "status": status}), flush=True)
        if status != 0:
            raise RuntimeError(f"device status: {pa.pa_strerror(status)}")
        return
    kv_es = 1 if fp8 else None
    dec_bytes = decode_algorithmic_bytes(batch, kv_es)
    step_bytes = dec_bytes["total"] + step_extra_bytes(batch, kv_es)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    timer = Timer(torch, stream, barrier)
    clk = ClockSampler(nvsmi_gpu_id(torch, local)).start()
    try:
        # Warm-up (untimed), then check the device status once.
        for _ in range(args.warmup):
            st.run()
        status = pa.pa_get_status()
        if status != 0:
            raise RuntimeError(f"device status after warm-up: {pa.pa_strerror(status)}")

        # Timed region: blocks of exactly K whole steps (PagedStep.run: one
        # call for a decode step, whose planning runs beside the cache side).
        # The block count is fixed from a first block, agreed over ranks.
        first, _, _ = timer.block(st.run, args.steps)
        reps = timed_block_count(reduce_max_over_ranks([first], world, "cuda")[0], args.min_timed_ms)
        blocks = []
        t_first = t_last = None
        for _ in range(reps):
            ms, t0, t1 = timer.block(st.run, args.steps)
            blocks.append(ms)
            t_first = t0 if t_first is None else t_first
            t_last = t1
        clocks = clk.summary(t_first, t_last)
        ms_step_local = statistics.median(blocks) / args.steps

        # The attention call alone (the roofline entry).
        calls = max(args.steps, 200)
        roof = attention_entry(pa, st, batch, kv_es, timer, calls, args.config, args.kv_cache)
        status = pa.pa_get_status()
        if status != 0:
            raise RuntimeError(f"device status after timed steps: {pa.pa_strerror(status)}")

        # End to end through the public API with host buffers: every step
        # copies its inputs from pinned host memory and reads the output back,
        # through the package's host-fed pipeline (copies on copy streams,
        # overlapped with the neighbouring steps' compute, two buffer sets).
        host = {
            "q": batch.q.pin_memory(), "k_new": batch.k_new.pin_memory(), "v_new": batch.v_new.pin_memory(),
            "block_tables": torch.from_numpy(batch.block_tables).pin_memory(),
            "kv_lens": torch.from_numpy(batch.kv_lens).pin_memory(),
            "new_seq_ids": torch.from_numpy(batch.new_seq_ids).pin_memory(),
            "new_positions": torch.from_numpy(batch.new_positions).pin_memory(),
        }
        if st.shared_prefix:
            host["group_starts"] = torch.from_numpy(batch.group_starts).pin_memory()
            host["prefix_lens"] = torch.from_numpy(batch.prefix_lens).pin_memory()
        if not st.is_decode:
            host["cu_q_lens"] = torch.from_numpy(batch.cu_q_lens).pin_memory()
            host["ctx_lens"] = torch.from_numpy(batch.ctx_lens).pin_memory()
        out_host = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_host.numel() * out_host.element_size()
        pipe = HostPipeline(st, stream)
        for _ in range(4):
            pipe.submit(host, out_host)
        pipe.drain()
        e2e_steps = max(args.steps, args.e2e_steps)
        e_start = torch.cuda.Event(enable_timing=True)
        e_stop = torch.cuda.Event(enable_timing=True)
        barrier()
        w0 = time.perf_counter()
        e_start.record(stream)
        for _ in range(e2e_steps):
            pipe.submit(host, out_host)
        pipe.drain()  # the last output copy is inside the timed span
        e_stop.record(stream)
        barrier()
        e2e_ms = e_start.elapsed_time(e_stop) / e2e_steps
        wall_ms = (time.perf_counter() - w0) * 1000.0 / e2e_steps

        per_config = None
        if world == 1 and not args.no_per_config:
            per_config = {}
            for name, kv in PER_CONFIG:
                b2 = batch if name == args.config else make_config(name)
                per_config[f"{name}/{kv}"] = per_config_entry(pa, torch, b2, kv, timer, args.steps, args.warmup)
                del b2
            clocks_all = clk.summary()
        else:
            clocks_all = None
    finally:
        clk.stop()

    ms_step, e2e_ms = reduce_max_over_ranks([ms_step_local, e2e_ms], world, "cuda")
    peak, peak_kind = measured_peak_hbm()
    value = weak_scaling_value(world, step_bytes, ms_step)
    e2e_value = weak_scaling_value(world, step_bytes, e2e_ms)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline and st.is_decode:
        # Passes over the batch until about cpu_seconds are timed; the first
        # pass (worker start-up, first touch of the pools) is not counted.
        runs = run_oracle_sample(args.config, args.cpu_seconds, 1000, fmt=args.kv_cache, total_s=args.cpu_seconds)
        timed = runs[1:] or runs
        res = {"seconds": sum(r["seconds"] for r in timed), "seqs": [i for r in timed for i in r["seqs"]],
               "tokens": sum(r["tokens"] for r in timed), "workers": timed[0]["workers"]}
        gbs, sps = oracle_rate(res, per_seq_decode_bytes(batch, kv_es))
        cpu = cpu_baseline_entry(res, gbs, "GB/s", args.kv_cache, batch.num_seqs * len(timed))
        cpu["sample"] = f"{len(timed)} passes over the batch after one untimed pass: " + cpu["sample"]
        cpu["seq_steps_per_s"] = round(sps, 4)
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": args.kv_cache if fp8 else batch.dtype,
            "data": "synthetic (seeded)"
                    + (f", {args.kv_cache} pools drawn as codes + per-block scales" if fp8 else ""),
            "pct_of_peak": round(100.0 * value / world / peak, 2),
            "seq_steps_per_s": round(world * batch.num_seqs / (ms_step * 1e-3), 1),
            "timing": {"timed_blocks": reps, "steps_per_block": args.steps,
                       "block_ms_median": round(statistics.median(blocks), 5),
                       "block_ms_min": round(min(blocks), 5), "block_ms_max": round(max(blocks), 5),
                       "ms_per_step": "median block / steps, max over ranks"},
            "config": {
                "workload": args.config, "num_seqs": batch.num_seqs, "num_q_heads": batch.num_q_heads,
                "num_kv_heads": batch.num_kv_heads, "head_dim": batch.head_dim, "block_size": batch.block_size,
                "max_seq_len": batch.max_seq_len, "sum_seq_len": int(batch.kv_lens.sum()),
                "cow_pairs": int(len(batch.cow_pairs)), "partition": pa.pa_decode_partition_size(
                    batch.num_seqs, batch.num_q_heads, batch.num_kv_heads, batch.block_size, batch.max_seq_len,
                    args.partition),
                "kv_cache": (f"{args.kv_cache} codes + fp32 (K, V) scale per (block, KV head); q/out " + batch.dtype)
                if fp8 else batch.dtype,
                "step": st.step_calls, "step_bytes": step_bytes, "decode_bytes": dec_bytes,
                "launches_per_step": st.launches,
                "l2": "inputs larger than L2 (KV pools %.2f GB vs 129 MB L2); no flush" % (
                    2 * st.k_cache.numel() * st.k_cache.element_size() / 1e9),
                "parallelism": f"replicas x{world}",
            },
            "roofline": roof,
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5), "steps": e2e_steps,
                    "wall_ms_per_step": round(wall_ms, 5),
                    "path": "paged_kv_cache_14_gb300.step.HostPipeline (pinned host in, pinned host out)"},
            "gpu_launches": st.launches * args.steps * reps,
            "clocks": clocks,
            "clocks_whole_run": clocks_all,
            "cpu_baseline": cpu,
            "per_config": per_config,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--decode", choices=("auto", "plain", "shared_prefix"), default="auto",
                    help="auto: shared-prefix decode when the workload's sequences share prefix blocks")
    ap.add_argument("--kv-cache", choices=("native", "e4m3", "e5m2"), default="native",
                    help="native: the pools hold q's dtype; e4m3 / e5m2: 8-bit codes with per-block scales")
    ap.add_argument("--attention-once", action="store_true",
                    help="run warm-up steps, then one cache side and one attention call, and exit (for ncu)")
    ap.add_argument("--min-timed-ms", type=float, default=1000.0,
                    help="device time the repeated K-step blocks cover")
    ap.add_argument("--e2e-steps", type=int, default=400)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        reference_arm(args)
    else:
        native_arm(args)


if __name__ == "__main__":
    main()
