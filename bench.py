"""Benchmark of the paged-attention hot path on GB300.

A step is one pass of the hot path over one batch: copy-on-write block
copies, slot derivation, cache write of the new tokens, and paged decode
attention (split-KV with merge). The default workload is the Llama-3-70B
layer shape with prefix sharing: 256 sequences, 64 query / 8 KV heads,
head_dim 128, block size 16, lengths log-uniform in [512, 8192], groups of 16
sharing a 1024-token prefix, one copy-on-write per sequence, bf16.

Metric: algorithmic HBM GB/s of the step (each distinct live KV tile read
once per KV head, plus q, out, tables, the cache write and the block copies),
with seq-steps/s alongside. The roofline entry reports the decode launch
(main + merge kernels) against the measured HBM copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

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

DEFAULT_CONFIG = "llama3_70b_prefix_bf16"
PROFILES = os.path.join(ROOT, "profiles")


def profile_summary(config: str, fp8: bool) -> str:
    """The committed ncu summary of the decode kernel on this workload."""
    return os.path.join(PROFILES, f"decode_e4m3_{config}.md" if fp8 else f"decode_{config}.md")
DECODE_SRC = os.path.join(ROOT, "paged_kv_cache_14_gb300", "csrc", "pa_decode.cu")


# ---------------------------------------------------------------------------
# Algorithmic bytes (metric bookkeeping on host arrays).
# ---------------------------------------------------------------------------

def decode_algorithmic_bytes(batch, kv_esize: int | None = None) -> dict:
    """Bytes decode must move: every distinct live (physical block, KV head)
    tile once, counting its valid tokens (the largest count any sequence
    reading it uses), for K and V; plus q, out, the block-table entries read
    and seq_lens. kv_esize = 1 for an e4m3 cache, which adds the (K, V)
    scale pair (8 bytes) of every distinct live tile."""
    B = batch.block_size
    esize = batch.q.element_size()
    kv_es = esize if kv_esize is None else kv_esize
    valid = {}
    whole = set()
    entries = 0
    for i in range(batch.num_seqs):
        L = int(batch.kv_lens[i])
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
    q_bytes = batch.q.numel() * esize
    out_bytes = q_bytes
    meta = entries * 4 + batch.num_seqs * 4
    if kv_esize is not None and kv_esize == 1:
        meta += len(valid) * batch.num_kv_heads * 8
    logical_tok = int(np.sum(batch.kv_lens))
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
# Clocks sampled during the timed region.
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def __enter__(self):
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
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, flag in zip(names, parts[3:7]):
                if flag.lower().startswith("active"):
                    reasons.add(n)
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


def profiled_traffic(summary: str) -> float | None:
    """DRAM bytes per decode launch from a committed ncu summary, if the
    decode source has not changed since it was captured."""
    try:
        text = open(summary).read()
    except OSError:
        return None
    m_sha = re.search(r"decode_source_sha256:\s*([0-9a-f]{64})", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_tr:
        return None
    sha = hashlib.sha256(open(DECODE_SRC, "rb").read()).hexdigest()
    return float(m_tr.group(1)) if sha == m_sha.group(1) else None


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


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


# ---------------------------------------------------------------------------
# CPU oracle timing (the reported baseline and the reference arm).
# ---------------------------------------------------------------------------

ORACLE_SNIPPET = r"""
import json, sys, time, numpy as np
sys.path.insert(0, {root!r})
import oracle
import oracle.fp8_kv as f8
from workloads import make_config, e4m3_pool
b = make_config({config!r})
fp8 = {fp8!r}
if fp8:
    kc, vc, sc = (x.numpy() for x in e4m3_pool(b.meta.get("seed", 0), b.num_blocks, b.num_kv_heads,
                                               b.block_size, b.head_dim))
    f8.copy_blocks_fp8(kc, vc, sc, b.cow_pairs)
    slots = oracle.slot_mapping(b.block_tables, b.new_seq_ids, b.new_positions, b.block_size)
    f8.reshape_and_cache_fp8(b.k_new.float().numpy(), b.v_new.float().numpy(), slots, kc, vc, sc, b.block_size)
else:
    kc = b.k_cache.clone(); vc = b.v_cache.clone()
    oracle.copy_blocks(kc, vc, b.cow_pairs)
    slots = oracle.slot_mapping(b.block_tables, b.new_seq_ids, b.new_positions, b.block_size)
    oracle.reshape_and_cache(b.k_new, b.v_new, slots, kc, vc, b.block_size)


def decode_one(i):
    if not fp8:
        return oracle.decode(b.q, kc, vc, b.block_tables, b.kv_lens, b.scale, b.block_size, seqs=[i])
    # e4m3: dequantise the sequence's blocks, then the same decode.
    nb = -(-int(b.kv_lens[i]) // b.block_size)
    blocks = b.block_tables[i][:nb]
    kd = f8.dequantize(kc[blocks], sc[blocks, :, 0])
    vd = f8.dequantize(vc[blocks], sc[blocks, :, 1])
    tables = np.zeros_like(b.block_tables)
    tables[i, :nb] = np.arange(nb)
    return oracle.decode(b.q, kd, vd, tables, b.kv_lens, b.scale, b.block_size, seqs=[i])


rng = np.random.default_rng(123)
order = rng.permutation(b.num_seqs)
budget = {budget!r}
results = []
for rep in range({reps!r}):
    t0 = time.perf_counter(); done = []; toks = 0
    for i in order:
        decode_one(int(i))
        done.append(int(i)); toks += int(b.kv_lens[i])
        if time.perf_counter() - t0 > budget:
            break
    dt = time.perf_counter() - t0
    order = np.roll(order, -len(done))
    results.append(dict(seconds=dt, seqs=done, tokens=toks))
print("ORACLE_JSON " + json.dumps(results))
"""


def run_oracle_sample(config: str, budget_s: float, reps: int, fp8: bool = False) -> list[dict]:
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = ORACLE_SNIPPET.format(root=ROOT, config=config, budget=budget_s, reps=reps, fp8=fp8)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    for line in r.stdout.splitlines():
        if line.startswith("ORACLE_JSON "):
            return json.loads(line[len("ORACLE_JSON "):])
    raise RuntimeError("oracle sample failed:\n" + r.stdout[-2000:] + r.stderr[-4000:])


def oracle_rate(batch, res: dict, per_seq_bytes: np.ndarray) -> tuple[float, float]:
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
    line = {
        "impl": "reference", "metric": "paged decode attention HBM GB/s (% of GB300 peak) & seq-steps/s at 70B layer",
        "value": round(value, 6), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000.0 * secs / len(timed), 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "seq_steps_per_s": round(nseq / secs, 4),
        "config": {"workload": args.config, "sample": "sequences in a seeded random order until ~%.1f s per step"
                   % budget},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{nseq} sequences over {len(timed)} steps of ~{budget:.1f} s"},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def native_arm(args) -> None:
    import torch
    import torch.distributed as dist

    import paged_kv_cache_14_gb300 as pa
    from paged_kv_cache_14_gb300.step import HostPipeline, step_from_host
    from workloads import e4m3_pool, make_config

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    pa.load()
    batch = make_config(args.config)
    fp8 = args.kv_cache == "e4m3"
    if fp8 and (args.decode == "shared_prefix" or not batch.is_decode):
        raise SystemExit("the e4m3 cache runs plain decode only")
    shared = not fp8 and (args.decode == "shared_prefix" or (
        args.decode == "auto" and batch.is_decode and batch.prefix_lens is not None and bool(batch.prefix_lens.any())))
    pool = e4m3_pool(batch.meta["seed"], batch.num_blocks, batch.num_kv_heads, batch.block_size,
                     batch.head_dim) if fp8 else None
    st = step_from_host(batch, partition_size=args.partition, shared_prefix=shared, fp8_pool=pool)
    kv_es = 1 if fp8 else None
    dec_bytes = decode_algorithmic_bytes(batch, kv_es)
    step_bytes = dec_bytes["total"] + step_extra_bytes(batch, kv_es)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # Warm-up (untimed), then check the device status once.
    for _ in range(args.warmup):
        st.run()
    status = pa.pa_get_status()
    if status != 0:
        raise RuntimeError(f"device status after warm-up: {pa.pa_strerror(status)}")

    # Timed region: K whole steps (PagedStep.run: one call for a
    # shared-prefix step, whose prefix check runs beside the cache side),
    # bracketed by CUDA events on the launching stream.
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        start.record(stream)
        for i in range(args.steps):
            st.run()
        stop.record(stream)
        barrier()
        clocks = clk.summary()
    ms_total = start.elapsed_time(stop)
    # The attention call alone (the roofline entry): K more steps run as
    # cache side + attention call, with events around each attention call.
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    for i in range(args.steps):
        st.prepare()
        ev[i][0].record(stream)
        st.attend()
        ev[i][1].record(stream)
    barrier()
    dec_ms = [a.elapsed_time(b) for a, b in ev]
    status = pa.pa_get_status()
    if status != 0:
        raise RuntimeError(f"device status after timed steps: {pa.pa_strerror(status)}")

    # End to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory and reads the output back.
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
    e2e_steps = max(1, args.steps // 4)
    # Through the package's host-fed pipeline: every step's inputs are copied
    # in and its output copied out on copy streams, overlapped with the
    # neighbouring steps' compute (two device buffer sets).
    pipe = HostPipeline(st, stream)
    for _ in range(2):
        pipe.submit(host, out_host)
    pipe.drain()
    barrier()
    t0 = time.perf_counter()
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for _ in range(e2e_steps):
        pipe.submit(host, out_host)
    pipe.drain()
    e_stop.record(stream)
    barrier()
    e2e_ms = e_start.elapsed_time(e_stop) / e2e_steps
    wall_ms = (time.perf_counter() - t0) * 1000.0 / e2e_steps

    # Max over ranks.
    ms_total, e2e_ms, dec_mean = reduce_max_over_ranks([ms_total, e2e_ms, statistics.mean(dec_ms)], world, "cuda")
    ms_step = ms_total / args.steps

    peak, peak_kind = measured_peak_hbm()
    if not st.is_decode:
        flops = prefill_flops(batch)
        tpeak, tkind = measured_peak_tensor()
        achieved_tf = flops / (dec_mean * 1e-3) / 1e12
    value = weak_scaling_value(world, step_bytes, ms_step)
    e2e_value = weak_scaling_value(world, step_bytes, e2e_ms)
    dec_gbs = dec_bytes["total"] / (dec_mean * 1e-3) / 1e9
    cpu = None
    if rank == 0 and not args.no_cpu_baseline and st.is_decode:
        res = run_oracle_sample(args.config, args.cpu_seconds, 1, fp8=fp8)[0]
        gbs, sps = oracle_rate(batch, res, per_seq_decode_bytes(batch, kv_es))
        cpu = {"value": round(gbs, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"decode of {len(res['seqs'])} of {batch.num_seqs} sequences "
                         f"({res['tokens']} keys) in {res['seconds']:.1f} s, fp64 numpy, 1 thread"
                         + (" (e4m3 pools dequantised per sequence)" if fp8 else ""),
               "seq_steps_per_s": round(sps, 4)}
    if rank == 0:
        line = {
            "metric": "paged decode attention HBM GB/s (% of GB300 peak) & seq-steps/s at 70B layer",
            "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if fp8 else batch.dtype,
            "data": "synthetic (seeded)" + (", e4m3 pools drawn as codes + per-block scales" if fp8 else ""),
            "pct_of_peak": round(100.0 * value / world / peak, 2),
            "seq_steps_per_s": round(world * batch.num_seqs / (ms_step * 1e-3), 1),
            "config": {
                "workload": args.config, "num_seqs": batch.num_seqs, "num_q_heads": batch.num_q_heads,
                "num_kv_heads": batch.num_kv_heads, "head_dim": batch.head_dim, "block_size": batch.block_size,
                "max_seq_len": batch.max_seq_len, "sum_seq_len": int(batch.kv_lens.sum()),
                "cow_pairs": int(len(batch.cow_pairs)), "partition": pa.pa_decode_partition_size(
                    batch.num_seqs, batch.num_q_heads, batch.num_kv_heads, batch.block_size, batch.max_seq_len,
                    args.partition),
                "kv_cache": ("e4m3 codes + fp32 (K, V) scale per (block, KV head); q/out " + batch.dtype)
                if fp8 else batch.dtype,
                "step": ("copy_blocks_fp8 + slot_mapping + reshape_and_cache_fp8 + pa_decode_fp8" if fp8 else
                         "pa_decode_step_shared_prefix (copy_blocks + slot_mapping + reshape_and_cache + "
                         "pa_decode_shared_prefix in one call)" if st.shared_prefix else
                         "pa_decode_step (copy_blocks + slot_mapping + reshape_and_cache + pa_decode in one call)"
                         if st.is_decode and st.q.dtype != torch.float32 else
                         "copy_blocks + slot_mapping + reshape_and_cache + " + (
                             "pa_decode" if st.is_decode else "pa_chunked_prefill")),
                "step_bytes": step_bytes, "decode_bytes": dec_bytes,
                "l2": "inputs larger than L2 (KV pools %.2f GB vs 129 MB L2); no flush" % (
                    2 * st.k_cache.numel() * st.k_cache.element_size() / 1e9),
                "parallelism": f"replicas x{world}",
            },
            "roofline": ({"kernel": ("paged decode, shared-prefix (prefix check + tcgen05 prefix pass + split-KV "
                                     "suffix decode + merge)" if st.shared_prefix else
                                     "paged decode over the e4m3 cache (plan + main + split-KV merge)" if fp8 else
                                     "paged decode (plan + main + split-KV merge)"), "bound": "hbm",
                          "achieved": round(dec_gbs, 2), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                          "frac": round(dec_gbs / peak, 4),
                          "traffic": profiled_traffic(profile_summary(args.config, fp8)),
                          "algorithmic_bytes": dec_bytes["total"], "ms_per_launch": round(dec_mean, 5)}
                         if st.is_decode else
                         {"kernel": "chunked prefill call (tcgen05 chunk tiles + decode rows)", "bound": "tensor",
                          "achieved": round(achieved_tf, 2), "peak": tpeak, "peak_kind": tkind,
                          "unit": "TFLOP/s", "frac": round(achieved_tf / tpeak, 4), "traffic": None,
                          "algorithmic_flops": flops, "ms_per_launch": round(dec_mean, 5)}),
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5),
                    "wall_ms_per_step": round(wall_ms, 5)},
            "gpu_launches": st.launches * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--decode", choices=("auto", "plain", "shared_prefix"), default="auto",
                    help="auto: shared-prefix decode when the workload's sequences share prefix blocks")
    ap.add_argument("--kv-cache", choices=("native", "e4m3"), default="native",
                    help="native: the pools hold q's dtype; e4m3: e4m3 codes with per-block scales")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        reference_arm(args)
    else:
        native_arm(args)


if __name__ == "__main__":
    main()
