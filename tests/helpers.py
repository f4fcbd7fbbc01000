"""Shared test helpers: oracle references for a seeded batch and the
tolerances the CUDA path must meet.

Tolerances (attention outputs, compared after an exact up-cast to float64):
  * bf16 / fp16 I/O: max |gpu - oracle| <= 2e-2 and mean |gpu - oracle| <= 2e-3
  * fp32 I/O: per output row (one query token, one head), max |gpu - oracle|
    / max |oracle| <= 1e-5
Cache writes, block copies and slot mappings must be bit-exact.
"""
from __future__ import annotations

import dataclasses
import functools

import numpy as np
import torch

import oracle

BF_MAX_ABS = 2e-2
BF_MEAN_ABS = 2e-3
F32_REL = 1e-5


def assert_attention_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "") -> dict:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    stats = {"max_abs": float(err.max()), "mean_abs": float(err.mean())}
    if dtype == "f32":
        rows_err = err.reshape(-1, err.shape[-1]).max(axis=1)
        rows_ref = np.abs(ref).reshape(-1, ref.shape[-1]).max(axis=1)
        rel = rows_err / np.maximum(rows_ref, 1e-30)
        stats["max_rel"] = float(rel.max())
        assert rel.max() <= F32_REL, f"{what}: fp32 row relative error {rel.max():.3e} > {F32_REL}"
    else:
        assert err.max() <= BF_MAX_ABS, f"{what}: max abs error {err.max():.3e} > {BF_MAX_ABS}"
        assert err.mean() <= BF_MEAN_ABS, f"{what}: mean abs error {err.mean():.3e} > {BF_MEAN_ABS}"
    return stats


def oracle_caches_after_step(batch):
    """CPU copies of the pools after the step's copy-on-write and cache write."""
    kc = batch.k_cache.clone()
    vc = batch.v_cache.clone()
    oracle.copy_blocks(kc, vc, batch.cow_pairs)
    slots = oracle.slot_mapping(batch.block_tables, batch.new_seq_ids, batch.new_positions, batch.block_size)
    oracle.reshape_and_cache(batch.k_new, batch.v_new, slots, kc, vc, batch.block_size)
    return kc, vc, slots


def oracle_decode(batch, kc, vc, seqs=None):
    return oracle.decode(batch.q, kc, vc, batch.block_tables, batch.kv_lens, batch.scale, batch.block_size,
                         seqs=seqs)


def oracle_prefill(batch, kc, vc, seqs=None, rows=None):
    return oracle.prefill(batch.q, batch.cu_q_lens, batch.ctx_lens, kc, vc, batch.block_tables, batch.scale,
                          batch.block_size, seqs=seqs, rows=rows)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_step(batch, **replace):
    """Oracle output of a whole step on `batch` (copy-on-write copies, the
    cache write of the new tokens, then decode or chunked prefill), with any
    of the batch's fields (q, k_new, v_new, block_tables, ...) replaced by
    host arrays: what a replayed or pipelined step must produce."""
    if replace:
        batch = dataclasses.replace(batch, **replace)
    kc, vc, _ = oracle_caches_after_step(batch)
    if batch.is_decode:
        return oracle_decode(batch, kc, vc)
    return oracle_prefill(batch, kc, vc)


@functools.lru_cache(maxsize=2)
def full_config(name: str):
    """A named full-size workload, generated once per test session (the
    generator takes tens of seconds). Callers must not modify it."""
    from workloads import make_config
    return make_config(name)
