"""Chunked prefill (tcgen05 chunk tiles + decode rows) on the GPU against the
fp64 oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import assert_attention_close, full_config, oracle_caches_after_step, oracle_prefill, oracle_step, to_f64
from workloads import build_batch

pytestmark = pytest.mark.gpu


def run_step(lib, b):
    from paged_kv_cache_14_gb300.step import step_from_host
    st = step_from_host(b)
    out = st.run()
    status = lib.pa_get_status()
    assert status == 0, lib.pa_strerror(status)
    return st, to_f64(out)


CASES = [
    # dtype, B, Hq, Hkv, q_lens, ctx_lens
    ("f16", 32, 64, 8, [2, 17, 1, 100], [0, 5, 40, 63]),
    ("bf16", 16, 64, 8, [16, 33, 1, 129], [64, 0, 3, 200]),
    ("f16", 16, 8, 8, [130, 5], [1, 300]),            # group 1: 128 positions per tile
    ("bf16", 32, 16, 8, [64, 9], [65, 0]),           # group 2
    ("f16", 16, 32, 8, [31, 2, 1, 1], [15, 16, 0, 700]),  # group 4
    ("bf16", 32, 32, 2, [40, 3], [128, 1]),          # group 16: 8 positions per tile
    ("f16", 32, 64, 8, [512], [1000]),               # a long chunk over a long context
    ("bf16", 16, 64, 2, [9, 4, 13], [30, 0, 100]),   # group 32: 4 positions per Q tile
    ("f16", 16, 128, 1, [3, 2, 5, 1], [7, 40, 0, 9]),  # group 128: one position per Q tile
    # Groups that do not divide 128: a Q tile holds floor(128 / G) positions
    # x G heads and its last rows hold nothing.
    ("bf16", 16, 24, 8, [33, 1, 70, 130], [10, 50, 0, 3]),  # group 3: 42 positions, 126 rows
    ("f16", 32, 28, 4, [100, 9, 1, 37], [0, 200, 31, 64]),  # group 7: 18 positions, 126 rows
    ("bf16", 32, 96, 8, [20, 5, 23], [100, 7, 0]),          # group 12: 10 positions, 120 rows
    ("f16", 16, 80, 8, [13, 1, 25], [3, 9, 40]),            # group 10: 12 positions, 120 rows
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-B{c[1]}-G{c[2] // c[3]}-q{sum(c[4])}")
def test_prefill_small(lib, case):
    dtype, B, hq, hkv, qls, ctxs = case
    kv = [c + q for c, q in zip(ctxs, qls)]
    b = build_batch(name="pf", seed=CASES.index(case) + 50, dtype=dtype, block_size=B, num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=128, q_lens=qls, kv_lens=kv)
    _, out = run_step(lib, b)
    kc, vc, _ = oracle_caches_after_step(b)
    ref = oracle_prefill(b, kc, vc)
    assert_attention_close(out, ref, dtype, str(case))


CASES_D64 = [
    # dtype, B, Hq, Hkv, q_lens, ctx_lens: head_dim 64 (one 64-column half per tile row)
    ("f16", 16, 32, 8, [17, 1, 130, 40], [5, 60, 0, 300]),   # group 4
    ("bf16", 32, 24, 8, [64, 3, 1], [100, 0, 7]),           # group 3
    ("f16", 16, 8, 8, [129, 1], [10, 20]),                  # group 1
    ("bf16", 16, 64, 8, [512, 1], [600, 33]),               # group 8, a long chunk
]


@pytest.mark.parametrize("case", CASES_D64, ids=lambda c: f"{c[0]}-B{c[1]}-G{c[2] // c[3]}-q{sum(c[4])}-D64")
def test_prefill_head_dim_64(lib, case):
    dtype, B, hq, hkv, qls, ctxs = case
    kv = [c + q for c, q in zip(ctxs, qls)]
    b = build_batch(name="pf64", seed=CASES_D64.index(case) + 150, dtype=dtype, block_size=B, num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=64, q_lens=qls, kv_lens=kv)
    _, out = run_step(lib, b)
    kc, vc, _ = oracle_caches_after_step(b)
    assert_attention_close(out, oracle_prefill(b, kc, vc), dtype, f"{case} head_dim 64")


CASES_F32 = [
    # B, Hq, Hkv, D, q_lens, ctx_lens: fp32 I/O (chunk rows on the exact fp32 CUDA-core kernel)
    (16, 8, 2, 64, [17, 1, 40], [5, 30, 100]),
    (32, 32, 8, 128, [70, 1, 3, 129], [200, 10, 0, 31]),
    (16, 12, 4, 96, [9, 130, 1], [0, 33, 64]),   # group 3, head_dim 96
]


@pytest.mark.parametrize("case", CASES_F32, ids=lambda c: f"f32-B{c[0]}-G{c[1] // c[2]}-D{c[3]}-q{sum(c[4])}")
def test_prefill_fp32(lib, case):
    B, hq, hkv, D, qls, ctxs = case
    kv = [c + q for c, q in zip(ctxs, qls)]
    b = build_batch(name="pf32", seed=CASES_F32.index(case) + 170, dtype="f32", block_size=B, num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=D, q_lens=qls, kv_lens=kv)
    _, out = run_step(lib, b)
    kc, vc, _ = oracle_caches_after_step(b)
    assert_attention_close(out, oracle_prefill(b, kc, vc), "f32", f"{case} fp32")


def test_prefill_garbage_in_unused_slots(lib):
    qls, ctxs = [40, 7], [10, 90]
    b = build_batch(name="pfnan", seed=9, dtype="f16", block_size=32, num_q_heads=64, num_kv_heads=8,
                    head_dim=128, q_lens=qls, kv_lens=[c + q for c, q in zip(ctxs, qls)])
    kc, vc, _ = oracle_caches_after_step(b)
    ref = oracle_prefill(b, kc, vc)
    for i, L in enumerate(b.kv_lens):
        last = b.block_tables[i, (L - 1) // 32]
        b.k_cache[last, :, (L % 32) or 32:, :] = float("nan")
        b.v_cache[last, :, (L % 32) or 32:, :] = float("inf")
    _, out = run_step(lib, b)
    assert_attention_close(out, ref, "f16", "garbage slots")


def test_prefill_repeat_is_deterministic(lib):
    from paged_kv_cache_14_gb300.step import step_from_host
    b = build_batch(name="pfdet", seed=10, dtype="bf16", block_size=16, num_q_heads=64, num_kv_heads=8,
                    head_dim=128, q_lens=[300, 1, 77], kv_lens=[900, 50, 77])
    st = step_from_host(b)
    a = st.run().clone()
    c = st.run().clone()
    assert lib.pa_get_status() == 0
    assert torch.equal(a, c)
    assert_attention_close(to_f64(a), oracle_step(b), "bf16", "repeated prefill vs oracle")


@pytest.mark.slow
def test_mixed_prefill_config_sampled(lib):
    b = full_config("mixed_prefill_fp16")
    st, out = run_step(lib, b)
    assert np.all(np.isfinite(out))
    kr, vr, slots = oracle_caches_after_step(b)
    touched = torch.from_numpy(np.unique(slots // b.block_size))
    assert torch.equal(st.k_cache.cpu()[touched].view(torch.int16), kr[touched].view(torch.int16))
    rng = np.random.default_rng(5)
    dec = [int(i) for i in rng.choice(96, 6, replace=False)] + [int(np.argmax(b.kv_lens[:96]))]
    chunks = list(range(96, 104))
    rows = {}
    for i in chunks:
        ql = int(b.q_lens[i])
        rows[i] = sorted({0, 1, 15, 16, 127, 128, ql - 2, ql - 1} | set(rng.integers(0, ql, 4).tolist()))
    seqs = dec + chunks
    ref = oracle_prefill(b, kr, vr, seqs=seqs, rows=rows)
    cu = b.cu_q_lens
    sel = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in dec] + [cu[i] + np.array(rows[i]) for i in chunks])
    assert_attention_close(out[sel], ref[sel], "f16", "mixed_prefill_fp16")


def test_prefill_many_items_mixed_q_tiles(lib):
    # A work item is 256 packed rows in two Q tiles (16 positions each at
    # group 8). A 48-row chunk gives one item with both tiles and one whose
    # second tile is empty. With 24 such chunks x 8 KV heads (384 items)
    # every CTA runs several items of both kinds in turn, which exercises
    # the second tile's own barrier phases.
    rng = np.random.default_rng(404)
    qls = [48] * 24 + [17, 33]
    ctxs = rng.integers(0, 600, size=len(qls)).tolist()
    b = build_batch(name="pf_many", seed=404, dtype="bf16", block_size=16, num_q_heads=64, num_kv_heads=8,
                    head_dim=128, q_lens=qls, kv_lens=[c + q for c, q in zip(ctxs, qls)])
    _, out = run_step(lib, b)
    kc, vc, _ = oracle_caches_after_step(b)
    assert_attention_close(out, oracle_prefill(b, kc, vc), "bf16", "many items, mixed Q tiles")
