"""Paged decode attention on the GPU against the fp64 oracle."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from helpers import assert_attention_close, full_config, oracle_caches_after_step, oracle_decode, to_f64
from workloads import build_batch, make_config, random_lengths

pytestmark = pytest.mark.gpu


def run_decode(lib, b, partition_size=0):
    from paged_kv_cache_14_gb300.step import step_from_host
    st = step_from_host(b, partition_size=partition_size)
    out = st.run()
    status = lib.pa_get_status()
    assert status == 0, lib.pa_strerror(status)
    return st, to_f64(out)


SMALL = [
    # dtype, B, Hq, Hkv, D, lens
    ("f32", 16, 2, 1, 64, [1, 15, 16, 17, 33]),
    ("f32", 32, 8, 2, 128, [1, 31, 32, 33, 100]),
    ("f32", 16, 16, 1, 32, [5, 64, 65]),
    ("f32", 16, 4, 4, 256, [3, 47]),
    ("bf16", 16, 8, 1, 128, [1, 15, 16, 17, 33, 200]),
    ("bf16", 16, 32, 8, 128, [1, 2, 300, 1000]),
    ("bf16", 32, 64, 8, 128, [1, 31, 32, 33, 513, 1025]),
    ("bf16", 16, 4, 4, 64, [7, 16, 129]),
    ("f16", 16, 16, 2, 128, [1, 17, 160, 999]),
    ("f16", 32, 2, 2, 64, [1, 32, 64, 95]),
    ("bf16", 16, 32, 1, 128, [9, 70]),       # group 32: two row groups per KV head
    ("f16", 32, 40, 2, 128, [33, 77, 300]),  # group 20: ragged second row group
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"{c[0]}-B{c[1]}-Hq{c[2]}-Hkv{c[3]}-D{c[4]}")
@pytest.mark.parametrize("partition", [0, 1, 2, 7])
def test_decode_small(lib, case, partition):
    dtype, B, hq, hkv, D, lens = case
    b = build_batch(name="small", seed=SMALL.index(case), dtype=dtype, block_size=B, num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=D, q_lens=np.ones(len(lens), np.int32), kv_lens=lens)
    _, out = run_decode(lib, b, partition_size=partition * B)
    kc, vc, _ = oracle_caches_after_step(b)
    ref = oracle_decode(b, kc, vc)
    assert_attention_close(out, ref, dtype, f"{case} partition {partition}")


def test_decode_random_lengths_many_tiles(lib):
    lens = random_lengths(7, 48, 1, 3000)
    b = build_batch(name="ragged", seed=7, dtype="bf16", block_size=16, num_q_heads=32, num_kv_heads=8,
                    head_dim=128, q_lens=np.ones(48, np.int32), kv_lens=lens)
    for part in (0, 256, 16):
        _, out = run_decode(lib, b, part)
        kc, vc, _ = oracle_caches_after_step(b)
        assert_attention_close(out, oracle_decode(b, kc, vc), "bf16", f"partition {part}")


def test_decode_prefix_sharing_and_cow(lib):
    lens = [5, 64, 64, 65, 200, 31, 1, 129]
    b = build_batch(name="share", seed=12, dtype="bf16", block_size=16, num_q_heads=16, num_kv_heads=2,
                    head_dim=128, q_lens=np.ones(8, np.int32), kv_lens=lens, share_group=4,
                    share_prefix_tokens=64, cow_per_seq=True)
    st, out = run_decode(lib, b)
    kc, vc, _ = oracle_caches_after_step(b)
    assert_attention_close(out, oracle_decode(b, kc, vc), "bf16", "shared prefix")
    assert torch.equal(st.k_cache.cpu().view(torch.int16), kc.view(torch.int16))


def test_decode_garbage_in_unused_slots(lib):
    """Slots past a sequence's end may hold any bits (NaN, Inf); they must not
    leak into the output."""
    b = build_batch(name="nan", seed=3, dtype="bf16", block_size=16, num_q_heads=8, num_kv_heads=2,
                    head_dim=128, q_lens=np.ones(4, np.int32), kv_lens=[1, 17, 31, 40])
    kc, vc, _ = oracle_caches_after_step(b)
    ref = oracle_decode(b, kc, vc)
    for i, L in enumerate(b.kv_lens):
        last = b.block_tables[i, (L - 1) // 16]
        b.k_cache[last, :, (L % 16) or 16:, :] = float("nan")
        b.v_cache[last, :, (L % 16) or 16:, :] = float("inf")
    _, out = run_decode(lib, b)
    assert_attention_close(out, ref, "bf16", "garbage slots")


def test_decode_device_errors_are_reported(lib):
    b = build_batch(name="err", seed=4, dtype="bf16", block_size=16, num_q_heads=8, num_kv_heads=2,
                    head_dim=128, q_lens=np.ones(3, np.int32), kv_lens=[10, 40, 70])
    dev = "cuda"
    q, kc, vc = b.q.to(dev), b.k_cache.to(dev), b.v_cache.to(dev)
    bt = torch.from_numpy(b.block_tables).to(dev)
    sl = torch.from_numpy(b.kv_lens).to(dev)
    # A sequence longer than the host bound.
    lib.pa_decode(q, kc, vc, bt, sl, 40, b.scale)
    assert lib.pa_get_status() == -8
    # A block id outside the pool.
    bt_bad = bt.clone()
    bt_bad[1, 0] = b.num_blocks + 5
    lib.pa_decode(q, kc, vc, bt_bad, sl, 70, b.scale)
    assert lib.pa_get_status() == -7
    # Zero-length sequence.
    sl0 = sl.clone()
    sl0[0] = 0
    out = lib.pa_decode(q, kc, vc, bt, sl0, 70, b.scale)
    assert lib.pa_get_status() == -8
    assert out[0].float().abs().sum().item() == 0.0
    assert lib.pa_get_status() == 0


def test_tiny_fp32_config(lib):
    b = make_config("tiny_fp32")
    _, out = run_decode(lib, b)
    kc, vc, _ = oracle_caches_after_step(b)
    stats = assert_attention_close(out, oracle_decode(b, kc, vc), "f32", "tiny_fp32")
    assert stats["max_rel"] < 1e-5


def _full_config(lib, name):
    """The named workload at full size, in the launch configuration the bench
    times: the cache blocks the step touched equal the oracle's bit for bit,
    and EVERY sequence's output is compared with the oracle."""
    b = full_config(name)
    st, out = run_decode(lib, b)
    assert np.all(np.isfinite(out))
    kc = st.k_cache.cpu()
    vc = st.v_cache.cpu()
    kr, vr, slots = oracle_caches_after_step(b)
    touched = np.unique(np.concatenate([b.cow_pairs[:, 1] if len(b.cow_pairs) else np.zeros(0, np.int64),
                                        slots // b.block_size]))
    tt = torch.from_numpy(touched)
    assert torch.equal(kc[tt].view(torch.int16), kr[tt].view(torch.int16))
    assert torch.equal(vc[tt].view(torch.int16), vr[tt].view(torch.int16))
    ref = oracle_decode(b, kr, vr)
    stats = assert_attention_close(out, ref, b.dtype, name)
    return b, st, out, stats


@pytest.mark.slow
def test_llama3_8b_config_all_sequences(lib):
    _full_config(lib, "llama3_8b_bf16")


@pytest.mark.slow
def test_llama3_70b_prefix_config_all_sequences(lib):
    b, st, out, _ = _full_config(lib, "llama3_70b_prefix_bf16")
    # Invariant at full size: the copy-on-write copies change nothing that a
    # sequence reads except the new token's slot. Decoding again on the
    # pre-copy tables (shared blocks) gives the same result for every
    # sequence whose new token is not in its copied block.
    pre = b.block_tables.copy()
    for i, (src, dst) in enumerate(b.cow_pairs):
        pre[i][pre[i] == dst] = src
    new_in_copy = np.array([b.block_tables[i][(b.kv_lens[i] - 1) // 16] == b.cow_pairs[i][1]
                            for i in range(b.num_seqs)])
    out2 = lib.pa_decode(st.q, st.k_cache, st.v_cache, torch.from_numpy(pre).cuda(), st.kv_lens, st.max_seq_len,
                         b.scale)
    assert lib.pa_get_status() == 0
    keep = ~new_in_copy
    assert torch.equal(out2[torch.from_numpy(keep).cuda()], st.out[torch.from_numpy(keep).cuda()])


@pytest.mark.slow
def test_long_splitkv_config_all_sequences(lib):
    b, st, out, _ = _full_config(lib, "long_splitkv_bf16")
    part = lib.pa_decode_partition_size(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.block_size, b.max_seq_len, 0)
    assert math.ceil(b.max_seq_len / part) > 1  # the split-KV path ran
