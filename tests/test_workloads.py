"""The seeded workload generator (shared by the CUDA path's tests and bench and
by the oracle) draws structure only; these CPU tests check that structure:
same seed, same batch; every table entry a valid block; sharing only where a
group shares a prefix; copy-on-write pairs that repoint exactly one shared
block per sequence to a fresh block; new tokens at the last positions; the
named configurations' documented shapes; e4m3 pools without NaN codes."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from workloads import CONFIG_NAMES, build_batch, e4m3_pool, make_config


def _batch(seed=3, **o):
    a = dict(name="wl", seed=seed, dtype="bf16", block_size=16, num_q_heads=8, num_kv_heads=2, head_dim=64,
             q_lens=np.ones(10, np.int32), kv_lens=[5, 16, 17, 64, 65, 130, 200, 31, 48, 300], share_group=4,
             share_prefix_tokens=32, cow_per_seq=True)
    a.update(o)
    return build_batch(**a)


def _live_entries(b):
    for i in range(b.num_seqs):
        nb = -(-int(b.kv_lens[i]) // b.block_size)
        yield i, b.block_tables[i, :nb]


def test_same_seed_same_batch_and_new_seed_differs():
    a, b, c = _batch(), _batch(), _batch(seed=4)
    assert np.array_equal(a.block_tables, b.block_tables) and np.array_equal(a.cow_pairs, b.cow_pairs)
    for f in ("q", "k_cache", "v_cache", "k_new", "v_new"):
        assert torch.equal(getattr(a, f), getattr(b, f))
    assert not torch.equal(a.q, c.q)
    assert not np.array_equal(a.block_tables, c.block_tables)


def test_table_entries_are_valid_and_only_prefix_blocks_are_shared():
    b = _batch()
    owners = {}
    for i, row in _live_entries(b):
        assert np.all((row >= 0) & (row < b.num_blocks))
        for j, blk in enumerate(row.tolist()):
            owners.setdefault(blk, []).append((i, j))
    pb = 32 // b.block_size
    for blk, users in owners.items():
        if len(users) == 1:
            continue
        # A block used by several sequences is one shared prefix block of one
        # group, at the same logical index in every user.
        groups = {np.searchsorted(b.group_starts, i, side="right") - 1 for i, _ in users}
        idx = {j for _, j in users}
        assert len(groups) == 1 and len(idx) == 1 and next(iter(idx)) < pb, (blk, users)


def test_copy_on_write_pairs_repoint_the_last_shared_block():
    b = _batch()
    assert b.cow_pairs.shape == (b.num_seqs, 2)
    dsts = b.cow_pairs[:, 1]
    assert len(set(dsts.tolist())) == len(dsts)  # every destination fresh and distinct
    live = {int(x) for _, row in _live_entries(b) for x in row}
    assert not set(b.cow_pairs[:, 0].tolist()) & set(dsts.tolist())
    for i in range(b.num_seqs):
        nb = -(-int(b.kv_lens[i]) // b.block_size)
        last_shared = min(nb, 32 // b.block_size) - 1
        src, dst = (int(x) for x in b.cow_pairs[i])
        assert b.block_tables[i, last_shared] == dst  # the table already points at the copy
        assert dst in live
        g = np.searchsorted(b.group_starts, i, side="right") - 1
        # The source is the group's shared block at that index, which the
        # group's other members that cover it still use.
        for k in range(b.group_starts[g], b.group_starts[g + 1]):
            nbk = -(-int(b.kv_lens[k]) // b.block_size)
            if k != i and min(nbk, 32 // b.block_size) - 1 > last_shared:
                assert b.block_tables[k, last_shared] == src
    # After the copy every member still shares its prefix_lens tokens with
    # the group member that keeps the longest prefix (the hint is valid by
    # construction, as the shared-prefix decode requires).
    for g in range(len(b.group_starts) - 1):
        s0, s1 = int(b.group_starts[g]), int(b.group_starts[g + 1])
        ref = s0 + int(np.argmax(b.prefix_lens[s0:s1]))
        for i in range(s0, s1):
            k = int(b.prefix_lens[i]) // b.block_size
            assert b.prefix_lens[i] % b.block_size == 0 and (k == 0 or b.prefix_lens[i] < b.kv_lens[i])
            assert np.array_equal(b.block_tables[i, :k], b.block_tables[ref, :k])


def test_new_tokens_are_the_last_positions():
    qls = [1, 3, 1, 17]
    b = build_batch(name="wl_new", seed=9, dtype="f16", block_size=32, num_q_heads=4, num_kv_heads=4, head_dim=64,
                    q_lens=qls, kv_lens=[10, 40, 33, 100])
    assert b.new_seq_ids.tolist() == [0, 1, 1, 1, 2] + [3] * 17
    want = [9, 37, 38, 39, 32] + list(range(83, 100))
    assert b.new_positions.tolist() == want
    assert b.k_new.shape == (sum(qls), 4, 64) and b.q.shape == (sum(qls), 4, 64)
    assert b.cu_q_lens.tolist() == [0, 1, 4, 5, 22]
    assert b.ctx_lens.tolist() == [9, 37, 32, 83]


@pytest.mark.parametrize("name", CONFIG_NAMES)
def test_named_configs_have_their_documented_shapes(name):
    b = make_config(name, with_values=False)
    shapes = {
        "tiny_fp32": (4, 2, 1, 64, 16, "f32"),
        "llama3_8b_bf16": (64, 32, 8, 128, 16, "bf16"),
        "llama3_70b_prefix_bf16": (256, 64, 8, 128, 16, "bf16"),
        "long_splitkv_bf16": (8, 64, 8, 128, 16, "bf16"),
        "mixed_prefill_fp16": (104, 64, 8, 128, 32, "f16"),
    }
    n, hq, hkv, d, bs, dt = shapes[name]
    assert (b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size, b.dtype) == (n, hq, hkv, d, bs, dt)
    assert b.num_blocks >= b.meta["need_blocks"]
    for _, row in _live_entries(b):
        assert np.all((row >= 0) & (row < b.num_blocks))
    if name == "llama3_70b_prefix_bf16":
        assert b.cow_pairs.shape == (256, 2)
        assert np.all(np.diff(b.group_starts) == 16)
        # 1024 shared tokens (64 blocks), fewer for shorter sequences; the last
        # shared block of each sequence is copied on write.
        covered = np.minimum(-(-b.kv_lens // 16), 64)
        assert np.array_equal(b.prefix_lens, (covered - 1) * 16)
    if name == "long_splitkv_bf16":
        assert b.kv_lens.min() >= 32768 and b.kv_lens.max() <= 131072
    if name == "mixed_prefill_fp16":
        assert int((b.q_lens == 1).sum()) == 96 and sorted(set(b.q_lens[b.q_lens > 1].tolist())) == [512]


def test_e4m3_pool_has_no_nan_codes_and_scales_in_range():
    k, v, sc = e4m3_pool(5, 64, 2, 16, 128, log2_scale_range=(-9.0, -8.0))
    for c in (k, v):
        assert c.dtype == torch.uint8 and c.shape == (64, 2, 16, 128)
        vals = set(torch.unique(c).tolist())
        assert 0x7F not in vals and 0xFF not in vals
        assert len(vals) > 240  # close to uniform over the 254 finite codes
    assert sc.shape == (64, 2, 2) and sc.dtype == torch.float32
    assert float(sc.min()) >= 2.0 ** -9 and float(sc.max()) <= 2.0 ** -8
    k2, _, sc2 = e4m3_pool(5, 64, 2, 16, 128, log2_scale_range=(-9.0, -8.0))
    assert torch.equal(k, k2) and torch.equal(sc, sc2)
