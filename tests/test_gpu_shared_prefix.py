"""Shared-prefix (cascade) decode on the GPU: the same attention as plain
decode, computed as one tcgen05 pass over each group's shared blocks plus a
split-KV pass over every member's private suffix, merged with log-sum-exp
weights. Checked against the fp64 oracle and against pa_decode."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

from helpers import assert_attention_close, full_config, oracle_caches_after_step, oracle_decode, to_f64
from workloads import build_batch

pytestmark = pytest.mark.gpu


def _device_step(lib, b):
    from paged_kv_cache_14_gb300.step import step_from_host
    st = step_from_host(b)
    st.run()  # copy-on-write, slots, cache write, plain decode
    assert lib.pa_get_status() == 0
    return st


def _shared(lib, st, b, group_starts=None, prefix_lens=None, partition=0):
    gs = torch.from_numpy(b.group_starts if group_starts is None else group_starts).cuda()
    pl = torch.from_numpy(b.prefix_lens if prefix_lens is None else prefix_lens).cuda()
    out = lib.pa_decode_shared_prefix(st.q, st.k_cache, st.v_cache, st.block_tables, st.kv_lens, st.max_seq_len,
                                      gs, pl, b.scale, partition_size=partition)
    return out


CASES = [
    # dtype, B, Hq, Hkv, lens, group, prefix tokens
    ("bf16", 16, 64, 8, [5, 64, 64, 65, 200, 31, 1000, 129, 17, 80], 4, 64),
    ("f16", 32, 64, 8, [40, 300, 1000, 2000, 33, 64, 65, 999], 8, 256),
    ("bf16", 16, 32, 8, [300] * 20 + [20, 700], 20, 256),      # group 4: 20 members > 32/tile? no: 32/tile
    ("bf16", 16, 64, 8, list(range(100, 100 + 37 * 45, 45)), 37, 512),  # 37 members: 3 tiles of 16
    ("f16", 16, 128, 8, [129, 400, 1024, 77], 2, 128),        # group 16: 8 members per tile
    ("bf16", 16, 48, 8, list(range(90, 90 + 45 * 30, 30)), 45, 64),  # GQA group 6: 21 members per tile
    ("f16", 32, 96, 8, [300, 40, 900, 64, 65, 500, 33, 128] * 3, 12, 64),  # GQA group 12: 10 per tile
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-B{c[1]}-G{c[2] // c[3]}-grp{c[5]}")
@pytest.mark.parametrize("partition", [0, 64])
def test_shared_prefix_matches_oracle_and_decode(lib, case, partition):
    dtype, B, hq, hkv, lens, grp, pref = case
    b = build_batch(name="cascade", seed=CASES.index(case) + 70, dtype=dtype, block_size=B, num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=128, q_lens=np.ones(len(lens), np.int32), kv_lens=lens,
                    share_group=grp, share_prefix_tokens=pref, cow_per_seq=True)
    assert (b.prefix_lens > 0).any()
    st = _device_step(lib, b)
    ref_plain = to_f64(st.out)
    out = to_f64(_shared(lib, st, b, partition=partition * (B // 16)))
    assert lib.pa_get_status() == 0
    kc, vc, _ = oracle_caches_after_step(b)
    assert_attention_close(out, oracle_decode(b, kc, vc), dtype, f"{case} vs oracle")
    assert_attention_close(out, ref_plain, dtype, f"{case} vs pa_decode")


@pytest.mark.parametrize("case", [("bf16", 16, 32, 8, [5, 64, 300, 65, 700, 31, 1000, 129], 4, 64),
                                  ("f16", 32, 24, 8, [200, 40, 900, 64, 65, 500] * 2, 6, 128)],
                         ids=["bf16-B16-G4-D64", "f16-B32-G3-D64"])
def test_shared_prefix_head_dim_64(lib, case):
    dtype, B, hq, hkv, lens, grp, pref = case
    b = build_batch(name="cascade64", seed=len(lens) + 160, dtype=dtype, block_size=B, num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=64, q_lens=np.ones(len(lens), np.int32), kv_lens=lens,
                    share_group=grp, share_prefix_tokens=pref, cow_per_seq=True)
    assert (b.prefix_lens > 0).any()
    st = _device_step(lib, b)
    out = to_f64(_shared(lib, st, b))
    assert lib.pa_get_status() == 0
    kc, vc, _ = oracle_caches_after_step(b)
    assert_attention_close(out, oracle_decode(b, kc, vc), dtype, f"{case} vs oracle")
    assert_attention_close(out, to_f64(st.out), dtype, f"{case} vs pa_decode")


def test_shared_prefix_bad_hints_still_correct(lib):
    lens = [300, 300, 900, 64, 500, 33]
    b = build_batch(name="cascade_bad", seed=81, dtype="bf16", block_size=16, num_q_heads=64, num_kv_heads=8,
                    head_dim=128, q_lens=np.ones(6, np.int32), kv_lens=lens, share_group=3,
                    share_prefix_tokens=256, cow_per_seq=True)
    st = _device_step(lib, b)
    kc, vc, _ = oracle_caches_after_step(b)
    ref = oracle_decode(b, kc, vc)
    pl = b.prefix_lens.copy()
    pl[0] = 288            # claims a private block as shared: rejected by the table check
    pl[1] = 17             # not a multiple of the block size: ignored
    pl[4] = lens[4]        # the whole sequence: ignored (the newest token is private)
    out = to_f64(_shared(lib, st, b, prefix_lens=pl))
    assert lib.pa_get_status() == 0
    assert_attention_close(out, ref, "bf16", "bad hints")
    # Malformed groups: every hint is dropped and the call records PA_ERR_ARG.
    gs = b.group_starts.copy()
    gs[1], gs[2] = gs[2], gs[1]
    out = to_f64(_shared(lib, st, b, group_starts=gs))
    assert lib.pa_get_status() == -1
    assert_attention_close(out, ref, "bf16", "malformed groups")


@pytest.mark.slow
def test_llama3_70b_prefix_config_shared_prefix(lib):
    """The full 70B prefix-sharing batch through the one-call shared-prefix
    step, the launch configuration the bench times: the blocks the step
    touched equal the oracle's bit for bit and every sequence's output is
    compared with the oracle (and with plain decode)."""
    from paged_kv_cache_14_gb300.step import step_from_host
    b = full_config("llama3_70b_prefix_bf16")
    st = step_from_host(b, shared_prefix=True)
    st.run()
    assert lib.pa_get_status() == 0
    out = to_f64(st.out)
    kr, vr, slots = oracle_caches_after_step(b)
    touched = torch.from_numpy(np.unique(np.concatenate([b.cow_pairs[:, 1], slots // b.block_size])))
    assert torch.equal(st.k_cache.cpu()[touched].view(torch.int16), kr[touched].view(torch.int16))
    assert torch.equal(st.v_cache.cpu()[touched].view(torch.int16), vr[touched].view(torch.int16))
    assert_attention_close(out, oracle_decode(b, kr, vr), "bf16", "shared-prefix step vs oracle, every sequence")
    plain = lib.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.kv_lens, st.max_seq_len, b.scale)
    assert lib.pa_get_status() == 0
    assert_attention_close(out, to_f64(plain), "bf16", "shared-prefix vs pa_decode, full size")


def _oracle_rows(b, block_tables, pick):
    """Oracle rows of the sequences in `pick` after the batch's step, on the
    given (possibly edited) block tables."""
    kr, vr, _ = oracle_caches_after_step(b)
    return oracle.decode(b.q, kr, vr, block_tables, b.kv_lens, b.scale, b.block_size, seqs=pick)


@pytest.mark.parametrize("n", [5000, 17000], ids=["staged_large", "unstaged"])
def test_shared_prefix_many_sequences(lib, n):
    # The preparation kernel keeps its per-sequence state in shared memory up
    # to a size cap (5000 sequences: above the 48 KB default, so the opt-in
    # size is used) and works on the workspace arrays beyond it (17000).
    rng = np.random.default_rng(n)
    lens = rng.integers(33, 97, size=n).astype(np.int32)
    b = build_batch(name="cascade_many", seed=91, dtype="bf16", block_size=16, num_q_heads=8, num_kv_heads=1,
                    head_dim=128, q_lens=np.ones(n, np.int32), kv_lens=lens, share_group=8,
                    share_prefix_tokens=32, cow_per_seq=False)
    assert (b.prefix_lens > 0).all()
    st = _device_step(lib, b)
    plain = to_f64(st.out)
    out = to_f64(_shared(lib, st, b))
    assert lib.pa_get_status() == 0
    assert_attention_close(out, plain, "bf16", f"{n} sequences: shared-prefix vs pa_decode")
    # Against the oracle: every member of the first, a middle and the last
    # groups, plus 400 sequences drawn at random.
    gs = b.group_starts
    mid = len(gs) // 2
    pick = set(range(gs[0], gs[1])) | set(range(gs[mid], gs[mid + 1])) | set(range(gs[-2], gs[-1]))
    pick |= set(np.random.default_rng(n + 1).choice(n, 400, replace=False).tolist())
    pick = sorted(int(i) for i in pick)
    ref = _oracle_rows(b, b.block_tables, pick)
    assert_attention_close(out[pick], ref[pick], "bf16", f"{n} sequences: shared-prefix vs oracle")


def test_shared_prefix_many_groups_mixed_q_tiles(lib):
    # Groups of 20 members (at group 8: two Q tiles, the second with 4
    # members) alternate with groups of 10 (one Q tile). 48 groups x 8 KV
    # heads give 384 prefix-pass items, more than that pass has CTAs, so
    # each CTA runs both kinds in turn.
    sizes = [20, 10] * 24
    lens, starts = [], [0]
    rng = np.random.default_rng(505)
    for g in sizes:
        lens += rng.integers(130, 400, size=g).tolist()
        starts.append(starts[-1] + g)
    b = build_batch(name="cascade_mixed", seed=505, dtype="bf16", block_size=16, num_q_heads=64, num_kv_heads=8,
                    head_dim=128, q_lens=np.ones(len(lens), np.int32), kv_lens=lens, share_group=1,
                    share_prefix_tokens=0, cow_per_seq=False)
    st = _device_step(lib, b)
    gs = np.array(starts, np.int32)
    pl = np.full(len(lens), 128, np.int32)  # hint: the first 8 blocks are shared
    # Make every group share its first 8 blocks: point each member's first
    # table entries at the group's first member's blocks, then compare
    # against plain decode on the same tables.
    bt = st.block_tables.clone()
    for gi in range(len(sizes)):
        s0, s1 = starts[gi], starts[gi + 1]
        bt[s0 + 1:s1, :8] = bt[s0, :8]
    st.block_tables.copy_(bt)
    plain = to_f64(lib.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.kv_lens, st.max_seq_len, b.scale))
    out = to_f64(_shared(lib, st, b, group_starts=gs, prefix_lens=pl))
    assert lib.pa_get_status() == 0
    assert_attention_close(out, plain, "bf16", "mixed group sizes: shared-prefix vs pa_decode")
    ref = _oracle_rows(b, bt.cpu().numpy(), list(range(len(lens))))
    assert_attention_close(out, ref, "bf16", "mixed group sizes: shared-prefix vs oracle")


@pytest.mark.parametrize("case", [CASES[0], CASES[3]], ids=["grp4", "grp37"])
def test_step_in_one_call_matches_separate_calls(lib, case):
    # pa_decode_step_shared_prefix runs the prefix check beside the
    # copy-on-write copies, slots and cache write; the result must be the
    # four separate calls' to the bit: output, both pools and the slots.
    from paged_kv_cache_14_gb300.step import step_from_host
    dtype, B, hq, hkv, lens, grp, pref = case
    b = build_batch(name="cascade_step", seed=606, dtype=dtype, block_size=B, num_q_heads=hq, num_kv_heads=hkv,
                    head_dim=128, q_lens=np.ones(len(lens), np.int32), kv_lens=lens, share_group=grp,
                    share_prefix_tokens=pref, cow_per_seq=True)
    assert len(b.cow_pairs) > 0
    sep = step_from_host(b, shared_prefix=True)
    sep.prepare()
    sep.attend()
    one = step_from_host(b, shared_prefix=True)
    one.run()
    torch.cuda.synchronize()
    assert lib.pa_get_status() == 0
    assert torch.equal(one.slot_mapping, sep.slot_mapping)
    assert torch.equal(one.k_cache, sep.k_cache) and torch.equal(one.v_cache, sep.v_cache)
    assert torch.equal(one.out, sep.out)
    kc, vc, _ = oracle_caches_after_step(b)
    assert_attention_close(to_f64(one.out), oracle_decode(b, kc, vc), dtype, "one-call step vs oracle")


def test_step_in_one_call_rejects_before_launching(lib):
    # A bad copy-on-write pair is caught on the host: nothing is launched,
    # so the pools and the output are untouched.
    from paged_kv_cache_14_gb300.step import step_from_host
    dtype, B, hq, hkv, lens, grp, pref = CASES[0]
    b = build_batch(name="cascade_step_bad", seed=607, dtype=dtype, block_size=B, num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=128, q_lens=np.ones(len(lens), np.int32), kv_lens=lens,
                    share_group=grp, share_prefix_tokens=pref, cow_per_seq=True)
    st = step_from_host(b, shared_prefix=True)
    k0, v0 = st.k_cache.clone(), st.v_cache.clone()
    st.out.fill_(7)
    bad = np.asarray(st.cow_pairs).copy()
    bad[0, 1] = st.k_cache.shape[0]  # destination out of range
    with pytest.raises(lib.PagedAttnError):
        lib.pa_decode_step_shared_prefix(bad, st.new_seq_ids, st.new_positions, st.k_new, st.v_new,
                                         st.slot_mapping, st.q, st.k_cache, st.v_cache, st.block_tables,
                                         st.kv_lens, st.max_seq_len, st.group_starts, st.prefix_lens, b.scale,
                                         out=st.out, workspace=st.workspace)
    torch.cuda.synchronize()
    assert torch.equal(st.k_cache, k0) and torch.equal(st.v_cache, v0)
    assert bool((st.out == 7).all())


def test_shared_prefix_long_prefix_mismatch_past_64_blocks(lib):
    # Hints of 96 shared blocks: the table check compares 64 entries per pass,
    # so a member whose block 80 differs from the reference's must still be
    # caught (its hint dropped). Compared against plain decode on the same
    # tables.
    lens = [1700, 1800, 1650, 2000, 1900, 1750]
    b = build_batch(name="cascade_long", seed=808, dtype="bf16", block_size=16, num_q_heads=64, num_kv_heads=8,
                    head_dim=128, q_lens=np.ones(len(lens), np.int32), kv_lens=lens, share_group=3,
                    share_prefix_tokens=1536, cow_per_seq=False)
    st = _device_step(lib, b)
    bt = st.block_tables.clone()
    bt[1, 80] = bt[1, 100]  # member 1 of group 0 now reads a private block at position 80
    bt[4, 95] = bt[4, 99]   # member 1 of group 1: the last shared entry
    st.block_tables.copy_(bt)
    plain = to_f64(lib.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.kv_lens, st.max_seq_len,
                                 b.scale))
    out = to_f64(_shared(lib, st, b))
    assert lib.pa_get_status() == 0
    assert_attention_close(out, plain, "bf16", "mismatch past the first 64 shared blocks")
    ref = _oracle_rows(b, bt.cpu().numpy(), list(range(len(lens))))
    assert_attention_close(out, ref, "bf16", "mismatch past the first 64 shared blocks vs oracle")
