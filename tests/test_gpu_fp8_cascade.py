"""The e4m3 cache beyond plain decode, on the GPU: shared-prefix decode
(pa_decode_shared_prefix_fp8: the tcgen05 prefix pass with the codes widened
in shared memory, the e4m3 suffix decode, the merge) and chunked prefill
(pa_chunked_prefill_fp8: e4m3 decode rows beside the tcgen05 chunk kernel),
against the fp64 oracle on the dequantised pools (each stored value = e4m3
code x its (block, KV head) scale)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import oracle.fp8_kv as f8
from helpers import assert_attention_close, full_config, to_f64
from workloads import build_batch, e4m3_pool

pytestmark = pytest.mark.gpu


def _quantised(b):
    """e4m3 pools of a batch's 16-bit values (the oracle's whole-block quantiser)."""
    kc, ks = f8.quantize_fresh_blocks(b.k_cache.float().numpy())
    vc, vs = f8.quantize_fresh_blocks(b.v_cache.float().numpy())
    return kc, vc, np.stack([ks, vs], axis=-1).astype(np.float32)


def _random_codes(b, seed):
    """Codes uniform over every finite e4m3 value, scales over three binades."""
    kc, vc, sc = e4m3_pool(seed, b.num_blocks, b.num_kv_heads, b.block_size, b.head_dim)
    return kc.numpy(), vc.numpy(), sc.numpy()


def _dequantised(kc, vc, sc):
    return f8.dequantize(kc, sc[..., 0]), f8.dequantize(vc, sc[..., 1])


def _dev(pool):
    return tuple(torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in pool)


def _oracle_decode_rows(b, kc, vc, sc, block_tables=None, seqs=None):
    """Oracle decode, dequantising one sequence's blocks at a time (bounded
    memory at full size)."""
    bt = b.block_tables if block_tables is None else block_tables
    out = np.full((b.num_seqs, b.num_q_heads, b.head_dim), np.nan)
    for i in (range(b.num_seqs) if seqs is None else seqs):
        nb = -(-int(b.kv_lens[i]) // b.block_size)
        blocks = bt[i][:nb]
        kd = f8.dequantize(kc[blocks], sc[blocks, :, 0])
        vd = f8.dequantize(vc[blocks], sc[blocks, :, 1])
        tables = np.zeros_like(bt)
        tables[i, :nb] = np.arange(nb)
        out[i] = oracle.decode(b.q, kd, vd, tables, b.kv_lens, b.scale, b.block_size, seqs=[i])[i]
    return out


def _shared_fp8(lib, b, pool, prefix_lens=None, group_starts=None, partition=0):
    kc, vc, sc = _dev(pool)
    gs = torch.from_numpy(b.group_starts if group_starts is None else group_starts).cuda()
    pl = torch.from_numpy(b.prefix_lens if prefix_lens is None else prefix_lens).cuda()
    out = lib.pa_decode_shared_prefix_fp8(b.q.cuda(), kc, vc, sc, torch.from_numpy(b.block_tables).cuda(),
                                          torch.from_numpy(b.kv_lens).cuda(), b.max_seq_len, gs, pl, b.scale,
                                          partition_size=partition)
    return out


# ---------------------------------------------------------------------------
# Shared-prefix decode over the e4m3 cache
# ---------------------------------------------------------------------------

SP_CASES = [
    # dtype, B, Hq, Hkv, lens, group, prefix tokens
    ("bf16", 16, 64, 8, [5, 64, 64, 65, 200, 31, 1000, 129, 17, 80], 4, 64),
    ("f16", 32, 64, 8, [40, 300, 1000, 2000, 33, 64, 65, 999], 8, 256),
    ("bf16", 32, 32, 8, [300] * 20 + [20, 700], 20, 256),               # group 4: 32 members per tile
    ("bf16", 16, 64, 8, list(range(100, 100 + 37 * 45, 45)), 37, 512),  # 37 members: 3 tiles of 16
    ("f16", 16, 128, 8, [129, 400, 1024, 77], 2, 128),                  # group 16: 8 members per tile
    ("bf16", 16, 48, 8, list(range(90, 90 + 45 * 30, 30)), 45, 64),     # GQA group 6: 21 members per tile
]


@pytest.mark.parametrize("pool_kind", ["quantised", "random"])
@pytest.mark.parametrize("case", SP_CASES, ids=lambda c: f"{c[0]}-B{c[1]}-G{c[2] // c[3]}-grp{c[5]}")
@pytest.mark.parametrize("partition", [0, 64])
def test_shared_prefix_fp8_matches_oracle(lib, case, partition, pool_kind):
    dtype, B, hq, hkv, lens, grp, pref = case
    b = build_batch(name="fp8cascade", seed=SP_CASES.index(case) + 170, dtype=dtype, block_size=B, num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=128, q_lens=np.ones(len(lens), np.int32), kv_lens=lens,
                    share_group=grp, share_prefix_tokens=pref, cow_per_seq=True)
    assert (b.prefix_lens > 0).any()
    pool = _quantised(b) if pool_kind == "quantised" else _random_codes(b, 171)
    out = to_f64(_shared_fp8(lib, b, pool, partition=partition * (B // 16)))
    assert lib.pa_get_status() == 0
    assert_attention_close(out, _oracle_decode_rows(b, *pool), dtype, f"{case} vs oracle")


def test_shared_prefix_fp8_bad_hints_still_correct(lib):
    lens = [300, 300, 900, 64, 500, 33]
    b = build_batch(name="fp8cascade_bad", seed=181, dtype="bf16", block_size=16, num_q_heads=64, num_kv_heads=8,
                    head_dim=128, q_lens=np.ones(6, np.int32), kv_lens=lens, share_group=3,
                    share_prefix_tokens=256, cow_per_seq=True)
    pool = _quantised(b)
    ref = _oracle_decode_rows(b, *pool)
    pl = b.prefix_lens.copy()
    pl[0] = 288            # claims a private block as shared: rejected by the table check
    pl[1] = 17             # not a multiple of the block size: ignored
    pl[4] = lens[4]        # the whole sequence: ignored (the newest token is private)
    out = to_f64(_shared_fp8(lib, b, pool, prefix_lens=pl))
    assert lib.pa_get_status() == 0
    assert_attention_close(out, ref, "bf16", "bad hints")
    gs = b.group_starts.copy()
    gs[1], gs[2] = gs[2], gs[1]
    out = to_f64(_shared_fp8(lib, b, pool, group_starts=gs))
    assert lib.pa_get_status() == -1
    assert_attention_close(out, ref, "bf16", "malformed groups")


def test_shared_prefix_fp8_ignores_nan_codes_past_the_end(lib):
    """Codes past every sequence's end (and past a group's shared prefix
    inside its blocks) may be NaN patterns: they must not reach the output."""
    lens = [70, 75, 90, 300, 301, 305]
    b = build_batch(name="fp8cascade_nan", seed=182, dtype="f16", block_size=16, num_q_heads=32, num_kv_heads=4,
                    head_dim=128, q_lens=np.ones(6, np.int32), kv_lens=lens, share_group=3,
                    share_prefix_tokens=64, cow_per_seq=False)
    kc, vc, sc = _quantised(b)
    ref = _oracle_decode_rows(b, kc, vc, sc)
    kn, vn = kc.copy(), vc.copy()
    for i, L in enumerate(lens):
        last = b.block_tables[i][(L - 1) // 16]
        kn[last, :, L % 16 or 16:, :] = 0x7F
        vn[last, :, L % 16 or 16:, :] = 0xFF
    out = to_f64(_shared_fp8(lib, b, (kn, vn, sc)))
    assert lib.pa_get_status() == 0
    assert_attention_close(out, ref, "f16", "NaN codes past the end")


def _oracle_step_pools(b, pool):
    """The oracle's pools after the step: copy-on-write of codes and scales,
    then the quantising cache write of the new tokens."""
    ko, vo, so = (x.copy() for x in pool)
    f8.copy_blocks_fp8(ko, vo, so, b.cow_pairs)
    slots = oracle.slot_mapping(b.block_tables, b.new_seq_ids, b.new_positions, b.block_size)
    f8.reshape_and_cache_fp8(b.k_new.float().numpy(), b.v_new.float().numpy(), slots, ko, vo, so, b.block_size)
    return ko, vo, so


def test_step_fp8_shared_prefix_matches_oracle(lib):
    """The whole step on an e4m3 cache with prefix sharing: copy-on-write of
    codes and scales, slots, the quantising cache write, shared-prefix decode."""
    from paged_kv_cache_14_gb300.step import step_from_host
    lens = [5, 64, 300, 700, 1300, 31, 900, 17]
    b = build_batch(name="fp8cstep", seed=183, dtype="bf16", block_size=16, num_q_heads=64, num_kv_heads=8,
                    head_dim=128, q_lens=np.ones(8, np.int32), kv_lens=lens, share_group=4,
                    share_prefix_tokens=256, cow_per_seq=True)
    pool = _quantised(b)
    st = step_from_host(b, shared_prefix=True, fp8_pool=tuple(torch.from_numpy(x) for x in pool))
    out = to_f64(st.run())
    assert lib.pa_get_status() == 0
    ko, vo, so = _oracle_step_pools(b, pool)
    assert np.array_equal(st.k_cache.cpu().numpy(), ko) and np.array_equal(st.v_cache.cpu().numpy(), vo)
    assert_attention_close(out, _oracle_decode_rows(b, ko, vo, so), "bf16", "fp8 shared-prefix step")


@pytest.mark.slow
def test_llama3_70b_prefix_config_fp8_shared_prefix(lib):
    """The full 70B prefix-sharing batch on a synthetic e4m3 pool, through the
    step the bench times (copy-on-write, cache write, shared-prefix decode):
    every sequence against the oracle, and against plain e4m3 decode."""
    from paged_kv_cache_14_gb300.step import step_from_host
    b = full_config("llama3_70b_prefix_bf16")
    pool = tuple(x.numpy() for x in e4m3_pool(b.meta["seed"], b.num_blocks, b.num_kv_heads, b.block_size,
                                               b.head_dim))
    st = step_from_host(b, shared_prefix=True, fp8_pool=tuple(torch.from_numpy(x) for x in pool))
    out = to_f64(st.run())
    assert lib.pa_get_status() == 0
    plain = to_f64(lib.pa_decode_fp8(st.q, st.k_cache, st.v_cache, st.kv_scales, st.block_tables, st.kv_lens,
                                     st.max_seq_len, b.scale))
    assert lib.pa_get_status() == 0
    ko, vo, so = _oracle_step_pools(b, pool)
    assert_attention_close(out, _oracle_decode_rows(b, ko, vo, so), "bf16", "70B fp8 shared prefix, every sequence")
    assert_attention_close(out, plain, "bf16", "70B fp8 shared prefix vs plain e4m3 decode")


# ---------------------------------------------------------------------------
# Chunked prefill over the e4m3 cache
# ---------------------------------------------------------------------------

PF_CASES = [
    # dtype, B, Hq, Hkv, q_lens, ctx_lens
    ("f16", 32, 64, 8, [2, 17, 1, 100], [0, 5, 40, 63]),
    ("bf16", 16, 64, 8, [16, 33, 1, 129], [64, 0, 3, 200]),
    ("f16", 16, 8, 8, [130, 5], [1, 300]),               # group 1: 128 positions per tile
    ("bf16", 32, 16, 8, [64, 9], [65, 0]),              # group 2
    ("bf16", 32, 64, 8, [512, 1, 1], [1000, 700, 30]),  # a long chunk over a long context
    ("f16", 16, 128, 1, [3, 2, 5, 1], [7, 40, 0, 9]),   # group 128: one position per Q tile
    ("bf16", 16, 28, 4, [50, 1, 130], [20, 9, 0]),      # group 7: 18 positions, 126 rows per tile
]


def _prefill_fp8(lib, b, pool):
    kc, vc, sc = _dev(pool)
    out = lib.pa_chunked_prefill_fp8(b.q.cuda(), torch.from_numpy(b.cu_q_lens).cuda(), kc, vc, sc,
                                     torch.from_numpy(b.block_tables).cuda(), torch.from_numpy(b.ctx_lens).cuda(),
                                     b.max_q_len, b.max_seq_len, b.scale)
    st = lib.pa_get_status()
    assert st == 0, lib.pa_strerror(st)
    return to_f64(out)


@pytest.mark.parametrize("pool_kind", ["quantised", "random"])
@pytest.mark.parametrize("case", PF_CASES, ids=lambda c: f"{c[0]}-B{c[1]}-G{c[2] // c[3]}-q{sum(c[4])}")
def test_chunked_prefill_fp8_matches_oracle(lib, case, pool_kind):
    dtype, B, hq, hkv, qls, ctxs = case
    kv = [c + q for c, q in zip(ctxs, qls)]
    b = build_batch(name="pf8", seed=PF_CASES.index(case) + 190, dtype=dtype, block_size=B, num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=128, q_lens=qls, kv_lens=kv)
    pool = _quantised(b) if pool_kind == "quantised" else _random_codes(b, 191)
    out = _prefill_fp8(lib, b, pool)
    kd, vd = _dequantised(*pool)
    ref = oracle.prefill(b.q, b.cu_q_lens, b.ctx_lens, kd, vd, b.block_tables, b.scale, b.block_size)
    assert_attention_close(out, ref, dtype, f"{case} {pool_kind}")


@pytest.mark.slow
def test_mixed_prefill_config_fp8(lib):
    """The full mixed batch (96 decode rows, 8 chunks of 512) on a synthetic
    e4m3 pool through the step (quantising cache write of all 4192 new
    tokens, then pa_chunked_prefill_fp8): every decode row and sampled chunk
    rows against the oracle."""
    from paged_kv_cache_14_gb300.step import step_from_host
    b = full_config("mixed_prefill_fp16")
    pool = tuple(x.numpy() for x in e4m3_pool(b.meta["seed"], b.num_blocks, b.num_kv_heads, b.block_size,
                                               b.head_dim))
    st = step_from_host(b, fp8_pool=tuple(torch.from_numpy(x) for x in pool))
    out = to_f64(st.run())
    assert lib.pa_get_status() == 0
    ko, vo, so = _oracle_step_pools(b, pool)
    rng = np.random.default_rng(195)
    dec = list(range(96))
    chunks = list(range(96, 104))
    cu = b.cu_q_lens
    sel_rows = {}
    for i in chunks:
        ql = int(b.q_lens[i])
        sel_rows[i] = sorted({0, 1, 127, 128, ql - 1} | set(rng.integers(0, ql, 3).tolist()))
    got, want = [], []
    for i in dec + chunks:
        nb = -(-int(b.kv_lens[i]) // b.block_size)
        blocks = b.block_tables[i][:nb]
        kd = f8.dequantize(ko[blocks], so[blocks, :, 0])
        vd = f8.dequantize(vo[blocks], so[blocks, :, 1])
        tables = np.zeros_like(b.block_tables)
        tables[i, :nb] = np.arange(nb)
        rows = {i: sel_rows[i]} if i in sel_rows else None
        ref = oracle.prefill(b.q, b.cu_q_lens, b.ctx_lens, kd, vd, tables, b.scale, b.block_size, seqs=[i],
                             rows=rows)
        idx = np.arange(cu[i], cu[i + 1]) if rows is None else cu[i] + np.array(rows[i])
        got.append(out[idx])
        want.append(ref[idx])
    assert_attention_close(np.concatenate(got), np.concatenate(want), "f16", "mixed batch over e4m3")
