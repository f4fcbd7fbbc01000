"""pa_decode_step: a decode step (copy-on-write copies, slots, cache write,
decode) in one call, whose decode plan runs beside the cache side. It must
give the four separate calls' results to the bit, and reject bad input
before launching anything."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import assert_attention_close, full_config, oracle_caches_after_step, oracle_decode, oracle_step, to_f64
from workloads import build_batch

pytestmark = pytest.mark.gpu

CASES = [
    # dtype, B, Hq, Hkv, D, lens, share group, shared tokens (copy-on-write when > 0)
    ("bf16", 16, 64, 8, 128, [5, 64, 300, 700, 1300, 2100, 31, 900], 4, 256),
    ("f16", 32, 32, 8, 128, [40, 3000, 65, 999, 2], 0, 0),
    ("bf16", 16, 16, 2, 64, [17, 160, 4100, 33], 2, 64),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-B{c[1]}-D{c[4]}-cow{c[7] > 0}")
def test_decode_step_in_one_call_matches_separate_calls(lib, case):
    from paged_kv_cache_14_gb300.step import step_from_host
    dtype, B, hq, hkv, D, lens, grp, pref = case
    b = build_batch(name="step_one", seed=CASES.index(case) + 700, dtype=dtype, block_size=B, num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=D, q_lens=np.ones(len(lens), np.int32), kv_lens=lens,
                    share_group=grp, share_prefix_tokens=pref, cow_per_seq=pref > 0)
    sep = step_from_host(b)
    sep.prepare()
    sep.attend()
    one = step_from_host(b)
    one.run()
    torch.cuda.synchronize()
    assert lib.pa_get_status() == 0
    assert torch.equal(one.slot_mapping, sep.slot_mapping)
    assert torch.equal(one.k_cache, sep.k_cache) and torch.equal(one.v_cache, sep.v_cache)
    assert torch.equal(one.out, sep.out)
    kc, vc, _ = oracle_caches_after_step(b)
    assert_attention_close(to_f64(one.out), oracle_decode(b, kc, vc), dtype, "one-call decode step vs oracle")


def test_decode_step_rejects_before_launching(lib):
    from paged_kv_cache_14_gb300.step import step_from_host
    dtype, B, hq, hkv, D, lens, grp, pref = CASES[0]
    b = build_batch(name="step_bad", seed=710, dtype=dtype, block_size=B, num_q_heads=hq, num_kv_heads=hkv,
                    head_dim=D, q_lens=np.ones(len(lens), np.int32), kv_lens=lens, share_group=grp,
                    share_prefix_tokens=pref, cow_per_seq=True)
    st = step_from_host(b)
    k0, v0 = st.k_cache.clone(), st.v_cache.clone()
    st.out.fill_(3)
    bad = np.asarray(st.cow_pairs).copy()
    bad[1, 1] = bad[0, 1]  # a repeated destination
    with pytest.raises(lib.PagedAttnError):
        lib.pa_decode_step(bad, st.new_seq_ids, st.new_positions, st.k_new, st.v_new, st.slot_mapping, st.q,
                           st.k_cache, st.v_cache, st.block_tables, st.kv_lens, st.max_seq_len, b.scale,
                           out=st.out, workspace=st.workspace)
    torch.cuda.synchronize()
    assert torch.equal(st.k_cache, k0) and torch.equal(st.v_cache, v0)
    assert bool((st.out == 3).all())


def test_decode_step_8b_config_matches_separate_calls(lib):
    from paged_kv_cache_14_gb300.step import step_from_host
    b = full_config("llama3_8b_bf16")
    sep = step_from_host(b)
    sep.prepare()
    sep.attend()
    one = step_from_host(b)
    one.run()
    torch.cuda.synchronize()
    assert lib.pa_get_status() == 0
    assert torch.equal(one.out, sep.out)
    assert torch.equal(one.k_cache, sep.k_cache) and torch.equal(one.v_cache, sep.v_cache)
    assert_attention_close(to_f64(one.out), oracle_step(b), "bf16", "8B one-call step vs oracle, every sequence")


def test_one_call_steps_with_empty_parts(lib):
    # No copy-on-write pairs and no new tokens: the one-call steps are the
    # plain attention calls; an empty batch still runs its cache side.
    from paged_kv_cache_14_gb300.step import step_from_host
    lens = [5, 64, 300, 700, 1300, 2100, 31, 900]
    b = build_batch(name="step_empty", seed=720, dtype="bf16", block_size=16, num_q_heads=64, num_kv_heads=8,
                    head_dim=128, q_lens=np.ones(len(lens), np.int32), kv_lens=lens, share_group=4,
                    share_prefix_tokens=256, cow_per_seq=False)
    for shared in (False, True):
        st = step_from_host(b, shared_prefix=shared)
        st.prepare()
        st.attend()
        ref = st.out.clone()
        e32 = torch.empty(0, dtype=torch.int32, device="cuda")
        e64 = torch.empty(0, dtype=torch.int64, device="cuda")
        ekv = torch.empty((0,) + tuple(st.k_new.shape[1:]), dtype=st.k_new.dtype, device="cuda")
        st.out.zero_()
        if shared:
            lib.pa_decode_step_shared_prefix(np.zeros((0, 2), np.int64), e32, e32, ekv, ekv, e64, st.q, st.k_cache,
                                             st.v_cache, st.block_tables, st.kv_lens, st.max_seq_len,
                                             st.group_starts, st.prefix_lens, b.scale, out=st.out,
                                             workspace=st.workspace)
        else:
            lib.pa_decode_step(np.zeros((0, 2), np.int64), e32, e32, ekv, ekv, e64, st.q, st.k_cache, st.v_cache,
                               st.block_tables, st.kv_lens, st.max_seq_len, b.scale, out=st.out,
                               workspace=st.workspace)
        torch.cuda.synchronize()
        assert lib.pa_get_status() == 0
        assert torch.equal(st.out, ref)
        assert_attention_close(to_f64(st.out), oracle_step(b), "bf16", f"empty parts (shared={shared}) vs oracle")
    # An empty batch with new tokens: only the cache side runs (slots of
    # sequences outside the batch are -1, so nothing is written).
    st = step_from_host(b)
    k0 = st.k_cache.clone()
    eq = torch.empty((0,) + tuple(st.q.shape[1:]), dtype=st.q.dtype, device="cuda")
    lib.pa_decode_step(np.zeros((0, 2), np.int64), st.new_seq_ids, st.new_positions, st.k_new, st.v_new,
                       st.slot_mapping, eq, st.k_cache, st.v_cache, st.block_tables, st.kv_lens[:0],
                       st.max_seq_len, b.scale, out=torch.empty_like(eq))
    torch.cuda.synchronize()
    assert bool((st.slot_mapping == -1).all())
    assert torch.equal(st.k_cache, k0)
    lib.pa_get_status()  # clears the slot errors recorded for tokens outside the batch


@pytest.mark.parametrize("shared", [False, True], ids=["plain", "shared_prefix"])
def test_one_call_step_with_more_than_1024_cow_pairs(lib, shared):
    # 1100 copy-on-write pairs take two chained copy launches (1024 pairs
    # per launch); the cache write must still see both complete.
    from paged_kv_cache_14_gb300.step import step_from_host
    rng = np.random.default_rng(730)
    n = 1100
    lens = rng.integers(20, 60, size=n).astype(np.int32)
    b = build_batch(name="step_cow_many", seed=730, dtype="bf16", block_size=16, num_q_heads=16, num_kv_heads=2,
                    head_dim=128, q_lens=np.ones(n, np.int32), kv_lens=lens, share_group=2,
                    share_prefix_tokens=16, cow_per_seq=True)
    assert len(b.cow_pairs) > 1024
    sep = step_from_host(b, shared_prefix=shared)
    sep.prepare()
    sep.attend()
    one = step_from_host(b, shared_prefix=shared)
    one.run()
    torch.cuda.synchronize()
    assert lib.pa_get_status() == 0
    assert torch.equal(one.k_cache, sep.k_cache) and torch.equal(one.v_cache, sep.v_cache)
    assert torch.equal(one.out, sep.out)
    assert_attention_close(to_f64(one.out), oracle_step(b), "bf16", "1100 CoW pairs: one-call step vs oracle")
