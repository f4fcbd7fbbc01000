"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each pin is a plain function that raises AssertionError on failure, so the
planted-mistake test at the bottom can check that every plausible mistake in
the oracle (a dropped term, a wrong index or sign, a swapped operand) is
caught by at least one pin.

What pins what:
  * torch's float64 scaled_dot_product_attention on CONTIGUOUS K/V (a library
    routine, no block table involved) pins gather + GQA + softmax for decode
    and, with its causal mask, for chunked prefill;
  * the paged pool in these tests is built by a numpy reshape of contiguous
    K/V into blocks, not by the oracle's position formula, and its padding is
    NaN so any read past a sequence's end shows up;
  * the block-size-4 walkthrough of "03 - PagedAttention & the vLLM V1
    Architecture" (tables, refcounts, which block holds which positions, the
    copy-on-write fork) pins slots, cache writes and block copies;
  * permutation of physical placement and prefix sharing vs private copies
    must leave outputs bit-identical;
  * closed forms (one key, zero query, constant V, vanishing scale);
  * the split-KV merge equals the unsplit softmax to ~1e-13;
  * the sizing examples printed on the pages.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.paged_attention as opa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# Independent helpers (built from numpy reshapes and torch library calls).
# ---------------------------------------------------------------------------

def paged_pool_from_contiguous(seqs_kv, block_size, pool_size, rng, share=None):
    """Pack contiguous [S, Hkv, D] arrays into a pool [P, Hkv, B, D] by
    padding each to whole blocks with NaN, reshaping to [nb, B, Hkv, D] and
    transposing to [nb, Hkv, B, D]; blocks go to a random permutation of ids.
    Returns (pool, tables) with tables padded by 0."""
    hkv, d = seqs_kv[0].shape[1:]
    pool = np.full((pool_size, hkv, block_size, d), -7.0)
    perm = rng.permutation(pool_size)
    cursor = 0
    rows = []
    for kv in seqs_kv:
        s = kv.shape[0]
        nb = -(-s // block_size)
        padded = np.full((nb * block_size, hkv, d), np.nan)
        padded[:s] = kv
        blocks = padded.reshape(nb, block_size, hkv, d).transpose(0, 2, 1, 3)
        ids = perm[cursor:cursor + nb]
        cursor += nb
        pool[ids] = blocks
        rows.append(ids)
    width = max(len(r) for r in rows)
    tables = np.zeros((len(rows), width), dtype=np.int64)
    for i, r in enumerate(rows):
        tables[i, :len(r)] = r
    return pool, tables


def sdpa(q_rows_h, k_seq, v_seq, scale, causal=False):
    """torch fp64 SDPA. q_rows_h [R, Hq, D]; k_seq, v_seq [L, Hkv, D];
    KV heads are expanded to query heads with repeat_interleave."""
    hq = q_rows_h.shape[1]
    hkv = k_seq.shape[1]
    qt = torch.from_numpy(np.ascontiguousarray(q_rows_h.transpose(1, 0, 2)))[None]
    kt = torch.from_numpy(np.ascontiguousarray(k_seq.transpose(1, 0, 2))).repeat_interleave(hq // hkv, dim=0)[None]
    vt = torch.from_numpy(np.ascontiguousarray(v_seq.transpose(1, 0, 2))).repeat_interleave(hq // hkv, dim=0)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)
    return o[0].numpy().transpose(1, 0, 2)


def random_case(seed, lens, B, hq, hkv, d, extra_blocks=5):
    rng = np.random.default_rng(seed)
    ks = [rng.standard_normal((L, hkv, d)) for L in lens]
    vs = [rng.standard_normal((L, hkv, d)) for L in lens]
    q = rng.standard_normal((len(lens), hq, d))
    need = sum(-(-L // B) for L in lens)
    P = need + extra_blocks
    prng = np.random.default_rng(seed + 1000)
    kpool, tables = paged_pool_from_contiguous(ks, B, P, prng)
    prng = np.random.default_rng(seed + 1000)
    vpool, tables_v = paged_pool_from_contiguous(vs, B, P, prng)
    assert np.array_equal(tables, tables_v)
    return q, ks, vs, kpool, vpool, tables


DECODE_CASES = [
    # (seed, lens, B, Hq, Hkv, D)
    (0, [1, 15, 16, 33], 16, 2, 1, 64),
    (1, [3, 4, 5, 9, 12], 4, 8, 2, 16),
    (2, [31, 32, 33, 64, 65], 32, 8, 1, 32),
    (3, [17, 1, 48], 16, 16, 2, 24),
    (4, [7, 100], 16, 4, 4, 8),
]


# ---------------------------------------------------------------------------
# Pins.
# ---------------------------------------------------------------------------

def pin_decode_vs_sdpa():
    for seed, lens, B, hq, hkv, d in DECODE_CASES:
        q, ks, vs, kpool, vpool, tables = random_case(seed, lens, B, hq, hkv, d)
        scale = 1.0 / math.sqrt(d)
        got = oracle.decode(q, kpool, vpool, tables, lens, scale, B)
        for i, L in enumerate(lens):
            ref = sdpa(q[i][None], ks[i], vs[i], scale)[0]
            assert np.max(np.abs(got[i] - ref)) < 1e-12, (seed, i)


def pin_prefill_vs_sdpa():
    rng = np.random.default_rng(11)
    for B, hq, hkv, d, ctxs, qls in [
        (16, 4, 2, 16, [0, 5, 16, 21], [1, 7, 16, 3]),
        (4, 8, 1, 8, [3, 0], [9, 4]),
        (32, 6, 3, 16, [40, 1], [33, 2]),
    ]:
        lens = [c + ql for c, ql in zip(ctxs, qls)]
        ks = [rng.standard_normal((L, hkv, d)) for L in lens]
        vs = [rng.standard_normal((L, hkv, d)) for L in lens]
        P = sum(-(-L // B) for L in lens) + 3
        kpool, tables = paged_pool_from_contiguous(ks, B, P, np.random.default_rng(5))
        vpool, _ = paged_pool_from_contiguous(vs, B, P, np.random.default_rng(5))
        qfull = [rng.standard_normal((L, hq, d)) for L in lens]
        q = np.concatenate([qf[c:] for qf, c in zip(qfull, ctxs)])
        cu = np.concatenate([[0], np.cumsum(qls)])
        scale = 0.37
        got = oracle.prefill(q, cu, ctxs, kpool, vpool, tables, scale, B)
        for i, (c, ql) in enumerate(zip(ctxs, qls)):
            ref = sdpa(qfull[i], ks[i], vs[i], scale, causal=True)[c:]
            assert np.max(np.abs(got[cu[i]:cu[i + 1]] - ref)) < 1e-12, (B, i)


def _worked_example():
    with open(os.path.join(GOLDEN, "worked_example_bs4.json")) as f:
        return json.load(f)


def _token_kv(tokens, p, d=8):
    """K and V at position p: a seeded function of the token prefix 0..p, so
    two sequences with the same prefix have identical K/V there."""
    key = "\x1f".join(tokens[:p + 1]).encode()
    seed = int.from_bytes(key[-8:].rjust(8, b"\0"), "little") ^ len(key) ^ (p * 7919)
    rng = np.random.default_rng([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF, len(key)])
    return rng.standard_normal(d), rng.standard_normal(d)


def pin_worked_example():
    ex = _worked_example()
    B = ex["block_size"]
    A, Bq = ex["sequences"]["A"], ex["sequences"]["B"]
    tables = {"A": A["block_table"], "B": Bq["block_table"]}
    # Refcounts printed on the page = how many tables name each block.
    for entry in ex["pool"]:
        count = sum(t.count(entry["block"]) for t in tables.values())
        assert count == entry["refcount"], entry
    # Every position the page lists for a block maps (through the holder's
    # table) to a slot inside that block, at distinct slots.
    for entry in ex["pool"]:
        lo, hi = entry["positions"]
        for name in entry["holders"]:
            slots = [oracle.slot_for(tables[name], p, B) for p in range(lo, hi + 1)]
            assert all(s // B == entry["block"] for s in slots), (entry, name, slots)
            assert len(set(slots)) == len(slots)
    # Shared prefix: the two sequences agree on positions 0..5 only.
    n_shared = ex["shared_prefix_tokens"]
    assert A["tokens"][:n_shared] == Bq["tokens"][:n_shared]
    assert A["tokens"][n_shared] != Bq["tokens"][n_shared]

    d = 8
    kvA = [_token_kv(A["tokens"], p, d) for p in range(len(A["tokens"]))]
    kvB = [_token_kv(Bq["tokens"], p, d) for p in range(len(Bq["tokens"]))]
    for p in range(n_shared):
        assert np.array_equal(kvA[p][0], kvB[p][0])
    assert not np.array_equal(kvA[n_shared][0], kvB[n_shared][0])

    # Build the pool the way the engine would: A is cached first; B was forked
    # from A after position 5 (sharing blocks 0 and 1), so its write at
    # position 6 hits shared block 1 -> copy-on-write into block 2, then B's
    # positions 6, 7 go to block 2 and 8, 9 to block 4.
    k_cache = np.full((5, 1, B, d), np.nan)
    v_cache = np.full((5, 1, B, d), np.nan)
    slotsA = oracle.slot_mapping(np.array([tables["A"]]), [0] * 12, list(range(12)), B)
    oracle.reshape_and_cache(np.array([kv[0][None] for kv in kvA]), np.array([kv[1][None] for kv in kvA]),
                             slotsA, k_cache, v_cache, B)
    oracle.copy_blocks(k_cache, v_cache, [(1, 2)])
    posB = [6, 7, 8, 9]
    slotsB = oracle.slot_mapping(np.array([tables["B"]]), [0] * 4, posB, B)
    oracle.reshape_and_cache(np.array([kvB[p][0][None] for p in posB]), np.array([kvB[p][1][None] for p in posB]),
                             slotsB, k_cache, v_cache, B)
    # Block 2 now holds B's own positions 4..7 (the copy carried 4, 5).
    for name, kv, tbl in (("A", kvA, tables["A"]), ("B", kvB, tables["B"])):
        L = len(kv)
        K = oracle.gather_sequence(k_cache, tbl, L, B)[:, 0]
        V = oracle.gather_sequence(v_cache, tbl, L, B)[:, 0]
        assert np.array_equal(K, np.array([x[0] for x in kv])), name
        assert np.array_equal(V, np.array([x[1] for x in kv])), name
    # Attention over the paged pool equals attention over each sequence's
    # own contiguous K/V, and block 0 serves both.
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 2, d))
    out = oracle.decode(q, k_cache, v_cache, np.array([tables["A"], tables["B"]]), [12, 10], 0.5, B)
    for i, kv in enumerate((kvA, kvB)):
        Kc = np.array([x[0] for x in kv])[:, None]
        Vc = np.array([x[1] for x in kv])[:, None]
        ref = sdpa(q[i][None], Kc, Vc, 0.5)[0]
        assert np.max(np.abs(out[i] - ref)) < 1e-12
    # Without the copy (the page-5 block manager allocates but never copies),
    # B's positions 4, 5 would be garbage: the copy is what makes CoW correct.
    k2 = np.full((5, 1, B, d), np.nan)
    v2 = np.full((5, 1, B, d), np.nan)
    oracle.reshape_and_cache(np.array([kv[0][None] for kv in kvA]), np.array([kv[1][None] for kv in kvA]),
                             slotsA, k2, v2, B)
    oracle.reshape_and_cache(np.array([kvB[p][0][None] for p in posB]), np.array([kvB[p][1][None] for p in posB]),
                             slotsB, k2, v2, B)
    assert np.isnan(oracle.gather_sequence(k2, tables["B"], 10, B)[4:6]).all()


def pin_slots_match_layout():
    """slot_for addresses, in the slot-major view of the pool (reshape of
    [P, Hkv, B, D] to [P*B, Hkv, D]), exactly where the reshape-built pool put
    each position."""
    for seed, lens, B, hq, hkv, d in DECODE_CASES:
        q, ks, vs, kpool, vpool, tables = random_case(seed, lens, B, hq, hkv, d)
        flat = kpool.transpose(0, 2, 1, 3).reshape(-1, hkv, d)
        for i, L in enumerate(lens):
            for p in range(L):
                assert np.array_equal(flat[oracle.slot_for(tables[i], p, B)], ks[i][p])
        seq_ids = np.repeat(np.arange(len(lens)), lens)
        pos = np.concatenate([np.arange(L) for L in lens])
        sm = oracle.slot_mapping(tables, seq_ids, pos, B)
        assert len(set(sm.tolist())) == len(sm)
        assert np.array_equal(flat[sm], np.concatenate(ks))


def pin_reshape_and_cache_roundtrip():
    """Writing every position with reshape_and_cache reproduces the reshape-
    built pool bit for bit; other blocks and slots < 0 are left alone."""
    for seed, lens, B, hq, hkv, d in DECODE_CASES:
        q, ks, vs, kpool, vpool, tables = random_case(seed, lens, B, hq, hkv, d)
        seq_ids = np.repeat(np.arange(len(lens)), lens)
        pos = np.concatenate([np.arange(L) for L in lens])
        slots = oracle.slot_mapping(tables, seq_ids, pos, B)
        slots_with_pad = np.concatenate([slots, [-1, -5]])
        kn = np.concatenate(ks + [np.full((2, hkv, d), 123.0)])
        vn = np.concatenate(vs + [np.full((2, hkv, d), 321.0)])
        kc = np.full_like(kpool, -7.0)
        vc = np.full_like(vpool, -7.0)
        oracle.reshape_and_cache(kn, vn, slots_with_pad, kc, vc, B)
        live = np.isfinite(kpool) & (kpool != -7.0)
        assert np.array_equal(kc[live], kpool[live])
        assert np.array_equal(vc[live], vpool[live])
        assert np.all(kc[~live] == -7.0) and np.all(vc[~live] == -7.0)


def pin_copy_blocks():
    rng = np.random.default_rng(9)
    kc = rng.standard_normal((10, 2, 4, 3))
    vc = rng.standard_normal((10, 2, 4, 3))
    k0, v0 = kc.copy(), vc.copy()
    pairs = [(1, 7), (1, 8), (4, 2)]
    oracle.copy_blocks(kc, vc, pairs)
    for s, t in pairs:
        assert np.array_equal(kc[t], k0[s]) and np.array_equal(vc[t], v0[s])
    untouched = [b for b in range(10) if b not in (7, 8, 2)]
    assert np.array_equal(kc[untouched], k0[untouched]) and np.array_equal(vc[untouched], v0[untouched])


def pin_permutation_invariance():
    for seed, lens, B, hq, hkv, d in DECODE_CASES:
        q, ks, vs, kpool, vpool, tables = random_case(seed, lens, B, hq, hkv, d)
        P = kpool.shape[0]
        base = oracle.decode(q, kpool, vpool, tables, lens, 0.3, B)
        perm = np.random.default_rng(seed + 5).permutation(P)
        kp2 = np.empty_like(kpool)
        vp2 = np.empty_like(vpool)
        kp2[perm] = kpool
        vp2[perm] = vpool
        t2 = perm[tables]
        moved = oracle.decode(q, kp2, vp2, t2, lens, 0.3, B)
        assert np.array_equal(base, moved)


def pin_prefix_sharing():
    """Sequences reading one shared prefix block vs private copies of it."""
    rng = np.random.default_rng(21)
    B, hkv, hq, d = 4, 2, 4, 8
    prefix_k = rng.standard_normal((8, hkv, d))
    prefix_v = rng.standard_normal((8, hkv, d))
    lens = [8, 11, 14]
    ks = [np.concatenate([prefix_k, rng.standard_normal((L - 8, hkv, d))]) for L in lens]
    vs = [np.concatenate([prefix_v, rng.standard_normal((L - 8, hkv, d))]) for L in lens]
    q = rng.standard_normal((3, hq, d))
    # Private layout (each sequence has its own copy of the prefix blocks).
    kpool, tables = paged_pool_from_contiguous(ks, B, 20, np.random.default_rng(1))
    vpool, _ = paged_pool_from_contiguous(vs, B, 20, np.random.default_rng(1))
    private = oracle.decode(q, kpool, vpool, tables, lens, 0.4, B)
    # Shared layout: all three tables point at sequence 0's two prefix blocks.
    shared_tables = tables.copy()
    shared_tables[1:, :2] = tables[0, :2]
    shared = oracle.decode(q, kpool, vpool, shared_tables, lens, 0.4, B)
    assert np.array_equal(private, shared)


def pin_closed_forms():
    rng = np.random.default_rng(4)
    B, hkv, hq, d = 16, 2, 4, 8
    # One key: the output is v_0 exactly, whatever q and scale are.
    ks = [rng.standard_normal((1, hkv, d))]
    vs = [rng.standard_normal((1, hkv, d))]
    kp, t = paged_pool_from_contiguous(ks, B, 3, np.random.default_rng(0))
    vp, _ = paged_pool_from_contiguous(vs, B, 3, np.random.default_rng(0))
    q = rng.standard_normal((1, hq, d)) * 10
    out = oracle.decode(q, kp, vp, t, [1], 0.9, B)
    for h in range(hq):
        assert np.array_equal(out[0, h], vs[0][0, h // 2])
    # Zero query, or a vanishing scale: the mean of V's rows.
    L = 37
    ks = [rng.standard_normal((L, hkv, d))]
    vs = [rng.standard_normal((L, hkv, d))]
    kp, t = paged_pool_from_contiguous(ks, B, 5, np.random.default_rng(0))
    vp, _ = paged_pool_from_contiguous(vs, B, 5, np.random.default_rng(0))
    out = oracle.decode(np.zeros((1, hq, d)), kp, vp, t, [L], 0.7, B)
    out2 = oracle.decode(rng.standard_normal((1, hq, d)), kp, vp, t, [L], 1e-300, B)
    for h in range(hq):
        assert np.max(np.abs(out[0, h] - vs[0][:, h // 2].mean(axis=0))) < 1e-14
        assert np.max(np.abs(out2[0, h] - vs[0][:, h // 2].mean(axis=0))) < 1e-14
    # All V rows equal c: the output is c.
    c = rng.standard_normal((hkv, d))
    vs = [np.broadcast_to(c, (L, hkv, d)).copy()]
    vp, _ = paged_pool_from_contiguous(vs, B, 5, np.random.default_rng(0))
    out = oracle.decode(rng.standard_normal((1, hq, d)), kp, vp, t, [L], 0.7, B)
    for h in range(hq):
        assert np.max(np.abs(out[0, h] - c[h // 2])) < 1e-14
    # One dominant key: softmax picks its value.
    kk = rng.standard_normal((L, hkv, d)) * 0.01
    qv = np.ones(d)
    kk[13, :, :] = 50.0 * qv
    kp, t = paged_pool_from_contiguous([kk], B, 5, np.random.default_rng(0))
    vv = rng.standard_normal((L, hkv, d))
    vp, _ = paged_pool_from_contiguous([vv], B, 5, np.random.default_rng(0))
    out = oracle.decode(np.broadcast_to(qv, (1, hq, d)).copy(), kp, vp, t, [L], 1.0, B)
    for h in range(hq):
        assert np.max(np.abs(out[0, h] - vv[13, h // 2])) < 1e-12


def pin_split_merge():
    rng = np.random.default_rng(8)
    for L, T in [(1, 16), (100, 16), (257, 64), (1000, 1000), (1000, 999), (64, 1)]:
        K = rng.standard_normal((L, 32))
        K[rng.random(L) < 0.05] *= 8
        V = rng.standard_normal((L, 32))
        q = rng.standard_normal(32)
        ref = oracle.softmax_attention(q[None], K, V, 0.25)[0]
        m, l, o = oracle.partition_partials(q, K, V, 0.25, T)
        assert len(m) == -(-L // T)
        got = oracle.merge_partials(m, l, o)
        assert np.max(np.abs(got - ref)) < 1e-13, (L, T)
        # A single partition's unnormalised output over its own sum is its softmax.
        if L >= T:
            one = oracle.softmax_attention(q[None], K[:T], V[:T], 0.25)[0]
            assert np.max(np.abs(o[0] / l[0] - one)) < 1e-13


def pin_sizing_examples():
    with open(os.path.join(GOLDEN, "sizing_examples.json")) as f:
        ex = json.load(f)
    f1 = ex["block_mapping_figure"]
    assert oracle.num_blocks_for(f1["seq_len"], f1["block_size"]) == f1["blocks"]
    frac = oracle.internal_fragmentation(f1["seq_len"], f1["block_size"])
    assert frac * f1["blocks"] * f1["block_size"] == f1["unused_slots"]
    # The figure prints 29.1 for 28/96 = 29.17 (truncated, not rounded).
    assert math.floor(frac * 1000) / 10 == f1["waste_percent_printed"]
    fb = ex["fragmentation_bound"]
    assert round(100.0 * fb["block_size"] / fb["seq_len"], 2) == fb["bound_percent"]
    for S in range(1, 600):
        for B in (4, 16, 32):
            assert oracle.internal_fragmentation(S, B) < B / S
    lc = ex["lifecycle"]
    assert oracle.num_blocks_for(lc["seq_len"], lc["block_size"]) == lc["blocks"]
    kb = ex["kv_bytes_70b"]
    gb = oracle.kv_bytes_per_sequence(kb["num_layers"], kb["num_kv_heads"], kb["head_dim"],
                                      kb["seq_len"], kb["elem_bytes"]) / 1e9
    assert round(gb, 2) == kb["gigabytes_printed"]
    # Block bytes for one layer of the 70B shape at B = 16, 2-byte elements:
    # K and V of 16 tokens x 8 heads x 128 dims.
    assert oracle.block_bytes(1, 8, 128, 16, 2) == 2 * 16 * 8 * 128 * 2
    # A whole block's bytes, times the block count, is the per-sequence bytes
    # whenever the length is block-aligned.
    assert oracle.block_bytes(80, 8, 128, 16, 1) * oracle.num_blocks_for(8192, 16) == \
        oracle.kv_bytes_per_sequence(80, 8, 128, 8192, 1)


def pin_swap_roundtrip():
    """Swap a sequence's blocks out to a host pool and back into other device
    blocks: the blocks come back bit for bit and the sequence's attention
    (with its table pointing at the new blocks) equals the attention before
    the swap."""
    rng = np.random.default_rng(31)
    lens = np.array([40, 70])
    q, _, _, kc, vc, tables = random_case(31, lens, B=16, hq=4, hkv=2, d=16, extra_blocks=12)
    before = oracle.decode(q, kc, vc, tables, lens, 0.3, 16)
    used = tables[1][: -(-int(lens[1]) // 16)]
    free = np.setdiff1d(np.arange(kc.shape[0]), np.concatenate([tables[0][: -(-int(lens[0]) // 16)], used]))
    host_k = np.zeros((len(used),) + kc.shape[1:])
    host_v = np.zeros_like(host_k)
    oracle.swap_blocks(kc, vc, host_k, host_v, [(int(b), i) for i, b in enumerate(used)])
    saved_k, saved_v = kc[used].copy(), vc[used].copy()
    kc[used] = np.nan                      # the device blocks are reused meanwhile
    vc[used] = np.nan
    new = rng.choice(free, size=len(used), replace=False)
    oracle.swap_blocks(host_k, host_v, kc, vc, [(i, int(b)) for i, b in enumerate(new)])
    assert np.array_equal(kc[new], saved_k, equal_nan=True) and np.array_equal(vc[new], saved_v, equal_nan=True)
    t2 = tables.copy()
    t2[1][: len(used)] = new
    after = oracle.decode(q, kc, vc, t2, lens, 0.3, 16)
    assert np.array_equal(before[1], after[1])


ALL_PINS = [
    pin_decode_vs_sdpa, pin_prefill_vs_sdpa, pin_worked_example, pin_slots_match_layout,
    pin_reshape_and_cache_roundtrip, pin_copy_blocks, pin_permutation_invariance,
    pin_prefix_sharing, pin_closed_forms, pin_split_merge, pin_sizing_examples, pin_swap_roundtrip,
]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# Planted mistakes: each must be caught by at least one pin.
# ---------------------------------------------------------------------------

def _mut_offset(monkeypatch):
    monkeypatch.setattr(opa, "logical_block_and_offset", lambda p, B: (p // B, (p + 1) % B))


def _mut_swap_block_offset_in_gather(monkeypatch):
    def bad(cache, row, length, B):
        pos = np.arange(int(length))
        blk = np.asarray(row, dtype=np.int64)[np.minimum(pos % B, len(row) - 1)]
        off = np.minimum(pos // B, B - 1)
        return opa.to_f64(np.asarray(cache)[blk, :, off, :])
    monkeypatch.setattr(opa, "gather_sequence", bad)
    monkeypatch.setattr(oracle, "gather_sequence", bad)


def _mut_gqa(monkeypatch):
    monkeypatch.setattr(opa, "kv_head_of", lambda h, hq, hkv: h % hkv)


def _mut_no_scale(monkeypatch):
    orig = opa.softmax_attention
    monkeypatch.setattr(opa, "softmax_attention", lambda q, k, v, s: orig(q, k, v, 1.0))


def _mut_k_for_v(monkeypatch):
    orig = opa.softmax_attention
    monkeypatch.setattr(opa, "softmax_attention", lambda q, k, v, s: orig(q, k, k, s))


def _mut_softmax_no_norm(monkeypatch):
    def bad(q, k, v, s):
        sc = (q @ k.T) * s
        p = np.exp(sc - sc.max(axis=1, keepdims=True))
        return p @ v
    monkeypatch.setattr(opa, "softmax_attention", bad)


def _mut_prefill_off_by_one(monkeypatch):
    monkeypatch.setattr(opa, "prefill", _prefill_excluding_self)
    monkeypatch.setattr(oracle, "prefill", _prefill_excluding_self)


def _prefill_excluding_self(q, cu, ctx_lens, kc, vc, bt, scale, B, seqs=None, rows=None):
    qf = opa.to_f64(q)
    out = np.full(qf.shape, np.nan)
    hq, hkv = qf.shape[1], kc.shape[1]
    for i in range(len(cu) - 1):
        ctx = int(ctx_lens[i])
        L = ctx + cu[i + 1] - cu[i]
        K = opa.gather_sequence(kc, bt[i], L, B)
        V = opa.gather_sequence(vc, bt[i], L, B)
        for r in range(cu[i + 1] - cu[i]):
            keys = max(ctx + r, 1)
            for h in range(hq):
                g = opa.kv_head_of(h, hq, hkv)
                out[cu[i] + r, h] = opa.softmax_attention(qf[cu[i] + r, h][None], K[:keys, g], V[:keys, g], scale)[0]
    return out


def _mut_merge_sign(monkeypatch):
    def bad(m, l, o):
        M = m.max()
        w = np.exp(M - m)
        return (w[:, None] * o).sum(axis=0) / (w * l).sum()
    monkeypatch.setattr(opa, "merge_partials", bad)
    monkeypatch.setattr(oracle, "merge_partials", bad)


def _mut_copy_k_only(monkeypatch):
    def bad(kc, vc, pairs):
        for s, t in np.asarray(pairs).reshape(-1, 2):
            kc[int(t)] = kc[int(s)]
    monkeypatch.setattr(opa, "copy_blocks", bad)
    monkeypatch.setattr(oracle, "copy_blocks", bad)


def _mut_cache_write_offset0(monkeypatch):
    def bad(kn, vn, slots, kc, vc, B):
        for t, slot in enumerate(np.asarray(slots)):
            if slot < 0:
                continue
            kc[int(slot) // B, :, 0, :] = kn[t]
            vc[int(slot) // B, :, 0, :] = vn[t]
    monkeypatch.setattr(opa, "reshape_and_cache", bad)
    monkeypatch.setattr(oracle, "reshape_and_cache", bad)


def _mut_slot_uses_logical_block(monkeypatch):
    def bad(row, p, B):
        blk, off = opa.logical_block_and_offset(int(p), B)
        return blk * B + off
    monkeypatch.setattr(opa, "slot_for", bad)
    monkeypatch.setattr(oracle, "slot_for", bad)


def _mut_fragmentation_floor(monkeypatch):
    monkeypatch.setattr(oracle, "num_blocks_for", lambda S, B: S // B)


def _mut_swap_k_only(monkeypatch):
    def bad(sk, sv, dk, dv, pairs):
        for s_, d in np.asarray(pairs).reshape(-1, 2):
            dk[int(d)] = sk[int(s_)]
    monkeypatch.setattr(opa, "swap_blocks", bad)
    monkeypatch.setattr(oracle, "swap_blocks", bad)


def _mut_swap_reversed(monkeypatch):
    def bad(sk, sv, dk, dv, pairs):
        for s_, d in np.asarray(pairs).reshape(-1, 2):
            dk[int(s_) % dk.shape[0]] = sk[int(d) % sk.shape[0]]
            dv[int(s_) % dv.shape[0]] = sv[int(d) % sv.shape[0]]
    monkeypatch.setattr(opa, "swap_blocks", bad)
    monkeypatch.setattr(oracle, "swap_blocks", bad)


MUTATIONS = [
    _mut_offset, _mut_swap_block_offset_in_gather, _mut_gqa, _mut_no_scale, _mut_k_for_v,
    _mut_softmax_no_norm, _mut_prefill_off_by_one, _mut_merge_sign, _mut_copy_k_only,
    _mut_cache_write_offset0, _mut_slot_uses_logical_block, _mut_fragmentation_floor, _mut_swap_k_only,
    _mut_swap_reversed,
]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=lambda f: f.__name__)
def test_planted_mistake_is_caught(mutation, monkeypatch):
    mutation(monkeypatch)
    caught = []
    for pin in ALL_PINS:
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught {mutation.__name__}"
