"""e5m2 KV cache on the GPU (the second 8-bit format of block-quantised
caching): the quantising cache write bit for bit against the oracle's e5m2
rule, and decode, shared-prefix decode and chunked prefill over the e5m2
pools against the fp64 oracle on the dequantised values (each stored value =
e5m2 code x its (block, KV head) scale)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import oracle.fp8_kv as f8
from helpers import assert_attention_close, full_config, to_f64
from workloads import build_batch, e5m2_pool

pytestmark = pytest.mark.gpu

FINITE = np.array([c for c in range(256) if (c >> 2) & 0x1F != 0x1F], dtype=np.uint8)


def _finite_codes(rng, shape) -> np.ndarray:
    return FINITE[rng.integers(0, FINITE.size, size=shape)]


def _f32_bits(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)


def _quantised(b):
    """e5m2 pools of a batch's 16-bit values (the oracle's whole-block quantiser)."""
    kc, ks = f8.quantize_fresh_blocks_e5m2(b.k_cache.float().numpy())
    vc, vs = f8.quantize_fresh_blocks_e5m2(b.v_cache.float().numpy())
    return kc, vc, np.stack([ks, vs], axis=-1).astype(np.float32)


def _random_codes(b, seed):
    """Codes uniform over every finite e5m2 value, scales over three binades."""
    kc, vc, sc = e5m2_pool(seed, b.num_blocks, b.num_kv_heads, b.block_size, b.head_dim)
    return kc.numpy(), vc.numpy(), sc.numpy()


def _dev(pool):
    return tuple(torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in pool)


def _oracle_decode_rows(b, kc, vc, sc, seqs=None):
    """Oracle decode, dequantising one sequence's blocks at a time."""
    out = np.full((b.num_seqs, b.num_q_heads, b.head_dim), np.nan)
    for i in (range(b.num_seqs) if seqs is None else seqs):
        nb = -(-int(b.kv_lens[i]) // b.block_size)
        blocks = b.block_tables[i][:nb]
        kd = f8.dequantize_e5m2(kc[blocks], sc[blocks, :, 0])
        vd = f8.dequantize_e5m2(vc[blocks], sc[blocks, :, 1])
        tables = np.zeros_like(b.block_tables)
        tables[i, :nb] = np.arange(nb)
        out[i] = oracle.decode(b.q, kd, vd, tables, b.kv_lens, b.scale, b.block_size, seqs=[i])[i]
    return out


def _oracle_step_pools(b, pool):
    ko, vo, so = (x.copy() for x in pool)
    f8.copy_blocks_fp8(ko, vo, so, b.cow_pairs)
    slots = oracle.slot_mapping(b.block_tables, b.new_seq_ids, b.new_positions, b.block_size)
    f8.reshape_and_cache_e5m2(b.k_new.float().numpy(), b.v_new.float().numpy(), slots, ko, vo, so, b.block_size)
    return ko, vo, so


# ---------------------------------------------------------------------------
# Cache write
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("D", [64, 128])
def test_cache_write_bit_exact(lib, dtype, B, D):
    rng = np.random.default_rng(B * 1000 + D + len(dtype) + 7)
    P, H = 14, 3
    kc0 = _finite_codes(rng, (P, H, B, D))
    vc0 = _finite_codes(rng, (P, H, B, D))
    sc0 = np.exp2(rng.uniform(-17, -10, size=(P, H, 2))).astype(np.float32)
    # A run that starts mid-block and crosses into a fresh block, padding
    # inside a run, single-token appends (one forcing the scale up), a fresh
    # block, a whole block, a full block's tail.
    slots = []
    slots += [3 * B + o for o in range(B // 2, B)] + [7 * B + o for o in range(0, 5)]
    slots += [-1]
    slots += [7 * B + 5, 7 * B + 6]
    slots += [5 * B + 9, -1, 9 * B + 2, 0 * B + 0, 11 * B + B - 1]
    slots += [12 * B + o for o in range(B)]
    slots = np.array(slots, dtype=np.int64)
    T = len(slots)
    mag = np.exp2(rng.uniform(-10, 3, size=(T, 1, 1)))
    mag[np.flatnonzero(slots == 5 * B + 9)] = 3000.0       # forces a larger scale on block 5
    k = torch.from_numpy((rng.standard_normal((T, H, D)) * mag).astype(np.float32)).to(
        {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype])
    v = (k.float() * -0.7 + 0.01).to(k.dtype)
    kd, vd = torch.from_numpy(kc0).cuda(), torch.from_numpy(vc0).cuda()
    sd = torch.from_numpy(sc0).cuda()
    lib.pa_reshape_and_cache_e5m2(k.cuda(), v.cuda(), torch.from_numpy(slots).cuda(), kd, vd, sd)
    assert lib.pa_get_status() == 0
    ko, vo, so = kc0.copy(), vc0.copy(), sc0.copy()
    f8.reshape_and_cache_e5m2(k.float().numpy(), v.float().numpy(), slots, ko, vo, so, B)
    assert np.array_equal(_f32_bits(sd.cpu().numpy()), _f32_bits(so)), "scales differ"
    assert np.array_equal(kd.cpu().numpy(), ko), "K codes differ"
    assert np.array_equal(vd.cpu().numpy(), vo), "V codes differ"
    assert so[5, 0, 0] > sc0[5, 0, 0]                       # the growth path ran


def test_cache_write_top_code_and_out_of_pool_slot(lib):
    """Each block's largest element takes the top finite code 0x7B (0xFB);
    a slot outside the pool is reported and nothing else is written."""
    P, H, B, D = 4, 2, 16, 128
    kc0 = np.zeros((P, H, B, D), np.uint8)
    kd, vd = torch.from_numpy(kc0).cuda(), torch.from_numpy(kc0).cuda()
    sd = torch.zeros(P, H, 2, device="cuda")
    k = torch.randn(3, H, D, dtype=torch.bfloat16, device="cuda")
    lib.pa_reshape_and_cache_e5m2(k, -k, torch.tensor([P * B + 3, 1 * B, 1 * B + 1], device="cuda"), kd, vd, sd)
    assert lib.pa_get_status() == -7
    got = kd.cpu().numpy()
    assert (got[[0, 2, 3]] == 0).all()
    for h in range(H):
        assert np.abs(f8.e5m2_decode(got[1, h, :2])).max() == 57344.0
        assert {0x7B, 0xFB} & set(got[1, h, :2].ravel().tolist())


# ---------------------------------------------------------------------------
# Decode
# ---------------------------------------------------------------------------

CASES = [
    # dtype, B, Hq, Hkv, lens
    ("bf16", 16, 8, 1, [1, 15, 16, 17, 33, 200]),
    ("bf16", 32, 64, 8, [1, 31, 32, 33, 513, 1025]),
    ("f16", 16, 16, 2, [1, 17, 160, 999]),
    ("bf16", 16, 32, 1, [9, 70]),       # group 32: two row groups per KV head
]


def _decode(lib, b, pool, partition=0):
    kc, vc, sc = _dev(pool)
    out = lib.pa_decode_e5m2(b.q.cuda(), kc, vc, sc, torch.from_numpy(b.block_tables).cuda(),
                             torch.from_numpy(b.kv_lens.astype(np.int32)).cuda(), b.max_seq_len, b.scale,
                             partition_size=partition)
    st = lib.pa_get_status()
    assert st == 0, lib.pa_strerror(st)
    return to_f64(out)


@pytest.mark.parametrize("pool_kind", ["quantised", "random"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-B{c[1]}-Hq{c[2]}-Hkv{c[3]}")
@pytest.mark.parametrize("partition", [0, 3])
def test_decode_e5m2_matches_oracle(lib, case, partition, pool_kind):
    dtype, B, hq, hkv, lens = case
    b = build_batch(name="e5m2", seed=CASES.index(case) + 240, dtype=dtype, block_size=B, num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=128, q_lens=np.ones(len(lens), np.int32), kv_lens=lens)
    pool = _quantised(b) if pool_kind == "quantised" else _random_codes(b, 241)
    out = _decode(lib, b, pool, partition * B)
    assert_attention_close(out, _oracle_decode_rows(b, *pool), dtype, f"{case} partition {partition}")


def test_decode_e5m2_ignores_inf_and_nan_codes_past_the_end(lib):
    lens = [5, 17, 40]
    b = build_batch(name="e5m2nan", seed=262, dtype="f16", block_size=16, num_q_heads=16, num_kv_heads=2,
                    head_dim=128, q_lens=np.ones(3, np.int32), kv_lens=lens)
    kc, vc, sc = _quantised(b)
    clean = _decode(lib, b, (kc, vc, sc))
    kn, vn = kc.copy(), vc.copy()
    for i, L in enumerate(lens):
        last = b.block_tables[i][(L - 1) // 16]
        kn[last, :, L % 16 or 16:, :] = 0x7C      # +infinity
        vn[last, :, L % 16 or 16:, :] = 0xFF      # NaN
    dirty = _decode(lib, b, (kn, vn, sc))
    assert np.array_equal(clean, dirty)
    assert_attention_close(dirty, _oracle_decode_rows(b, kc, vc, sc), "f16", "inf / NaN codes past the end")


def test_step_e5m2_matches_oracle(lib):
    """The whole step on an e5m2 cache: copy-on-write of codes and scales,
    slots, the quantising cache write (appends into partly filled blocks),
    decode; and the same with shared-prefix decode."""
    from paged_kv_cache_14_gb300.step import step_from_host
    lens = [5, 64, 300, 700, 1300, 31, 900, 17]
    b = build_batch(name="e5m2step", seed=263, dtype="bf16", block_size=16, num_q_heads=64, num_kv_heads=8,
                    head_dim=128, q_lens=np.ones(8, np.int32), kv_lens=lens, share_group=4,
                    share_prefix_tokens=256, cow_per_seq=True)
    pool = _quantised(b)
    ko, vo, so = _oracle_step_pools(b, pool)
    ref = _oracle_decode_rows(b, ko, vo, so)
    for shared in (False, True):
        st = step_from_host(b, shared_prefix=shared, fp8_pool=tuple(torch.from_numpy(x) for x in pool),
                            kv_format="e5m2")
        out = to_f64(st.run())
        assert lib.pa_get_status() == 0
        assert np.array_equal(st.k_cache.cpu().numpy(), ko) and np.array_equal(st.v_cache.cpu().numpy(), vo)
        assert np.array_equal(_f32_bits(st.kv_scales.cpu().numpy()), _f32_bits(so))
        assert_attention_close(out, ref, "bf16", f"e5m2 step (shared prefix {shared})")


# ---------------------------------------------------------------------------
# Shared-prefix decode
# ---------------------------------------------------------------------------

SP_CASES = [
    # dtype, B, Hq, Hkv, lens, group, prefix tokens
    ("bf16", 16, 64, 8, [5, 64, 64, 65, 200, 31, 1000, 129, 17, 80], 4, 64),
    ("f16", 32, 64, 8, [40, 300, 1000, 2000, 33, 64, 65, 999], 8, 256),
    ("bf16", 16, 64, 8, list(range(100, 100 + 37 * 45, 45)), 37, 512),  # 37 members: 3 tiles of 16
]


@pytest.mark.parametrize("pool_kind", ["quantised", "random"])
@pytest.mark.parametrize("case", SP_CASES, ids=lambda c: f"{c[0]}-B{c[1]}-G{c[2] // c[3]}-grp{c[5]}")
@pytest.mark.parametrize("partition", [0, 64])
def test_shared_prefix_e5m2_matches_oracle(lib, case, partition, pool_kind):
    dtype, B, hq, hkv, lens, grp, pref = case
    b = build_batch(name="e5m2cascade", seed=SP_CASES.index(case) + 270, dtype=dtype, block_size=B,
                    num_q_heads=hq, num_kv_heads=hkv, head_dim=128, q_lens=np.ones(len(lens), np.int32),
                    kv_lens=lens, share_group=grp, share_prefix_tokens=pref, cow_per_seq=True)
    assert (b.prefix_lens > 0).any()
    pool = _quantised(b) if pool_kind == "quantised" else _random_codes(b, 271)
    kc, vc, sc = _dev(pool)
    out = lib.pa_decode_shared_prefix_e5m2(b.q.cuda(), kc, vc, sc, torch.from_numpy(b.block_tables).cuda(),
                                           torch.from_numpy(b.kv_lens).cuda(), b.max_seq_len,
                                           torch.from_numpy(b.group_starts).cuda(),
                                           torch.from_numpy(b.prefix_lens).cuda(), b.scale,
                                           partition_size=partition * (B // 16))
    assert lib.pa_get_status() == 0
    assert_attention_close(to_f64(out), _oracle_decode_rows(b, *pool), dtype, f"{case} vs oracle")


@pytest.mark.slow
def test_llama3_70b_prefix_config_e5m2_shared_prefix(lib):
    """The full 70B prefix-sharing batch on a synthetic e5m2 pool through the
    step: every sequence against the oracle."""
    from paged_kv_cache_14_gb300.step import step_from_host
    b = full_config("llama3_70b_prefix_bf16")
    pool = tuple(x.numpy() for x in e5m2_pool(b.meta["seed"], b.num_blocks, b.num_kv_heads, b.block_size,
                                               b.head_dim))
    st = step_from_host(b, shared_prefix=True, fp8_pool=tuple(torch.from_numpy(x) for x in pool), kv_format="e5m2")
    out = to_f64(st.run())
    assert lib.pa_get_status() == 0
    ko, vo, so = _oracle_step_pools(b, pool)
    assert_attention_close(out, _oracle_decode_rows(b, ko, vo, so), "bf16", "70B e5m2 shared prefix, every sequence")


# ---------------------------------------------------------------------------
# Chunked prefill
# ---------------------------------------------------------------------------

PF_CASES = [
    # dtype, B, Hq, Hkv, q_lens, ctx_lens
    ("f16", 32, 64, 8, [2, 17, 1, 100], [0, 5, 40, 63]),
    ("bf16", 16, 64, 8, [16, 33, 1, 129], [64, 0, 3, 200]),
    ("f16", 16, 8, 8, [130, 5], [1, 300]),               # group 1: 128 positions per tile
    ("bf16", 32, 64, 8, [512, 1, 1], [1000, 700, 30]),  # a long chunk over a long context
]


@pytest.mark.parametrize("pool_kind", ["quantised", "random"])
@pytest.mark.parametrize("case", PF_CASES, ids=lambda c: f"{c[0]}-B{c[1]}-G{c[2] // c[3]}-q{sum(c[4])}")
def test_chunked_prefill_e5m2_matches_oracle(lib, case, pool_kind):
    dtype, B, hq, hkv, qls, ctxs = case
    kv = [c + q for c, q in zip(ctxs, qls)]
    b = build_batch(name="pf_e5m2", seed=PF_CASES.index(case) + 290, dtype=dtype, block_size=B, num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=128, q_lens=qls, kv_lens=kv)
    pool = _quantised(b) if pool_kind == "quantised" else _random_codes(b, 291)
    kc, vc, sc = _dev(pool)
    out = lib.pa_chunked_prefill_e5m2(b.q.cuda(), torch.from_numpy(b.cu_q_lens).cuda(), kc, vc, sc,
                                      torch.from_numpy(b.block_tables).cuda(), torch.from_numpy(b.ctx_lens).cuda(),
                                      b.max_q_len, b.max_seq_len, b.scale)
    st = lib.pa_get_status()
    assert st == 0, lib.pa_strerror(st)
    kd = f8.dequantize_e5m2(pool[0], pool[2][..., 0])
    vd = f8.dequantize_e5m2(pool[1], pool[2][..., 1])
    ref = oracle.prefill(b.q, b.cu_q_lens, b.ctx_lens, kd, vd, b.block_tables, b.scale, b.block_size)
    assert_attention_close(to_f64(out), ref, dtype, f"{case} {pool_kind}")
