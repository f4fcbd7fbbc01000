"""e4m3 KV cache on the GPU: the quantising cache write and the copy-on-write
of codes and scales bit for bit against the oracle's rule, and decode
attention over the e4m3 pools against the fp64 oracle on the dequantised
values (each stored value = e4m3 code x its (block, KV head) scale)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import oracle.fp8_kv as f8
from helpers import assert_attention_close, to_f64
from workloads import build_batch, e4m3_pool, make_config

pytestmark = pytest.mark.gpu


def _finite_codes(rng, shape) -> np.ndarray:
    r = rng.integers(0, 254, size=shape)
    return (r + (r >= 0x7F)).astype(np.uint8)


def _f32_bits(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)


def _oracle_fp8_from_batch(b):
    """e4m3 pools of a batch's 16-bit pool values, every block written in
    one call (the oracle's whole-block quantiser)."""
    kc, ks = f8.quantize_fresh_blocks(b.k_cache.float().numpy())
    vc, vs = f8.quantize_fresh_blocks(b.v_cache.float().numpy())
    return kc, vc, np.stack([ks, vs], axis=-1).astype(np.float32)


def _oracle_decode_fp8(b, kc, vc, sc, seqs=None):
    kd = f8.dequantize(kc, sc[..., 0])
    vd = f8.dequantize(vc, sc[..., 1])
    return oracle.decode(b.q, kd, vd, b.block_tables, b.kv_lens, b.scale, b.block_size, seqs=seqs)


# ---------------------------------------------------------------------------
# Cache write
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("D", [64, 128])
def test_cache_write_bit_exact(lib, dtype, B, D):
    rng = np.random.default_rng(B * 1000 + D + len(dtype))
    P, H = 14, 3
    kc0 = _finite_codes(rng, (P, H, B, D))
    vc0 = _finite_codes(rng, (P, H, B, D))
    sc0 = np.exp2(rng.uniform(-10, -3, size=(P, H, 2))).astype(np.float32)
    # Runs: a chunk that starts mid-block and crosses into a fresh block, a
    # padding entry inside a run, single-token appends (some forcing the
    # scale up, some not), a fresh block, a whole block, a full block's tail.
    slots = []
    slots += [3 * B + o for o in range(B // 2, B)] + [7 * B + o for o in range(0, 5)]
    slots += [-1]
    slots += [7 * B + 5, 7 * B + 6]
    slots += [5 * B + 9, -1, 9 * B + 2, 0 * B + 0, 11 * B + B - 1]
    slots += [12 * B + o for o in range(B)]
    slots = np.array(slots, dtype=np.int64)
    T = len(slots)
    mag = np.exp2(rng.uniform(-6, 3, size=(T, 1, 1)))
    mag[np.flatnonzero(slots == 5 * B + 9)] = 3000.0       # forces a larger scale on block 5
    k = torch.from_numpy((rng.standard_normal((T, H, D)) * mag).astype(np.float32)).to(
        {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype])
    v = (k.float() * -0.7 + 0.01).to(k.dtype)
    kd, vd = torch.from_numpy(kc0).cuda(), torch.from_numpy(vc0).cuda()
    sd = torch.from_numpy(sc0).cuda()
    lib.pa_reshape_and_cache_fp8(k.cuda(), v.cuda(), torch.from_numpy(slots).cuda(), kd, vd, sd)
    assert lib.pa_get_status() == 0
    ko, vo, so = kc0.copy(), vc0.copy(), sc0.copy()
    f8.reshape_and_cache_fp8(k.float().numpy(), v.float().numpy(), slots, ko, vo, so, B)
    assert np.array_equal(_f32_bits(sd.cpu().numpy()), _f32_bits(so)), "scales differ"
    assert np.array_equal(kd.cpu().numpy(), ko), "K codes differ"
    assert np.array_equal(vd.cpu().numpy(), vo), "V codes differ"
    assert so[5, 0, 0] > sc0[5, 0, 0]                       # the growth path ran


def test_cache_write_out_of_pool_slot_is_reported(lib):
    rng = np.random.default_rng(3)
    P, H, B, D = 4, 2, 16, 128
    kc0 = _finite_codes(rng, (P, H, B, D))
    kd = torch.from_numpy(kc0).cuda()
    vd = torch.from_numpy(kc0).cuda()
    sd = torch.ones(P, H, 2, device="cuda")
    k = torch.randn(2, H, D, dtype=torch.bfloat16, device="cuda")
    lib.pa_reshape_and_cache_fp8(k, k, torch.tensor([P * B + 3, 1 * B], device="cuda"), kd, vd, sd)
    assert lib.pa_get_status() == -7
    got = kd.cpu().numpy()
    assert np.array_equal(got[[0, 2, 3]], kc0[[0, 2, 3]])   # only block 1 was written


def test_copy_blocks_fp8_bit_exact(lib):
    rng = np.random.default_rng(4)
    P, H, B, D = 10, 2, 16, 128
    kc0, vc0 = _finite_codes(rng, (P, H, B, D)), _finite_codes(rng, (P, H, B, D))
    sc0 = rng.uniform(0.001, 0.1, size=(P, H, 2)).astype(np.float32)
    pairs = np.array([[1, 4], [1, 6], [8, 2]], dtype=np.int64)
    kd, vd, sd = (torch.from_numpy(x).cuda() for x in (kc0, vc0, sc0))
    lib.pa_copy_blocks_fp8(kd, vd, sd, pairs)
    assert lib.pa_get_status() == 0
    ko, vo, so = kc0.copy(), vc0.copy(), sc0.copy()
    f8.copy_blocks_fp8(ko, vo, so, pairs)
    assert np.array_equal(kd.cpu().numpy(), ko) and np.array_equal(vd.cpu().numpy(), vo)
    assert np.array_equal(_f32_bits(sd.cpu().numpy()), _f32_bits(so))


# ---------------------------------------------------------------------------
# Decode
# ---------------------------------------------------------------------------

CASES = [
    # dtype, B, Hq, Hkv, lens
    ("bf16", 16, 8, 1, [1, 15, 16, 17, 33, 200]),
    ("bf16", 16, 32, 8, [1, 2, 300, 1000]),
    ("bf16", 32, 64, 8, [1, 31, 32, 33, 513, 1025]),
    ("f16", 16, 16, 2, [1, 17, 160, 999]),
    ("f16", 32, 32, 2, [5, 64, 65, 2000]),
    ("bf16", 16, 32, 1, [9, 70]),       # group 32: two row groups per KV head
]


def _decode_fp8(lib, b, pool, partition=0):
    kc, vc, sc = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in pool)
    out = lib.pa_decode_fp8(b.q.cuda(), kc, vc, sc, torch.from_numpy(b.block_tables).cuda(),
                            torch.from_numpy(b.kv_lens.astype(np.int32)).cuda(), b.max_seq_len, b.scale,
                            partition_size=partition)
    st = lib.pa_get_status()
    assert st == 0, lib.pa_strerror(st)
    return to_f64(out)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-B{c[1]}-Hq{c[2]}-Hkv{c[3]}")
@pytest.mark.parametrize("partition", [0, 1, 3])
def test_decode_fp8_matches_oracle(lib, case, partition):
    dtype, B, hq, hkv, lens = case
    b = build_batch(name="fp8", seed=CASES.index(case) + 40, dtype=dtype, block_size=B, num_q_heads=hq,
                    num_kv_heads=hkv, head_dim=128, q_lens=np.ones(len(lens), np.int32), kv_lens=lens)
    pool = _oracle_fp8_from_batch(b)
    out = _decode_fp8(lib, b, pool, partition * B)
    ref = _oracle_decode_fp8(b, *pool)
    assert_attention_close(out, ref, dtype, f"{case} partition {partition}")


def test_decode_fp8_wide_scale_range(lib):
    """Codes uniform over every finite e4m3 value (subnormals included) and
    per-block scales over three binades: the fp16 widening, the per-block
    score and V scales and the power-of-two rescaling of the accumulator all
    get exercised."""
    lens = [3, 16, 77, 500, 1500]
    b = build_batch(name="fp8w", seed=61, dtype="bf16", block_size=16, num_q_heads=64, num_kv_heads=8,
                    head_dim=128, q_lens=np.ones(len(lens), np.int32), kv_lens=lens, with_values=True)
    kc, vc, sc = e4m3_pool(61, b.num_blocks, 8, 16, 128)
    pool = (kc.numpy(), vc.numpy(), sc.numpy())
    for part in (0, 64):
        out = _decode_fp8(lib, b, pool, part)
        assert_attention_close(out, _oracle_decode_fp8(b, *pool), "bf16", f"partition {part}")


def test_decode_fp8_ignores_nan_codes_past_the_end(lib):
    lens = [5, 17, 40]
    b = build_batch(name="fp8nan", seed=62, dtype="f16", block_size=16, num_q_heads=16, num_kv_heads=2,
                    head_dim=128, q_lens=np.ones(3, np.int32), kv_lens=lens)
    kc, vc, sc = _oracle_fp8_from_batch(b)
    clean = _decode_fp8(lib, b, (kc, vc, sc))
    kn, vn = kc.copy(), vc.copy()
    for i, L in enumerate(lens):
        last = b.block_tables[i][(L - 1) // 16]
        kn[last, :, L % 16 or 16:, :] = 0x7F
        vn[last, :, L % 16 or 16:, :] = 0xFF
    dirty = _decode_fp8(lib, b, (kn, vn, sc))
    assert np.array_equal(clean, dirty)
    assert_attention_close(dirty, _oracle_decode_fp8(b, kc, vc, sc), "f16", "NaN codes past the end")


def test_step_fp8_matches_oracle(lib):
    """The whole step on an e4m3 cache: copy-on-write of codes and scales,
    slot mapping, the quantising cache write of the new tokens (appends into
    partly filled blocks) and decode, against the oracle applying the same
    rule to its own copy of the pools."""
    from paged_kv_cache_14_gb300.step import step_from_host
    lens = [5, 64, 300, 700, 1300, 31, 900, 17]
    b = build_batch(name="fp8step", seed=63, dtype="bf16", block_size=16, num_q_heads=64, num_kv_heads=8,
                    head_dim=128, q_lens=np.ones(8, np.int32), kv_lens=lens, share_group=4,
                    share_prefix_tokens=256, cow_per_seq=True)
    kc, vc, sc = _oracle_fp8_from_batch(b)
    st = step_from_host(b, fp8_pool=(torch.from_numpy(kc), torch.from_numpy(vc), torch.from_numpy(sc)))
    out = to_f64(st.run())
    assert lib.pa_get_status() == 0
    ko, vo, so = kc.copy(), vc.copy(), sc.copy()
    f8.copy_blocks_fp8(ko, vo, so, b.cow_pairs)
    slots = oracle.slot_mapping(b.block_tables, b.new_seq_ids, b.new_positions, b.block_size)
    f8.reshape_and_cache_fp8(b.k_new.float().numpy(), b.v_new.float().numpy(), slots, ko, vo, so, b.block_size)
    assert np.array_equal(st.k_cache.cpu().numpy(), ko) and np.array_equal(st.v_cache.cpu().numpy(), vo)
    assert np.array_equal(_f32_bits(st.kv_scales.cpu().numpy()), _f32_bits(so))
    assert_attention_close(out, _oracle_decode_fp8(b, ko, vo, so), "bf16", "fp8 step")
    # The e4m3 cache stays close to the 16-bit one: a quantisation error (at
    # most 2^-4 of each stored value), not a parity bound.
    ref16 = oracle.decode(b.q, *_caches16(b), b.block_tables, b.kv_lens, b.scale, b.block_size)
    assert np.abs(out - ref16).max() < 0.3 and np.abs(out - ref16).mean() < 0.01


def _caches16(b):
    from helpers import oracle_caches_after_step
    kc, vc, _ = oracle_caches_after_step(b)
    return kc, vc


@pytest.mark.slow
def test_llama3_8b_config_fp8(lib):
    """Full-size 8B decode batch on a synthetic e4m3 pool, at the launch
    configuration the bench times, against the oracle on every sequence
    (each sequence's blocks dequantised exactly, one sequence at a time)."""
    b = make_config("llama3_8b_bf16")
    kc, vc, sc = e4m3_pool(1, b.num_blocks, b.num_kv_heads, b.block_size, b.head_dim)
    pool = (kc.numpy(), vc.numpy(), sc.numpy())
    out = _decode_fp8(lib, b, pool)
    ref = np.full(out.shape, np.nan)
    for i in range(b.num_seqs):
        nb = -(-int(b.kv_lens[i]) // b.block_size)
        blocks = b.block_tables[i][:nb]
        kd = f8.dequantize(pool[0][blocks], pool[2][blocks, :, 0])
        vd = f8.dequantize(pool[1][blocks], pool[2][blocks, :, 1])
        tables = np.zeros_like(b.block_tables)
        tables[i, :nb] = np.arange(nb)
        ref[i] = oracle.decode(b.q, kd, vd, tables, b.kv_lens, b.scale, b.block_size, seqs=[i])[i]
    assert_attention_close(out, ref, "bf16", "8B fp8, every sequence")
