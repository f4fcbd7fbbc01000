"""Slot derivation, cache write and copy-on-write copies on the GPU: bit-exact
against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from workloads import build_batch

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("block_size", [16, 32])
def test_slot_mapping_and_cache_write_bit_exact(lib, dtype, block_size):
    b = build_batch(name="cw", seed=31, dtype=dtype, block_size=block_size, num_q_heads=8, num_kv_heads=4,
                    head_dim=128 if dtype != "f32" else 64, q_lens=[1, 3, 17, 1, 40],
                    kv_lens=[1, 20, 17, 65, 100])
    dev = "cuda"
    bt = torch.from_numpy(b.block_tables).to(dev)
    sid = torch.from_numpy(b.new_seq_ids).to(dev)
    pos = torch.from_numpy(b.new_positions).to(dev)
    slots = lib.pa_slot_mapping(bt, sid, pos, block_size, b.num_blocks)
    ref_slots = oracle.slot_mapping(b.block_tables, b.new_seq_ids, b.new_positions, block_size)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    # Padding tokens (slot -1) are skipped.
    slots_pad = torch.cat([slots, torch.tensor([-1, -1], device=dev, dtype=torch.int64)])
    kn = torch.cat([b.k_new, torch.full((2,) + b.k_new.shape[1:], 9.0).to(b.k_new.dtype)]).to(dev)
    vn = torch.cat([b.v_new, torch.full((2,) + b.v_new.shape[1:], 9.0).to(b.v_new.dtype)]).to(dev)
    kc = b.k_cache.to(dev)
    vc = b.v_cache.to(dev)
    lib.pa_reshape_and_cache(kn, vn, slots_pad, kc, vc)
    assert lib.pa_get_status() == 0
    kr, vr = b.k_cache.clone(), b.v_cache.clone()
    oracle.reshape_and_cache(b.k_new, b.v_new, ref_slots, kr, vr, block_size)
    assert torch.equal(_bits(kc.cpu()), _bits(kr)) and torch.equal(_bits(vc.cpu()), _bits(vr))


def test_slot_mapping_out_of_range_reports(lib):
    dev = "cuda"
    bt = torch.tensor([[3, 7], [9, 99]], dtype=torch.int32, device=dev)  # 99 is outside a pool of 10
    sid = torch.tensor([0, 1, 1, 0, 2], dtype=torch.int32, device=dev)
    pos = torch.tensor([17, 3, 20, 40, 0], dtype=torch.int32, device=dev)
    slots = lib.pa_slot_mapping(bt, sid, pos, 16, 10)
    assert slots.cpu().tolist() == [7 * 16 + 1, 9 * 16 + 3, -1, -1, -1]
    assert lib.pa_get_status() == -7
    assert lib.pa_get_status() == 0  # cleared


def test_cache_write_out_of_pool_slot_reports_and_skips(lib):
    dev = "cuda"
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    k = torch.ones(2, 2, 64, dtype=torch.bfloat16, device=dev)
    slots = torch.tensor([5, 4 * 16], dtype=torch.int64, device=dev)
    lib.pa_reshape_and_cache(k, k, slots, kc, vc)
    assert lib.pa_get_status() == -7
    assert kc[0, :, 5].eq(1).all() and kc.sum().item() == 2 * 64


@pytest.mark.parametrize("num_pairs", [1, 256, 1500])
def test_copy_blocks_bit_exact(lib, num_pairs):
    rng = np.random.default_rng(num_pairs)
    P = 2 * num_pairs + 40
    kc = torch.from_numpy(rng.standard_normal((P, 8, 16, 128), dtype=np.float32)).to(torch.bfloat16)
    vc = torch.from_numpy(rng.standard_normal((P, 8, 16, 128), dtype=np.float32)).to(torch.bfloat16)
    perm = rng.permutation(P)
    dst = perm[:num_pairs]
    srcs = perm[num_pairs:]
    src = srcs[rng.integers(0, len(srcs), num_pairs)]  # sources may repeat
    pairs = np.stack([src, dst], axis=1).astype(np.int64)
    kd, vd = kc.cuda(), vc.cuda()
    lib.pa_copy_blocks(kd, vd, pairs)
    assert lib.pa_get_status() == 0
    kr, vr = kc.clone(), vc.clone()
    oracle.copy_blocks(kr, vr, pairs)
    assert torch.equal(kd.cpu().view(torch.int16), kr.view(torch.int16))
    assert torch.equal(vd.cpu().view(torch.int16), vr.view(torch.int16))


def test_copy_blocks_alias_rejected_before_launch(lib):
    kc = torch.arange(4 * 2 * 16 * 64, dtype=torch.float32).reshape(4, 2, 16, 64).cuda()
    before = kc.clone()
    with pytest.raises(lib.PagedAttnError) as e:
        lib.pa_copy_blocks(kc, kc, [(0, 1), (1, 2)])
    assert e.value.status == -6
    assert torch.equal(kc, before)
