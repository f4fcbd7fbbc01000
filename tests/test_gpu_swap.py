"""Swap preemption on the GPU: whole blocks between device pools and pinned
host pools, bit for bit against the oracle, and decode over swapped-back
blocks identical to decode before the swap."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from helpers import to_f64
from workloads import build_batch, e4m3_pool

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    return t.view(torch.uint8).numpy() if t.dtype != torch.uint8 else t.numpy()


def test_swap_out_and_back_bit_exact(lib):
    lens = [300, 700, 45, 1000]
    b = build_batch(name="swap", seed=95, dtype="bf16", block_size=16, num_q_heads=32, num_kv_heads=8,
                    head_dim=128, q_lens=np.ones(4, np.int32), kv_lens=lens, pool_size=200)
    kd, vd = b.k_cache.cuda(), b.v_cache.cuda()
    q, bt = b.q.cuda(), torch.from_numpy(b.block_tables).cuda()
    sl = torch.from_numpy(b.kv_lens.astype(np.int32)).cuda()
    before = lib.pa_decode(q, kd, vd, bt, sl, b.max_seq_len, b.scale).clone()
    # Swap sequence 1 out to a pinned host pool of 80 blocks, at scattered slots.
    nb = -(-lens[1] // 16)
    used = b.block_tables[1][:nb].astype(np.int64)
    rng = np.random.default_rng(5)
    slots = rng.choice(80, nb, replace=False)
    hk = torch.zeros((80,) + tuple(kd.shape[1:]), dtype=kd.dtype).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    out_pairs = np.stack([used, slots], 1)
    lib.pa_swap_blocks(kd, vd, hk, hv, out_pairs)
    torch.cuda.synchronize()
    assert lib.pa_get_status() == 0
    ok, ov = np.zeros(hk.shape, np.float32), np.zeros(hv.shape, np.float32)
    oracle.swap_blocks(b.k_cache.float().numpy(), b.v_cache.float().numpy(), ok, ov, out_pairs)
    ut = torch.from_numpy(used)
    assert np.array_equal(_bits(hk[torch.from_numpy(slots)]), _bits(b.k_cache[ut]))
    st_ = torch.from_numpy(slots)
    assert np.array_equal(hk[st_].float().numpy(), ok[slots]) and np.array_equal(hv[st_].float().numpy(), ov[slots])
    # The device blocks are reused meanwhile; bring the sequence back into free blocks.
    kd[torch.from_numpy(used).cuda()] = float("nan")
    vd[torch.from_numpy(used).cuda()] = float("nan")
    live = set(np.concatenate([b.block_tables[i][: -(-lens[i] // 16)] for i in range(4)]).tolist())
    free = np.array([p for p in range(b.num_blocks) if p not in live], np.int64)
    if free.size < nb:
        pytest.skip("pool too small")
    new = rng.choice(free, nb, replace=False)
    lib.pa_swap_blocks(hk, hv, kd, vd, np.stack([slots, new], 1))
    assert lib.pa_get_status() == 0
    assert np.array_equal(_bits(kd[torch.from_numpy(new).cuda()]), _bits(b.k_cache[ut]))
    assert np.array_equal(_bits(vd[torch.from_numpy(new).cuda()]), _bits(b.v_cache[ut]))
    t2 = b.block_tables.copy()
    t2[1][:nb] = new
    after = lib.pa_decode(q, kd, vd, torch.from_numpy(t2).cuda(), sl, b.max_seq_len, b.scale)
    assert torch.equal(before[1], after[1]) and torch.equal(before[0], after[0])


def test_swap_e4m3_codes_and_scales(lib):
    P, H, B, D = 24, 1, 16, 128            # one KV head: 8-byte scale blocks take the 4-byte path
    kc, vc, sc = e4m3_pool(3, P, H, B, D)
    kd, vd, sd = kc.cuda(), vc.cuda(), sc.cuda()
    hk = torch.zeros((10, H, B, D), dtype=torch.uint8).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    hs = torch.zeros((10, H, 2), dtype=torch.float32).pin_memory()
    pairs = np.array([[3, 0], [17, 9], [5, 4]])
    lib.pa_swap_blocks(kd, vd, hk, hv, pairs)
    lib.pa_swap_blocks(sd, None, hs, None, pairs)
    torch.cuda.synchronize()
    assert lib.pa_get_status() == 0
    for s_, d in pairs:
        assert torch.equal(hk[d], kc[s_]) and torch.equal(hv[d], vc[s_]) and torch.equal(hs[d], sc[s_])


def test_swap_device_to_device_and_errors(lib):
    P, H, B, D = 12, 2, 32, 64
    src = torch.randn(P, H, B, D, dtype=torch.float16, device="cuda")
    dst = torch.zeros(6, H, B, D, dtype=torch.float16, device="cuda")
    lib.pa_swap_blocks(src, None, dst, None, [[11, 0], [0, 5]])
    assert torch.equal(dst[0], src[11]) and torch.equal(dst[5], src[0])
    pageable = torch.zeros(6, H, B, D, dtype=torch.float16)
    with pytest.raises(TypeError):
        lib.pa_swap_blocks(src, None, pageable, None, [[1, 1]])
    with pytest.raises(lib.PagedAttnError):
        lib.pa_swap_blocks(src, None, dst, None, [[12, 1]])


@pytest.mark.slow
def test_swap_bandwidth_report(lib, capsys):
    """Swap-out and swap-in of 4096 blocks of 32 KB (a 70B layer's K and V
    blocks at bf16, B = 16): bit-exact, and the rate against one large
    cudaMemcpy of the same bytes."""
    P, H, B, D = 4096, 8, 16, 128
    kd = torch.randint(-30000, 30000, (P, H, B, D), dtype=torch.int16, device="cuda").view(torch.bfloat16)
    vd = torch.randint(-30000, 30000, (P, H, B, D), dtype=torch.int16, device="cuda").view(torch.bfloat16)
    hk = torch.empty_like(kd, device="cpu").pin_memory()
    hv = torch.empty_like(vd, device="cpu").pin_memory()
    perm = np.random.default_rng(1).permutation(P)
    pairs = np.stack([np.arange(P), perm], 1)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    lib.pa_swap_blocks(kd, vd, hk, hv, pairs)  # warm
    ev[0].record()
    lib.pa_swap_blocks(kd, vd, hk, hv, pairs)
    ev[1].record()
    k2, v2 = torch.empty_like(kd), torch.empty_like(vd)
    ev[2].record()
    lib.pa_swap_blocks(hk, hv, k2, v2, np.stack([perm, np.arange(P)], 1))
    ev[3].record()
    ev[4].record()
    hk.copy_(kd, non_blocking=True)
    hv.copy_(vd, non_blocking=True)
    ev[5].record()
    torch.cuda.synchronize()
    assert torch.equal(k2.view(torch.int16), kd.view(torch.int16)) and torch.equal(v2.view(torch.int16), vd.view(torch.int16))
    nbytes = 2 * kd.numel() * 2
    out_gbs = nbytes / (ev[0].elapsed_time(ev[1]) * 1e-3) / 1e9
    in_gbs = nbytes / (ev[2].elapsed_time(ev[3]) * 1e-3) / 1e9
    cp_gbs = nbytes / (ev[4].elapsed_time(ev[5]) * 1e-3) / 1e9
    with capsys.disabled():
        print(f"\nswap of {nbytes / 1e9:.2f} GB: out {out_gbs:.1f} GB/s, in {in_gbs:.1f} GB/s; "
              f"contiguous device->host copy {cp_gbs:.1f} GB/s")
    assert out_gbs > 0.3 * cp_gbs and in_gbs > 0.3 * cp_gbs
