"""Seeded synthetic inputs for paged KV-cache attention.

This module is shared by the CUDA path's tests and bench and by the CPU
oracle. It draws only *structure* (sequence lengths, which physical block each
logical block of a sequence uses, which blocks a group of sequences shares,
copy-on-write pairs, the positions of the new tokens) and *values* (normal
random numbers cast to the I/O dtype). It holds none of the method's
arithmetic: no token position is ever turned into a slot here. The physical
pool is filled with random values block by block, so whatever position a
block table makes a block stand for, its contents are the sequence's K/V at
those positions.

The workload shapes follow the Llama-3 layer shapes the pages use for sizing
("Inside vLLM: Anatomy of a High-Throughput LLM Inference System", section
"The KV-Cache Bottleneck": 70B with 8 KV heads of dimension 128) and the
block sizes 16 and 32 named there ("Physical Block Mapping and Kernel
Invocation"). No model weights are involved.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class PagedBatch:
    """One batch of sequences over one paged KV pool (CPU tensors).

    Layout conventions (the same on both sides of every parity test):
      k_cache, v_cache : [num_blocks, num_kv_heads, block_size, head_dim]
      q                : [sum(q_lens), num_q_heads, head_dim]; the rows of
                         sequence i are cu_q_lens[i] .. cu_q_lens[i+1]-1
      block_tables     : int32 [num_seqs, max_blocks_per_seq]; entries past a
                         sequence's last logical block are 0 (a valid block)
      kv_lens          : int32 [num_seqs]; keys the sequence's LAST query row
                         attends to once its new tokens are cached
      q_lens           : int32 [num_seqs]; 1 for a decode row
      k_new, v_new     : [num_new, num_kv_heads, head_dim], the K/V of the new
                         tokens, to be cached at (new_seq_ids, new_positions)
      cow_pairs        : int64 [n, 2] (src, dst) whole-block copies that must
                         run before the new tokens are cached; block_tables
                         already point at the dst blocks
    """

    name: str
    dtype: str
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    scale: float
    num_blocks: int
    block_tables: np.ndarray
    q_lens: np.ndarray
    kv_lens: np.ndarray
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    new_seq_ids: np.ndarray
    new_positions: np.ndarray
    cow_pairs: np.ndarray
    meta: dict = field(default_factory=dict)
    # Prefix-sharing structure: group g is sequences group_starts[g] ..
    # group_starts[g+1]-1; sequence i's first prefix_lens[i] tokens use the
    # group's shared physical blocks (after its copy-on-write). Without
    # sharing every sequence is its own group with prefix 0.
    group_starts: np.ndarray | None = None
    prefix_lens: np.ndarray | None = None

    @property
    def num_seqs(self) -> int:
        return int(self.kv_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def ctx_lens(self) -> np.ndarray:
        return (self.kv_lens - self.q_lens).astype(np.int32)

    @property
    def cu_q_lens(self) -> np.ndarray:
        out = np.zeros(self.num_seqs + 1, dtype=np.int32)
        np.cumsum(self.q_lens, out=out[1:])
        return out

    @property
    def is_decode(self) -> bool:
        return bool(np.all(self.q_lens == 1))

    @property
    def max_seq_len(self) -> int:
        return int(self.kv_lens.max()) if self.num_seqs else 0

    @property
    def max_q_len(self) -> int:
        return int(self.q_lens.max()) if self.num_seqs else 0

    @property
    def torch_dtype(self) -> torch.dtype:
        return TORCH_DTYPES[self.dtype]


def _normal(rng: np.random.Generator, shape, dtype: str, chunk: int = 1 << 26) -> torch.Tensor:
    """N(0, 1) float32 draws cast (round to nearest even) to the I/O dtype."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(n, dtype=TORCH_DTYPES[dtype])
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = torch.from_numpy(rng.standard_normal(e - s, dtype=np.float32))
    return out.view(*shape)


def _blocks_for(length: int, block_size: int) -> int:
    # Number of logical blocks a sequence of `length` tokens occupies.
    return -(-int(length) // block_size)


def build_batch(
    *,
    name: str,
    seed: int,
    dtype: str,
    block_size: int,
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    q_lens,
    kv_lens,
    scale: float | None = None,
    pool_size: int | None = None,
    free_frac: float = 0.10,
    share_group: int = 0,
    share_prefix_tokens: int = 0,
    cow_per_seq: bool = False,
    hot_key_frac: float = 0.0,
    hot_key_scale: float = 8.0,
    with_values: bool = True,
) -> PagedBatch:
    """Draw one paged batch.

    Structure: sequence i owns ceil(kv_lens[i] / B) logical blocks. With
    `share_group` > 0, consecutive groups of that many sequences share the
    physical blocks of a `share_prefix_tokens`-token prefix (a block-aligned
    prefix, so every shared block is full); a sequence shorter than the prefix
    uses only the prefix blocks it covers. With `cow_per_seq`, each sequence
    gets one copy-on-write pair: the last prefix block it shares is copied to
    a fresh block and its table is repointed there (refcount of the shared
    block drops by one). Physical ids are a seeded permutation of a pool of
    `pool_size` blocks (default: distinct blocks needed plus `free_frac`).

    Values: q, the pool and the new tokens' K/V are N(0, 1). With
    `hot_key_frac` > 0, that fraction of the pool's token slots (all heads)
    and of the new tokens get their K scaled by `hot_key_scale`.
    """
    q_lens = np.asarray(q_lens, dtype=np.int32).copy()
    kv_lens = np.asarray(kv_lens, dtype=np.int32).copy()
    n = int(kv_lens.shape[0])
    assert q_lens.shape == (n,)
    assert np.all(q_lens >= 1) and np.all(kv_lens >= q_lens)
    B = int(block_size)
    assert num_q_heads % num_kv_heads == 0
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)

    ss = np.random.SeedSequence(seed)
    rng_struct, rng_q, rng_k, rng_v, rng_kn, rng_vn, rng_hot = [np.random.default_rng(s) for s in ss.spawn(7)]

    nblk = np.array([_blocks_for(L, B) for L in kv_lens], dtype=np.int64)
    max_blocks = int(nblk.max()) if n else 1

    # Which logical blocks are shared (owner group) and which are private.
    prefix_blocks = 0
    n_groups = 0
    if share_group:
        assert share_prefix_tokens % B == 0
        prefix_blocks = share_prefix_tokens // B
        n_groups = -(-n // share_group)
    shared_counts = np.minimum(nblk, prefix_blocks) if share_group else np.zeros(n, np.int64)
    private_counts = nblk - shared_counts
    n_cow = n if (share_group and cow_per_seq) else 0
    need = int(n_groups * prefix_blocks + private_counts.sum() + n_cow)
    if pool_size is None:
        pool_size = int(math.ceil((1.0 + free_frac) * need))
    assert pool_size >= need, (pool_size, need)

    ids = rng_struct.permutation(pool_size).astype(np.int32)
    cursor = 0

    def take(k: int) -> np.ndarray:
        nonlocal cursor
        out = ids[cursor:cursor + k]
        cursor += k
        return out

    group_blocks = [take(prefix_blocks) for _ in range(n_groups)]
    tables = np.zeros((n, max_blocks), dtype=np.int32)
    for i in range(n):
        s = int(shared_counts[i])
        if s:
            tables[i, :s] = group_blocks[i // share_group][:s]
        tables[i, s:nblk[i]] = take(int(private_counts[i]))
    cow = np.zeros((0, 2), dtype=np.int64)
    if n_cow:
        pairs = []
        for i in range(n):
            # Last logical block this sequence shares with its group.
            c = int(shared_counts[i]) - 1
            src = int(tables[i, c])
            dst = int(take(1)[0])
            tables[i, c] = dst
            pairs.append((src, dst))
        cow = np.asarray(pairs, dtype=np.int64)

    # New tokens: the last q_len positions of every sequence.
    new_seq_ids = np.repeat(np.arange(n, dtype=np.int32), q_lens)
    new_positions = np.concatenate(
        [np.arange(kv_lens[i] - q_lens[i], kv_lens[i], dtype=np.int32) for i in range(n)]
    ) if n else np.zeros(0, np.int32)
    t_new = int(q_lens.sum())

    cache_shape = (pool_size, num_kv_heads, B, head_dim)
    if with_values:
        q = _normal(rng_q, (t_new, num_q_heads, head_dim), dtype)
        k_cache = _normal(rng_k, cache_shape, dtype)
        v_cache = _normal(rng_v, cache_shape, dtype)
        k_new = _normal(rng_kn, (t_new, num_kv_heads, head_dim), dtype)
        v_new = _normal(rng_vn, (t_new, num_kv_heads, head_dim), dtype)
        if hot_key_frac > 0:
            hot = torch.from_numpy(rng_hot.random((pool_size, B)) < hot_key_frac)
            factor = torch.where(hot, hot_key_scale, 1.0).to(k_cache.dtype)
            k_cache.mul_(factor[:, None, :, None])
            hot_new = rng_hot.random(t_new) < hot_key_frac
            k_new[torch.from_numpy(hot_new)] *= hot_key_scale
    else:
        td = TORCH_DTYPES[dtype]
        q = torch.empty((t_new, num_q_heads, head_dim), dtype=td)
        k_cache = torch.empty(cache_shape, dtype=td)
        v_cache = torch.empty(cache_shape, dtype=td)
        k_new = torch.empty((t_new, num_kv_heads, head_dim), dtype=td)
        v_new = torch.empty((t_new, num_kv_heads, head_dim), dtype=td)

    if share_group:
        group_starts = np.minimum(np.arange(0, n_groups + 1) * share_group, n).astype(np.int32)
        # Blocks still shared after the copy-on-write of the last shared one.
        shared_after = shared_counts - (1 if n_cow else 0)
        prefix_lens = (shared_after * B).astype(np.int32)
    else:
        group_starts = np.arange(0, n + 1, dtype=np.int32)
        prefix_lens = np.zeros(n, dtype=np.int32)

    meta = dict(
        seed=seed, need_blocks=need, share_group=share_group,
        share_prefix_tokens=share_prefix_tokens, hot_key_frac=hot_key_frac,
        group_blocks=[g.tolist() for g in group_blocks] if n_groups and n_groups <= 64 else None,
    )
    return PagedBatch(
        name=name, dtype=dtype, block_size=B, num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, scale=float(scale),
        num_blocks=pool_size, block_tables=tables, q_lens=q_lens, kv_lens=kv_lens,
        q=q, k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
        new_seq_ids=new_seq_ids, new_positions=new_positions, cow_pairs=cow, meta=meta,
        group_starts=group_starts, prefix_lens=prefix_lens,
    )


# ---------------------------------------------------------------------------
# The five named workloads.
# ---------------------------------------------------------------------------

CONFIG_NAMES = (
    "tiny_fp32",
    "llama3_8b_bf16",
    "llama3_70b_prefix_bf16",
    "long_splitkv_bf16",
    "mixed_prefill_fp16",
)


def tiny_fp32(with_values: bool = True) -> PagedBatch:
    """4 sequences {1, 15, 16, 33}, B=16, 2 query heads / 1 KV head, D=64,
    a pool of 32 blocks placed by a seeded permutation, fp32, seed 0."""
    return build_batch(
        name="tiny_fp32", seed=0, dtype="f32", block_size=16, num_q_heads=2,
        num_kv_heads=1, head_dim=64, q_lens=[1, 1, 1, 1], kv_lens=[1, 15, 16, 33],
        scale=1.0 / 8.0, pool_size=32, with_values=with_values,
    )


def llama3_8b_bf16(with_values: bool = True) -> PagedBatch:
    """Batch 64, 32 query / 8 KV heads, D=128, B=16, seq_lens U[128, 4096],
    pool = need + 10% shuffled, bf16, seed 1."""
    rng = np.random.default_rng(np.random.SeedSequence(1001))
    lens = rng.integers(128, 4096, size=64, endpoint=True)
    return build_batch(
        name="llama3_8b_bf16", seed=1, dtype="bf16", block_size=16, num_q_heads=32,
        num_kv_heads=8, head_dim=128, q_lens=np.ones(64, np.int32), kv_lens=lens,
        with_values=with_values,
    )


def llama3_70b_prefix_bf16(with_values: bool = True) -> PagedBatch:
    """Batch 256, 64 query / 8 KV heads, D=128, B=16, seq_lens log-uniform in
    [512, 8192]; groups of 16 share a 1024-token prefix (refcount 16); one
    copy-on-write of the last shared block per sequence; bf16, seed 2."""
    rng = np.random.default_rng(np.random.SeedSequence(1002))
    lens = np.floor(np.exp(rng.uniform(math.log(512), math.log(8192), size=256))).astype(np.int32)
    return build_batch(
        name="llama3_70b_prefix_bf16", seed=2, dtype="bf16", block_size=16,
        num_q_heads=64, num_kv_heads=8, head_dim=128, q_lens=np.ones(256, np.int32),
        kv_lens=lens, share_group=16, share_prefix_tokens=1024, cow_per_seq=True,
        with_values=with_values,
    )


def long_splitkv_bf16(with_values: bool = True) -> PagedBatch:
    """Batch 8, 64 query / 8 KV heads, D=128, B=16, seq_lens U[32768, 131072],
    shuffled blocks; 1% of K token slots scaled x8; bf16, seed 3."""
    rng = np.random.default_rng(np.random.SeedSequence(1003))
    lens = rng.integers(32768, 131072, size=8, endpoint=True)
    return build_batch(
        name="long_splitkv_bf16", seed=3, dtype="bf16", block_size=16,
        num_q_heads=64, num_kv_heads=8, head_dim=128, q_lens=np.ones(8, np.int32),
        kv_lens=lens, hot_key_frac=0.01, hot_key_scale=8.0, with_values=with_values,
    )


def mixed_prefill_fp16(with_values: bool = True) -> PagedBatch:
    """96 decode rows (q_len 1, prior context U[1024, 8192]) then 8 prefill
    chunks (q_len 512, prior context U[0, 16384]); 64 query / 8 KV heads,
    D=128, B=32, fp16, seed 4. A decode row with prior context c attends to
    c + 1 keys (its own new token included)."""
    rng = np.random.default_rng(np.random.SeedSequence(1004))
    dec_ctx = rng.integers(1024, 8192, size=96, endpoint=True)
    chunk_ctx = rng.integers(0, 16384, size=8, endpoint=True)
    q_lens = np.concatenate([np.ones(96, np.int32), np.full(8, 512, np.int32)])
    kv_lens = np.concatenate([dec_ctx + 1, chunk_ctx + 512]).astype(np.int32)
    return build_batch(
        name="mixed_prefill_fp16", seed=4, dtype="f16", block_size=32,
        num_q_heads=64, num_kv_heads=8, head_dim=128, q_lens=q_lens, kv_lens=kv_lens,
        with_values=with_values,
    )


CONFIGS = {
    "tiny_fp32": tiny_fp32,
    "llama3_8b_bf16": llama3_8b_bf16,
    "llama3_70b_prefix_bf16": llama3_70b_prefix_bf16,
    "long_splitkv_bf16": long_splitkv_bf16,
    "mixed_prefill_fp16": mixed_prefill_fp16,
}


def make_config(name: str, with_values: bool = True) -> PagedBatch:
    return CONFIGS[name](with_values=with_values)


def e4m3_pool(seed: int, num_blocks: int, num_kv_heads: int, block_size: int, head_dim: int,
              log2_scale_range: tuple[float, float] = (-10.0, -7.0)):
    """A synthetic e4m3 KV pool drawn directly as codes: K and V codes uniform
    over the 254 byte values that are not e4m3 NaN patterns (0x7F, 0xFF), and
    one K and one V scale per (block, KV head), log-uniform over
    2^log2_scale_range (the default keeps stored magnitudes below 448 * 2^-7
    = 3.5, like unit-normal data).
    Returns (k_codes, v_codes) uint8 [P, Hkv, B, D] and kv_scales float32
    [P, Hkv, 2] (CPU tensors). Random structure only: no value is encoded."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 4093]))
    shape = (num_blocks, num_kv_heads, block_size, head_dim)

    def codes():
        r = rng.integers(0, 254, size=shape, dtype=np.int32)   # 0..253
        r = r + (r >= 0x7F)                                      # skip 0x7F; 0xFF is never reached
        return torch.from_numpy(r.astype(np.uint8))

    k, v = codes(), codes()
    lo, hi = log2_scale_range
    sc = np.exp2(rng.uniform(lo, hi, size=(num_blocks, num_kv_heads, 2))).astype(np.float32)
    return k, v, torch.from_numpy(sc)


def e5m2_pool(seed: int, num_blocks: int, num_kv_heads: int, block_size: int, head_dim: int,
              log2_scale_range: tuple[float, float] = (-17.0, -14.0)):
    """A synthetic e5m2 KV pool drawn directly as codes: K and V codes uniform
    over the 248 byte values whose exponent field is not all ones (e5m2's
    infinities and NaNs), and one K and one V scale per (block, KV head),
    log-uniform over 2^log2_scale_range (the default keeps stored magnitudes
    below 57344 * 2^-14 = 3.5, like unit-normal data).
    Returns (k_codes, v_codes) uint8 [P, Hkv, B, D] and kv_scales float32
    [P, Hkv, 2] (CPU tensors). Random structure only: no value is encoded."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 5011]))
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    finite = np.array([c for c in range(256) if (c >> 2) & 0x1F != 0x1F], dtype=np.uint8)

    def codes():
        return torch.from_numpy(finite[rng.integers(0, finite.size, size=shape)])

    k, v = codes(), codes()
    lo, hi = log2_scale_range
    sc = np.exp2(rng.uniform(lo, hi, size=(num_blocks, num_kv_heads, 2))).astype(np.float32)
    return k, v, torch.from_numpy(sc)


def random_lengths(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """Uniform integer lengths in [lo, hi] (structure helper for small cases)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 77]))
    return rng.integers(lo, hi, size=n, endpoint=True).astype(np.int32)
