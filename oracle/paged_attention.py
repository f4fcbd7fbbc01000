"""CPU oracle for paged KV-cache attention.

TEST INFRASTRUCTURE ONLY. Only the test suite, the package smoke check and
the bench's CPU-baseline / reference legs may import this module. The CUDA
library never calls it, and it shares no code with the CUDA library: it
imports numpy and torch (CPU, for exact dtype up-casts) and nothing else.

Everything here is the plain definition, in float64 after an exact up-cast of
the stored values, with no blocking, fusion or reordering beyond what the
definition states. The sources are four web pages on PagedAttention:

[P2] "High-Throughput Local LLM Infrastructure: Architecting a Distributed Go
     API Gateway for vLLM & PagedAttention Clusters", section 1.2
     "PagedAttention Mechanics & Virtual Page Tables" (logical block index =
     floor(position / block size), block offset = position mod block size;
     kernels look the physical block up in the block table and gather K/V),
     subsection "Reference Counting & Copy-on-Write (CoW)", and section 2.1
     "PagedAttention Memory Allocation Life-Cycle".
[P3] "03 - PagedAttention & the vLLM V1 Architecture", sections "The block
     table walkthrough" (the block-size-4 example) and "The attention kernel
     side" (walk the table, fetch each block's K/V tiles, softmax(QK^T/sqrt d)V).
[P5] "Inside vLLM: Anatomy of a High-Throughput LLM Inference System (2025)",
     section "Physical Block Mapping and Kernel Invocation" (the attention
     equation and the block index / offset equation), section "The KV-Cache
     Bottleneck" (KV bytes per sequence).
[P5'] the same page, section "Preemption Mechanics: Swapping vs.
     Recomputation" (blocks of a preempted sequence swapped to a pinned host
     pool and back); [P3] "Preemption & eviction".
[P1] "Tech Radar: vLLM v1 Production Engine Architecture & Distributed KV
     Cache Optimization", section 2, subsection "Mathematical Modeling of
     PagedAttention v3 Memory Bounds" (block count, block bytes, internal
     fragmentation) and the figure "PagedAttention v3 Block Mapping Layout".

Readings where the pages are silent (each is listed in the design notes):
  * query head h uses KV head floor(h / G), G = Hq / Hkv (grouped-query
    attention with contiguous groups);
  * a decode sequence's length includes the token just cached: it attends to
    keys 0 .. seq_len - 1;
  * chunked prefill: ctx = tokens before the chunk; query row r of the chunk
    sits at position ctx + r and attends to keys 0 .. ctx + r;
  * cache layout [num_blocks, num_kv_heads, block_size, head_dim], separate
    K and V pools;
  * a slot < 0 in a slot mapping means "skip this token";
  * split-KV: partition p holds keys [p*T, (p+1)*T); it yields the running
    max m_p, the sum l_p = sum exp(s - m_p) and the unnormalised
    o_p = sum exp(s - m_p) v; merging takes M = max m_p and returns
    sum exp(m_p - M) o_p / sum exp(m_p - M) l_p (the pages are silent on
    split-KV; this is the plain log-sum-exp identity).

Pins: every function here is checked against something other than itself in
tests/test_oracle_pins.py (torch's fp64 scaled_dot_product_attention on
contiguous K/V, the block-size-4 worked example, permutation and sharing
invariants, closed forms, the pages' printed sizing examples, and planted
mistakes that each pin must catch). No function is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np
import torch


# ---------------------------------------------------------------------------
# Sizing formulas ([P1] "Mathematical Modeling of PagedAttention v3 Memory
# Bounds"; [P5] "The KV-Cache Bottleneck").
# ---------------------------------------------------------------------------

def num_blocks_for(seq_len: int, block_size: int) -> int:
    """N_blocks(i) = ceil(S_i / B)."""
    return int(math.ceil(seq_len / block_size))


def block_bytes(num_layers: int, num_kv_heads: int, head_dim: int, block_size: int, elem_bytes: int) -> int:
    """BlockSize_bytes = 2 * L * H_KV * D_head * B * sizeof(dtype)."""
    return 2 * num_layers * num_kv_heads * head_dim * block_size * elem_bytes


def internal_fragmentation(seq_len: int, block_size: int) -> float:
    """Frag_internal(i) = ((B - (S_i mod B)) mod B) / (N_blocks(i) * B)."""
    unused = (block_size - (seq_len % block_size)) % block_size
    return unused / (num_blocks_for(seq_len, block_size) * block_size)


def kv_bytes_per_sequence(num_layers: int, num_kv_heads: int, head_dim: int, seq_len: int, elem_bytes: int) -> int:
    """Memory_KV for one sequence = 2 * S * L * H * D * P."""
    return 2 * seq_len * num_layers * num_kv_heads * head_dim * elem_bytes


# ---------------------------------------------------------------------------
# Addressing ([P2] 1.2; [P5] "Physical Block Mapping and Kernel Invocation").
# ---------------------------------------------------------------------------

def logical_block_and_offset(position: int, block_size: int) -> tuple[int, int]:
    """Logical block index = floor(pos / B); block offset = pos mod B."""
    return position // block_size, position % block_size


def slot_for(block_table_row, position: int, block_size: int) -> int:
    """Physical slot of a token: its block's physical id times B plus its offset."""
    blk, off = logical_block_and_offset(int(position), block_size)
    return int(block_table_row[blk]) * block_size + off


def slot_mapping(block_tables, seq_ids, positions, block_size: int) -> np.ndarray:
    """Slot of every new token (one plain loop)."""
    bt = np.asarray(block_tables)
    out = np.empty(len(seq_ids), dtype=np.int64)
    for t, (s, p) in enumerate(zip(np.asarray(seq_ids), np.asarray(positions))):
        out[t] = slot_for(bt[int(s)], int(p), block_size)
    return out


# ---------------------------------------------------------------------------
# Cache writes ([P2] 2.1 step 4: kernels write new K/V into the assigned
# physical blocks) and copy-on-write ([P2] "Reference Counting & CoW";
# [P3] walkthrough: "you copy the whole block when a write inside it would
# diverge").
# These move stored values; they are exact for any dtype.
# ---------------------------------------------------------------------------

def reshape_and_cache(k_new, v_new, slots, k_cache, v_cache, block_size: int) -> None:
    """In place: cache[slot // B, h, slot % B, :] = new[t, h, :] for slot >= 0."""
    for t, slot in enumerate(np.asarray(slots)):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = logical_block_and_offset(slot, block_size)
        k_cache[blk, :, off, :] = k_new[t]
        v_cache[blk, :, off, :] = v_new[t]


def copy_blocks(k_cache, v_cache, pairs) -> None:
    """In place: for every (src, dst) pair, the whole K and V block dst <- src."""
    for src, dst in np.asarray(pairs).reshape(-1, 2):
        k_cache[int(dst)] = k_cache[int(src)]
        v_cache[int(dst)] = v_cache[int(src)]


def swap_blocks(src_k, src_v, dst_k, dst_v, pairs) -> None:
    """Swap preemption ([P5] "Preemption Mechanics: Swapping vs.
    Recomputation": a preempted sequence's blocks move to a host pool and
    back; [P3] "Preemption & eviction"): for every (src, dst) pair the whole
    K and V block dst_pool[dst] <- src_pool[src] (src_v / dst_v may be None
    for a single pool)."""
    for src, dst in np.asarray(pairs).reshape(-1, 2):
        dst_k[int(dst)] = src_k[int(src)]
        if src_v is not None:
            dst_v[int(dst)] = src_v[int(src)]


# ---------------------------------------------------------------------------
# Attention ([P5] Attention(Q,K,V) = softmax(QK^T / sqrt(d_k)) V with K_i, V_i
# fetched through block index / offset; [P3] "The attention kernel side").
# ---------------------------------------------------------------------------

def to_f64(x) -> np.ndarray:
    """Exact up-cast of stored values (fp32 / fp16 / bf16) to float64."""
    if isinstance(x, torch.Tensor):
        return x.detach().to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def gather_sequence(cache, block_table_row, length: int, block_size: int) -> np.ndarray:
    """Contiguous [length, Hkv, D] float64 K (or V) of one sequence: position p
    is read from physical block table[floor(p / B)] at offset p mod B."""
    pos = np.arange(int(length))
    blk = np.asarray(block_table_row, dtype=np.int64)[pos // block_size]
    off = pos % block_size
    if isinstance(cache, torch.Tensor):
        rows = cache[torch.from_numpy(blk), :, torch.from_numpy(off), :]
    else:
        rows = np.asarray(cache)[blk, :, off, :]
    return to_f64(rows)


def kv_head_of(q_head: int, num_q_heads: int, num_kv_heads: int) -> int:
    """Grouped-query attention: query head h reads KV head floor(h / G)."""
    return q_head // (num_q_heads // num_kv_heads)


def softmax_attention(q_rows: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float) -> np.ndarray:
    """softmax(q K^T * scale) V for each row of q_rows ([R, D]; keys, values [L, D])."""
    s = (q_rows @ keys.T) * scale
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    return (p @ values) / p.sum(axis=1, keepdims=True)


def decode(q, k_cache, v_cache, block_tables, seq_lens, scale: float, block_size: int, seqs=None) -> np.ndarray:
    """Paged decode attention. q: [N, Hq, D]; returns float64 [N, Hq, D]
    (rows of sequences not in `seqs` are left as NaN)."""
    qf = to_f64(q)
    n, hq, d = qf.shape
    hkv = k_cache.shape[1]
    out = np.full((n, hq, d), np.nan)
    for i in (range(n) if seqs is None else seqs):
        L = int(seq_lens[i])
        K = gather_sequence(k_cache, block_tables[i], L, block_size)
        V = gather_sequence(v_cache, block_tables[i], L, block_size)
        for h in range(hq):
            g = kv_head_of(h, hq, hkv)
            out[i, h] = softmax_attention(qf[i, h][None, :], K[:, g], V[:, g], scale)[0]
    return out


def prefill(q, cu_q_lens, ctx_lens, k_cache, v_cache, block_tables, scale: float, block_size: int,
            seqs=None, rows=None) -> np.ndarray:
    """Chunked-prefill attention over the paged context. q: [sum q_len, Hq, D].
    Row r of sequence i sits at position ctx_i + r and attends to keys
    0 .. ctx_i + r. Returns float64 [sum q_len, Hq, D]; rows not computed
    are NaN. `rows`, if given, maps a sequence to the chunk rows to compute."""
    qf = to_f64(q)
    total, hq, d = qf.shape
    hkv = k_cache.shape[1]
    out = np.full((total, hq, d), np.nan)
    cu = np.asarray(cu_q_lens)
    for i in (range(len(cu) - 1) if seqs is None else seqs):
        q0, q1 = int(cu[i]), int(cu[i + 1])
        ctx = int(ctx_lens[i])
        L = ctx + (q1 - q0)
        K = gather_sequence(k_cache, block_tables[i], L, block_size)
        V = gather_sequence(v_cache, block_tables[i], L, block_size)
        rr = range(q1 - q0) if rows is None or i not in rows else rows[i]
        for r in rr:
            keys = ctx + r + 1
            for h in range(hq):
                g = kv_head_of(h, hq, hkv)
                out[q0 + r, h] = softmax_attention(qf[q0 + r, h][None, :], K[:keys, g], V[:keys, g], scale)[0]
    return out


# ---------------------------------------------------------------------------
# Split-KV partition and merge (the pages are silent; this is the
# log-sum-exp identity for a softmax computed in pieces).
# ---------------------------------------------------------------------------

def partition_partials(q_row: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float, partition: int):
    """Per partition p (keys [p*T, (p+1)*T)): m_p = max s, l_p = sum exp(s - m_p),
    o_p = sum exp(s - m_p) v (unnormalised)."""
    ms, ls, os_ = [], [], []
    for start in range(0, keys.shape[0], partition):
        kk = keys[start:start + partition]
        vv = values[start:start + partition]
        s = (kk @ q_row) * scale
        m = s.max()
        p = np.exp(s - m)
        ms.append(m)
        ls.append(p.sum())
        os_.append(p @ vv)
    return np.array(ms), np.array(ls), np.array(os_)


def merge_partials(m: np.ndarray, l: np.ndarray, o: np.ndarray) -> np.ndarray:
    """out = sum_p exp(m_p - M) o_p / sum_p exp(m_p - M) l_p, M = max_p m_p."""
    M = m.max()
    w = np.exp(m - M)
    return (w[:, None] * o).sum(axis=0) / (w * l).sum()
