"""Decode at the host checks' limits, against the fp64 oracle: the largest
batch (65535 sequences) and the largest number of split-KV partitions of one
sequence (12288 partials merged). One more of either is refused before any
launch (tests/test_abi.py)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import assert_attention_close, oracle_decode, to_f64
from workloads import build_batch

pytestmark = pytest.mark.gpu


def _on_device(b):
    return (b.q.cuda(), b.k_cache.cuda(), b.v_cache.cuda(), torch.from_numpy(b.block_tables).cuda(),
            torch.from_numpy(b.kv_lens).cuda())


@pytest.mark.parametrize("partition", [0, 16], ids=["auto", "p16"])
def test_decode_largest_batch(lib, partition):
    """65535 sequences of 1..40 tokens. With 16-token partitions most of them
    split (up to three partials each), so the merge list holds tens of
    thousands of sequences. Compared on the first and last 64 sequences and
    2000 drawn between them."""
    n = 65535
    rng = np.random.default_rng(11)
    lens = rng.integers(1, 41, n).astype(np.int32)
    b = build_batch(name="largest_batch", seed=11, dtype="bf16", block_size=16, num_q_heads=4, num_kv_heads=1,
                    head_dim=64, q_lens=np.ones(n, np.int32), kv_lens=lens)
    q, kc, vc, bt, sl = _on_device(b)
    out = lib.pa_decode(q, kc, vc, bt, sl, b.max_seq_len, b.scale, partition_size=partition)
    assert lib.pa_get_status() == 0
    seqs = sorted(set(range(64)) | set(range(n - 64, n)) | set(rng.choice(n, 2000, replace=False).tolist()))
    ref = oracle_decode(b, b.k_cache, b.v_cache, seqs=seqs)
    assert_attention_close(to_f64(out)[seqs], ref[seqs], "bf16", f"65535 sequences, partition {partition}")


def test_decode_most_partitions(lib):
    """One sequence of 196608 tokens in 16-token partitions: 12288 partials,
    the most a call accepts, merged in one pass; beside it a sequence of 100
    tokens (seven partials)."""
    lens = np.array([12288 * 16, 100], np.int32)
    b = build_batch(name="most_partitions", seed=12, dtype="bf16", block_size=16, num_q_heads=2, num_kv_heads=1,
                    head_dim=64, q_lens=np.ones(2, np.int32), kv_lens=lens)
    q, kc, vc, bt, sl = _on_device(b)
    out = lib.pa_decode(q, kc, vc, bt, sl, b.max_seq_len, b.scale, partition_size=16)
    assert lib.pa_get_status() == 0
    assert_attention_close(to_f64(out), oracle_decode(b, b.k_cache, b.v_cache), "bf16", "12288 partitions")
