"""pa_decode_noalloc: decode with the library's fixed scratch array, for
callers that cannot allocate device memory when they call (a plugin inside
another runtime's memory pool, a serving loop that forbids cudaMalloc after
start-up, code that must not allocate while a stream is captured).

The test calls the allocation-free entry point through the C ABI twice in a
row and checks each result against pa_decode (the entry point that takes a
caller-provided workspace) on the same inputs, within the attention
tolerance the other tests use. The second call reuses the scratch left by the
first, which must not matter. This file is collected last on purpose."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from helpers import assert_attention_close, to_f64
from workloads import build_batch

pytestmark = pytest.mark.gpu


def _raw_noalloc(lib, q, kc, vc, bt, sl, max_len, scale, out, partition):
    N, hq, D = q.shape
    P, hkv, B, _ = kc.shape
    dt = {torch.bfloat16: lib.PA_BF16, torch.float16: lib.PA_F16, torch.float32: lib.PA_F32}[q.dtype]
    return lib.load().pa_decode_noalloc(
        q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), bt.shape[1], sl.data_ptr(), N, max_len, hq,
        hkv, D, B, P, ctypes.c_float(scale), out.data_ptr(), partition, dt,
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype,partition", [("bf16", 0), ("bf16", 256), ("f16", 64), ("f32", 128)])
def test_noalloc_matches_decode_twice(lib, dtype, partition):
    lens = [1, 17, 300, 1000, 2049, 64]
    D = 64 if dtype == "f32" else 128
    b = build_batch(name="noalloc", seed=77, dtype=dtype, block_size=16, num_q_heads=16, num_kv_heads=2,
                    head_dim=D, q_lens=np.ones(len(lens), np.int32), kv_lens=lens)
    dev = "cuda"
    q, kc, vc = b.q.to(dev), b.k_cache.to(dev), b.v_cache.to(dev)
    bt = torch.from_numpy(b.block_tables).to(dev)
    sl = torch.from_numpy(b.kv_lens).to(dev)
    ref = lib.pa_decode(q, kc, vc, bt, sl, b.max_seq_len, b.scale, partition_size=partition)
    assert lib.pa_get_status() == 0
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        rc = _raw_noalloc(lib, q, kc, vc, bt, sl, b.max_seq_len, b.scale, out, partition)
        assert rc == 0, lib.pa_strerror(rc)
        assert lib.pa_get_status() == 0
        assert_attention_close(to_f64(out), to_f64(ref), dtype, f"noalloc call {call}")


def test_noalloc_rejects_requests_beyond_its_scratch(lib):
    limit = lib.pa_decode_noalloc_scratch_limit()
    assert limit == 64 << 20
    # 4096 sequences x 64 heads x 64 partitions of fp32 partials is far more
    # than 64 MiB: refused before any launch, output untouched.
    n, hq, hkv, D = 4096, 64, 8, 128
    need = lib.pa_decode_workspace_size(n, hq, hkv, D, 16, 65536, 1024)
    assert need > limit
    q = torch.zeros(n, hq, D, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(8, hkv, 16, D, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(n, 4096, dtype=torch.int32, device="cuda")
    sl = torch.ones(n, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 3.0)
    rc = _raw_noalloc(lib, q, kc, kc, bt, sl, 65536, 0.1, out, 1024)
    assert rc == -13 and "PA_ERR_SCRATCH" in lib.pa_strerror(rc)
    assert bool((out == 3.0).all())
