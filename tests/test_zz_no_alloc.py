"""pa_decode_noalloc: decode with the library's fixed scratch array, for
callers that cannot allocate device memory when they call (a plugin inside
another runtime's memory pool, a serving loop that forbids cudaMalloc after
start-up, code that must not allocate while a stream is captured).

The test calls the allocation-free entry point through the C ABI twice in a
row, on two different batches (other lengths, so another number of split-KV
partitions and another layout of the scratch), and checks each result
against pa_decode (the entry point that takes a caller-provided workspace) and
against the fp64 oracle, within the attention tolerance the other tests use.
The second call reuses the scratch left by the first, which must not matter.
One more call goes through the Python wrapper. This file is collected last on
purpose."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from helpers import assert_attention_close, oracle_decode, to_f64
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


def _batch(dtype, seed, lens):
    D = 64 if dtype == "f32" else 128
    return build_batch(name="noalloc", seed=seed, dtype=dtype, block_size=16, num_q_heads=16, num_kv_heads=2,
                       head_dim=D, q_lens=np.ones(len(lens), np.int32), kv_lens=lens)


def _on_device(b):
    dev = "cuda"
    return (b.q.to(dev), b.k_cache.to(dev), b.v_cache.to(dev), torch.from_numpy(b.block_tables).to(dev),
            torch.from_numpy(b.kv_lens).to(dev))


# Two consecutive calls per case: the second batch has other lengths (so
# another partition count per sequence) and, where forced, another partition
# size than the first.
CASES = [
    ("bf16", (0, [1, 17, 300, 1000, 2049, 64]), (0, [4000, 3, 129, 700, 8191, 33, 1500])),
    ("bf16", (256, [1, 17, 300, 1000, 2049, 64]), (512, [5000, 2, 65, 6000])),
    ("f16", (64, [1, 17, 300, 1000, 2049, 64]), (0, [12000, 11, 3000])),
    ("f32", (128, [1, 17, 300, 1000, 2049, 64]), (32, [40, 900, 7])),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-p{c[1][0]}-p{c[2][0]}")
def test_noalloc_matches_decode_and_oracle_twice(lib, case):
    dtype, *calls = case
    for call, (partition, lens) in enumerate(calls):
        b = _batch(dtype, 77 + call, lens)
        q, kc, vc, bt, sl = _on_device(b)
        ref = lib.pa_decode(q, kc, vc, bt, sl, b.max_seq_len, b.scale, partition_size=partition)
        assert lib.pa_get_status() == 0
        out = torch.full_like(q, float("nan"))
        rc = _raw_noalloc(lib, q, kc, vc, bt, sl, b.max_seq_len, b.scale, out, partition)
        assert rc == 0, lib.pa_strerror(rc)
        assert lib.pa_get_status() == 0
        assert_attention_close(to_f64(out), to_f64(ref), dtype, f"noalloc call {call} vs pa_decode")
        # No cache write ran: the pools are the batch's as drawn.
        assert_attention_close(to_f64(out), oracle_decode(b, b.k_cache, b.v_cache), dtype,
                               f"noalloc call {call} vs oracle")


def test_noalloc_python_wrapper(lib):
    b = _batch("bf16", 79, [2, 640, 3000, 17])
    q, kc, vc, bt, sl = _on_device(b)
    out = torch.full_like(q, float("nan"))
    got = lib.pa_decode_noalloc(q, kc, vc, bt, sl, b.max_seq_len, b.scale, out=out, partition_size=256)
    assert got is out
    assert lib.pa_get_status() == 0
    assert_attention_close(to_f64(out), oracle_decode(b, b.k_cache, b.v_cache), "bf16", "noalloc wrapper")


def test_noalloc_checks_arguments_like_decode(lib):
    """An empty batch with a bad argument is refused as pa_decode refuses it."""
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(1, 4, dtype=torch.int32, device="cuda")
    sl = torch.ones(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    pa = lib.load()
    stream = torch.cuda.current_stream().cuda_stream
    # num_seqs = 0 with block size 24 (invalid), then with 6 query heads over
    # 4 KV heads (not a multiple).
    for bs, hq, hkv in ((24, 8, 2), (16, 6, 4)):
        args = (q.data_ptr(), kc.data_ptr(), kc.data_ptr(), bt.data_ptr(), 4, sl.data_ptr(), 0, 16, hq, hkv, 128,
                bs, 4, ctypes.c_float(0.1), out.data_ptr(), 0)
        want = pa.pa_decode(*args, None, 0, lib.PA_BF16, stream)
        got = pa.pa_decode_noalloc(*args, lib.PA_BF16, stream)
        assert want < 0 and got == want, (bs, hq, hkv, want, got)
    # A valid empty batch is a no-op for both.
    args = (q.data_ptr(), kc.data_ptr(), kc.data_ptr(), bt.data_ptr(), 4, sl.data_ptr(), 0, 16, 8, 2, 128, 16, 4,
            ctypes.c_float(0.1), out.data_ptr(), 0)
    assert pa.pa_decode_noalloc(*args, lib.PA_BF16, stream) == 0


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
