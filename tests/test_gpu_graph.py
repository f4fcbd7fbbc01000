"""The step (copy-on-write, slot mapping, cache write, attention) can be
captured in a CUDA graph and replayed with new inputs: the library's per-call
host work (argument checks, tensor-map encoding, copy-on-write pairs) is
baked into the captured kernel parameters, nothing synchronises, and every
replay gives the oracle's result on the inputs it replayed (and an eager
call's result on the same inputs, bit for bit). Graphs are captured per
batch-size bucket, as a serving engine captures one per predefined batch size
("High-Throughput Local LLM Infrastructure...", "CUDA Stream Management &
CUDA Graphs": 1, 2, 4, 8, 16, 32, 64)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import assert_attention_close, oracle_step, to_f64
from workloads import build_batch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind", ["decode", "shared_prefix", "prefill"])
def test_step_replays_from_cuda_graph(lib, kind):
    from paged_kv_cache_14_gb300.step import step_from_host
    if kind == "prefill":
        b = build_batch(name="graph", seed=90, dtype="f16", block_size=32, num_q_heads=64, num_kv_heads=8,
                        head_dim=128, q_lens=[1, 40, 1, 130], kv_lens=[300, 200, 1000, 700])
    else:
        lens = [5, 64, 300, 700, 1300, 2100, 31, 900]
        b = build_batch(name="graph", seed=91, dtype="bf16", block_size=16, num_q_heads=64, num_kv_heads=8,
                        head_dim=128, q_lens=np.ones(8, np.int32), kv_lens=lens, share_group=4,
                        share_prefix_tokens=256, cow_per_seq=True)
    st = step_from_host(b, shared_prefix=(kind == "shared_prefix"))
    st.run()  # first call outside capture (one-time per-kernel set-up)
    assert lib.pa_get_status() == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.run()
    new_q = torch.randn(st.q.shape, generator=torch.Generator().manual_seed(5)).to(st.q.dtype)
    st.q.copy_(new_q.cuda())
    g.replay()
    torch.cuda.synchronize()
    replayed = st.out.clone()
    assert_attention_close(to_f64(replayed), oracle_step(b, q=new_q), b.dtype, f"{kind}: replay vs oracle")
    st.run()
    assert lib.pa_get_status() == 0
    assert torch.equal(replayed, st.out)


@pytest.mark.parametrize("batch", [1, 2, 4, 8, 16, 32, 64])
def test_decode_graph_per_batch_bucket(lib, batch):
    """One captured decode step per batch-size bucket, replayed twice on new
    inputs (new q and new K/V of the appended token): each replay equals the
    oracle on those inputs, and an eager call."""
    from paged_kv_cache_14_gb300.step import step_from_host
    rng = np.random.default_rng(batch)
    lens = rng.integers(1, 3000, size=batch)
    b = build_batch(name="bucket", seed=100 + batch, dtype="bf16", block_size=16, num_q_heads=32, num_kv_heads=8,
                    head_dim=128, q_lens=np.ones(batch, np.int32), kv_lens=lens)
    st = step_from_host(b)
    st.run()
    assert lib.pa_get_status() == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.run()
    gen = torch.Generator().manual_seed(batch)
    for rep in range(2):
        q = torch.randn(st.q.shape, generator=gen).to(st.q.dtype)
        k_new = torch.randn(st.k_new.shape, generator=gen).to(st.k_new.dtype)
        v_new = torch.randn(st.v_new.shape, generator=gen).to(st.v_new.dtype)
        st.q.copy_(q.cuda())
        st.k_new.copy_(k_new.cuda())
        st.v_new.copy_(v_new.cuda())
        g.replay()
        torch.cuda.synchronize()
        replayed = st.out.clone()
        assert_attention_close(to_f64(replayed), oracle_step(b, q=q, k_new=k_new, v_new=v_new), "bf16",
                               f"bucket {batch} replay {rep} vs oracle")
        st.run()
        assert lib.pa_get_status() == 0
        assert torch.equal(replayed, st.out)


def test_host_pipeline_matches_oracle(lib):
    """Steps fed from pinned host memory through HostPipeline (copies on
    their own streams, two buffer sets) give, for each step, the oracle's
    output on that step's inputs, and the eager step's output bit for bit."""
    from paged_kv_cache_14_gb300.step import HostPipeline, step_from_host
    lens = [5, 64, 300, 700, 1300, 2100, 31, 900]
    b = build_batch(name="pipe", seed=93, dtype="bf16", block_size=16, num_q_heads=64, num_kv_heads=8,
                    head_dim=128, q_lens=np.ones(8, np.int32), kv_lens=lens, share_group=4,
                    share_prefix_tokens=256, cow_per_seq=True)
    st = step_from_host(b, shared_prefix=True)
    gen = torch.Generator().manual_seed(3)
    qs = [torch.randn(st.q.shape, generator=gen).to(st.q.dtype).pin_memory() for _ in range(4)]
    ks = [torch.randn(st.k_new.shape, generator=gen).to(st.k_new.dtype).pin_memory() for _ in range(4)]
    outs = [torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory() for _ in range(4)]
    pipe = HostPipeline(st)
    for q, k, o in zip(qs, ks, outs):
        pipe.submit({"q": q, "k_new": k}, o)
    pipe.drain()
    torch.cuda.synchronize()
    assert lib.pa_get_status() == 0
    for i, (q, k, o) in enumerate(zip(qs, ks, outs)):
        assert_attention_close(to_f64(o), oracle_step(b, q=q, k_new=k), "bf16", f"pipelined step {i} vs oracle")
        st.q.copy_(q)
        st.k_new.copy_(k)
        st.run()
        torch.cuda.synchronize()
        assert torch.equal(o, st.out.cpu())
