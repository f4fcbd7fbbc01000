"""The bench's multi-rank path on CPU with gloo (world size 2): each rank is
an independent replica; the step time is the max over ranks and the value
counts every rank's bytes (weak scaling). No GPU needed."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        mine = [1.0 + rank, 10.0 - rank, 0.5 * (rank + 1)]
        got = bench.reduce_max_over_ranks(mine, world, "cpu")
        dist.barrier()
        q.put((rank, got, bench.weak_scaling_value(world, 2e9, got[0])))
    finally:
        dist.destroy_process_group()


def test_reduce_and_value_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == [2.0, 10.0, 1.0]  # elementwise max over the two ranks
        # 2 replicas x 2 GB each in 2 ms -> 2000 GB/s
        assert abs(value - 2 * 2e9 / 2e-3 / 1e9) < 1e-6


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.weak_scaling_value(1, 1e9, 1.0) == pytest.approx(1000.0)


def test_profiled_traffic_only_for_the_profiled_source(tmp_path):
    # The bench reports an attention call's DRAM traffic from a committed ncu
    # summary only while the library's CUDA sources are the ones that summary
    # was taken on.
    import bench
    sha = bench.source_sha256()
    good = tmp_path / "good.md"
    good.write_text(f"source_sha256: {sha}\ncall_dram_bytes: 123456\nkernel_dram_bytes: 1000\n"
                    "dominant_kernel: decode_tc_kernel\n")
    assert bench.profiled_traffic(str(good)) == {"call": 123456.0, "kernel": 1000.0,
                                                 "kernel_name": "decode_tc_kernel"}
    stale = tmp_path / "stale.md"
    stale.write_text("source_sha256: " + "0" * 64 + "\ncall_dram_bytes: 123456\n")
    assert bench.profiled_traffic(str(stale)) is None
    assert bench.profiled_traffic(str(tmp_path / "missing.md")) is None


def test_clock_samples_are_taken_from_the_timed_window():
    import bench
    clk = bench.ClockSampler(0)
    line = "{sm}, 2070, Active, {hw}, Not Active, Not Active, Not Active"
    clk.samples = [(1.0, line.format(sm=1000, hw="Not Active")),   # before the window
                   (2.0, line.format(sm=2070, hw="Not Active")),
                   (2.5, line.format(sm=2060, hw="Not Active")),
                   (3.0, line.format(sm=2050, hw="Not Active")),
                   (9.0, line.format(sm=900, hw="Active")),         # after the window
                   (9.5, "garbage")]
    s = clk.summary(2.0, 3.0)
    assert s == {"sm_mhz": 2060.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3}
    whole = clk.summary()
    assert whole["samples"] == 5 and whole["reasons"] == ["hw_slowdown"]
    assert bench.ClockSampler(0).summary(0, 1)["samples"] == 0


def test_timed_block_count():
    import bench
    assert bench.timed_block_count(6.3, 1000.0) == 159     # 20 steps of 0.315 ms: about 1 s
    assert bench.timed_block_count(500.0, 1000.0) == 3      # at least three blocks
    assert bench.timed_block_count(0.01, 1000.0) == 1000    # at most a thousand
