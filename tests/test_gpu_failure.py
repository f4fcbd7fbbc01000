"""Failure detection without a GPU fault: a bounded device wait that nothing
completes gives up after its limit, records PA_ERR_TIMEOUT in the status
word, and the context stays usable for the next call."""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

from helpers import assert_attention_close, oracle_caches_after_step, oracle_decode, to_f64
from workloads import build_batch

pytestmark = pytest.mark.gpu

PA_ERR_TIMEOUT = -11


def test_bounded_wait_gives_up_and_context_stays_usable(lib):
    from paged_kv_cache_14_gb300.step import step_from_host
    lib.pa_get_status()  # clear any earlier record
    t0 = time.perf_counter()
    lib.pa_selftest_bounded_wait(2_000_000)  # 2 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert lib.pa_get_status() == PA_ERR_TIMEOUT
    assert elapsed < 5.0
    assert lib.pa_get_status() == 0  # reading cleared it
    # The next step runs normally and is correct.
    lens = [5, 64, 300, 31]
    b = build_batch(name="after_timeout", seed=740, dtype="bf16", block_size=16, num_q_heads=16, num_kv_heads=4,
                    head_dim=128, q_lens=np.ones(len(lens), np.int32), kv_lens=lens)
    st = step_from_host(b)
    st.run()
    torch.cuda.synchronize()
    assert lib.pa_get_status() == 0
    kc, vc, _ = oracle_caches_after_step(b)
    assert_attention_close(to_f64(st.out), oracle_decode(b, kc, vc), "bf16", "decode after a timed-out wait")
