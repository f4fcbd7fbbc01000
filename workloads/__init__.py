"""Seeded synthetic workloads shared by the CUDA path's harness and the oracle.

Holds structure and random values only; no attention or slot arithmetic.
"""
from .generate import (  # noqa: F401
    CONFIG_NAMES,
    CONFIGS,
    TORCH_DTYPES,
    PagedBatch,
    build_batch,
    e4m3_pool,
    e5m2_pool,
    make_config,
    random_lengths,
)
