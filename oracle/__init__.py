"""Plain fp64 CPU oracle for paged KV-cache attention.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
bench's CPU-baseline / reference legs, never by the CUDA library or its
binding. See paged_attention.py for the definitions and their sources.
"""
from .paged_attention import *  # noqa: F401,F403
from .paged_attention import (  # noqa: F401
    block_bytes,
    copy_blocks,
    decode,
    gather_sequence,
    internal_fragmentation,
    kv_bytes_per_sequence,
    kv_head_of,
    logical_block_and_offset,
    merge_partials,
    num_blocks_for,
    partition_partials,
    prefill,
    reshape_and_cache,
    slot_for,
    slot_mapping,
    softmax_attention,
    swap_blocks,
    to_f64,
)
