"""libpagedattn: paged KV-cache attention for one NVIDIA GB300 (sm_103a).

The compute lives in hand-written CUDA kernels behind a C ABI
(include/pagedattn.h, built into libpagedattn.so by build.build()); this
package is the thin ctypes binding plus the host-side step helper.
"""
from ._binding import (  # noqa: F401
    EXPORTS,
    PA_BF16,
    PA_F16,
    PA_F32,
    PagedAttnError,
    exported_symbols,
    load,
    pa_chunked_prefill,
    pa_chunked_prefill_e5m2,
    pa_chunked_prefill_fp8,
    pa_chunked_prefill_workspace_size,
    pa_copy_blocks,
    pa_copy_blocks_fp8,
    pa_decode,
    pa_decode_e5m2,
    pa_decode_fp8,
    pa_decode_noalloc,
    pa_decode_noalloc_scratch_limit,
    pa_decode_partition_size,
    pa_decode_shared_prefix,
    pa_decode_shared_prefix_e5m2,
    pa_decode_shared_prefix_fp8,
    pa_decode_step,
    pa_selftest_bounded_wait,
    pa_decode_step_shared_prefix,
    pa_decode_shared_prefix_workspace_size,
    pa_decode_workspace_size,
    pa_get_status,
    pa_reshape_and_cache,
    pa_reshape_and_cache_e5m2,
    pa_reshape_and_cache_fp8,
    pa_slot_mapping,
    pa_strerror,
    pa_swap_blocks,
    pa_version,
)
from .builder import LIB_PATH, build  # noqa: F401
