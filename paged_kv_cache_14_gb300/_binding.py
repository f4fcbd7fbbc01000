"""ctypes binding of libpagedattn (argument marshalling only).

Every function here takes torch tensors, checks that they are CUDA tensors of
the expected dtype and layout, passes their data pointers and the current (or
given) CUDA stream to the C entry point of the same name, and raises
PagedAttnError on a non-zero status. All computation happens in the library's
CUDA kernels; there is no fallback of any kind: if the library is missing,
load() raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from .builder import LIB_PATH

_lib: ctypes.CDLL | None = None

PA_F32, PA_F16, PA_BF16 = 0, 1, 2
_DT = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16}

EXPORTS = (
    "pa_strerror", "pa_version", "pa_get_status", "pa_slot_mapping", "pa_reshape_and_cache",
    "pa_copy_blocks", "pa_decode_partition_size", "pa_decode_workspace_size", "pa_decode",
    "pa_chunked_prefill_workspace_size", "pa_chunked_prefill", "pa_decode_shared_prefix_workspace_size",
    "pa_decode_shared_prefix", "pa_decode_noalloc_scratch_limit", "pa_decode_noalloc",
    "pa_reshape_and_cache_fp8", "pa_copy_blocks_fp8", "pa_decode_fp8", "pa_swap_blocks",
    "pa_decode_step_shared_prefix", "pa_decode_step", "pa_selftest_bounded_wait", "pa_decode_shared_prefix_fp8",
    "pa_chunked_prefill_fp8", "pa_reshape_and_cache_e5m2", "pa_decode_e5m2", "pa_decode_shared_prefix_e5m2",
    "pa_chunked_prefill_e5m2",
)

_i32, _i64, _f32, _vp, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {pa_strerror(status)} ({status})")


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libpagedattn.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "(there is no fallback path)")
    lib = ctypes.CDLL(path)
    sig = {
        "pa_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "pa_version": (ctypes.c_int, []),
        "pa_get_status": (ctypes.c_int, [_vp]),
        "pa_slot_mapping": (ctypes.c_int, [_vp, _i32, _i32, _vp, _vp, _i64, _i32, _i32, _vp, _vp]),
        "pa_reshape_and_cache": (ctypes.c_int, [_vp, _vp, _vp, _i64, _vp, _vp, _i32, _i32, _i32, _i32,
                                                ctypes.c_int, _vp]),
        "pa_copy_blocks": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _i64, _vp]),
        "pa_decode_partition_size": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32]),
        "pa_decode_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32]),
        "pa_decode": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                     _f32, _vp, _i32, _vp, _sz, ctypes.c_int, _vp]),
        "pa_chunked_prefill_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32]),
        "pa_chunked_prefill": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                              _i32, _i32, _i32, _i32, _f32, _vp, _vp, _sz, ctypes.c_int, _vp]),
        "pa_decode_shared_prefix_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32]),
        "pa_decode_shared_prefix": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _vp, _vp, _i32, _i32,
                                                   _i32, _i32, _i32, _i32, _f32, _vp, _i32, _vp, _sz, ctypes.c_int,
                                                   _vp]),
        "pa_decode_noalloc_scratch_limit": (_sz, []),
        "pa_decode_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                             _i32, _f32, _vp, _i32, ctypes.c_int, _vp]),
        "pa_reshape_and_cache_fp8": (ctypes.c_int, [_vp, _vp, _vp, _i64, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                                    ctypes.c_int, _vp]),
        "pa_copy_blocks_fp8": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp]),
        "pa_swap_blocks": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64, _vp]),
        "pa_selftest_bounded_wait": (ctypes.c_int, [_i64, _vp]),
        "pa_decode_step": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _i32, _vp,
                                          _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _i32, _vp, _sz,
                                          ctypes.c_int, _vp]),
        "pa_decode_step_shared_prefix": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp,
                                                        _vp, _i32, _vp, _i32, _i32, _vp, _vp, _i32, _i32, _i32,
                                                        _i32, _i32, _i32, _f32, _vp, _i32, _vp, _sz, ctypes.c_int,
                                                        _vp]),
        "pa_decode_fp8": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                         _i32, _f32, _vp, _i32, _vp, _sz, ctypes.c_int, _vp]),
        "pa_decode_shared_prefix_fp8": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _vp, _vp,
                                                       _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _i32, _vp,
                                                       _sz, ctypes.c_int, _vp]),
        "pa_chunked_prefill_fp8": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32,
                                                  _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _sz, ctypes.c_int,
                                                  _vp]),
    }
    for name in ("reshape_and_cache", "decode", "decode_shared_prefix", "chunked_prefill"):
        sig[f"pa_{name}_e5m2"] = sig[f"pa_{name}_fp8"]  # same arguments, e5m2 codes
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def exported_symbols(path: str | None = None) -> dict[str, bool]:
    """Which of the header's entry points the library exports (no GPU needed)."""
    lib = ctypes.CDLL(path or LIB_PATH)
    return {name: hasattr(lib, name) for name in EXPORTS}


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _cuda(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise PagedAttnError(rc, where)


def pa_strerror(status: int) -> str:
    return load().pa_strerror(int(status)).decode()


def pa_version() -> int:
    return int(load().pa_version())


def pa_get_status(stream=None) -> int:
    """Synchronise the stream, return and clear the device error word."""
    return int(load().pa_get_status(_stream(stream)))


def pa_slot_mapping(block_tables: torch.Tensor, seq_ids: torch.Tensor, positions: torch.Tensor,
                    block_size: int, num_blocks: int, slot_mapping: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    n = positions.shape[0]
    if slot_mapping is None:
        slot_mapping = torch.empty(n, dtype=torch.int64, device=positions.device)
    rc = load().pa_slot_mapping(
        _cuda(block_tables, "block_tables", torch.int32), block_tables.shape[1], block_tables.shape[0],
        _cuda(seq_ids, "seq_ids", torch.int32), _cuda(positions, "positions", torch.int32), n,
        block_size, num_blocks, _cuda(slot_mapping, "slot_mapping", torch.int64), _stream(stream))
    _check(rc, "pa_slot_mapping")
    return slot_mapping


def pa_reshape_and_cache(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                         k_cache: torch.Tensor, v_cache: torch.Tensor, stream=None) -> None:
    P, hkv, B, D = k_cache.shape
    dt = k_cache.dtype
    rc = load().pa_reshape_and_cache(
        _cuda(k, "k", dt), _cuda(v, "v", dt), _cuda(slot_mapping, "slot_mapping", torch.int64), k.shape[0],
        _cuda(k_cache, "k_cache", dt), _cuda(v_cache, "v_cache", dt), P, B, hkv, D, _DT[dt], _stream(stream))
    _check(rc, "pa_reshape_and_cache")


def pa_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_dst_pairs, stream=None) -> None:
    """src_dst_pairs: HOST int64 [n, 2] (numpy array, list or CPU tensor)."""
    pairs = np.ascontiguousarray(np.asarray(src_dst_pairs, dtype=np.int64).reshape(-1, 2))
    P = k_cache.shape[0]
    block_bytes = k_cache[0].numel() * k_cache.element_size()
    rc = load().pa_copy_blocks(
        _cuda(k_cache, "k_cache"), _cuda(v_cache, "v_cache", k_cache.dtype),
        pairs.ctypes.data_as(ctypes.c_void_p), pairs.shape[0], P, block_bytes, _stream(stream))
    _check(rc, "pa_copy_blocks")


def pa_decode_partition_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, block_size: int,
                             max_seq_len: int, partition_size: int = 0) -> int:
    r = int(load().pa_decode_partition_size(num_seqs, num_q_heads, num_kv_heads, block_size, max_seq_len,
                                            partition_size))
    if r < 0:
        raise PagedAttnError(r, "pa_decode_partition_size")
    return r


def pa_decode_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                             block_size: int, max_seq_len: int, partition_size: int = 0) -> int:
    return int(load().pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                               max_seq_len, partition_size))


def pa_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
              seq_lens: torch.Tensor, max_seq_len: int, scale: float, out: torch.Tensor | None = None,
              partition_size: int = 0, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    N, hq, D = q.shape
    P, hkv, B, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("q and k_cache head_dim differ")
    dt = q.dtype
    if out is None:
        out = torch.empty_like(q)
    need = pa_decode_workspace_size(N, hq, hkv, D, B, max_seq_len, partition_size)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().pa_decode(
        _cuda(q, "q", dt), _cuda(k_cache, "k_cache", dt), _cuda(v_cache, "v_cache", dt),
        _cuda(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _cuda(seq_lens, "seq_lens", torch.int32), N, int(max_seq_len), hq, hkv, D, B, P, float(scale),
        _cuda(out, "out", dt), int(partition_size), ws_ptr, ws_bytes, _DT[dt], _stream(stream))
    _check(rc, "pa_decode")
    return out


def pa_chunked_prefill_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                                      block_size: int, total_q: int, max_kv_len: int) -> int:
    return int(load().pa_chunked_prefill_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                        block_size, total_q, max_kv_len))


def pa_chunked_prefill(q: torch.Tensor, cu_q_lens: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                       block_tables: torch.Tensor, ctx_lens: torch.Tensor, max_q_len: int, max_kv_len: int,
                       scale: float, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    T, hq, D = q.shape
    P, hkv, B, _ = k_cache.shape
    n = ctx_lens.shape[0]
    dt = q.dtype
    if out is None:
        out = torch.empty_like(q)
    need = pa_chunked_prefill_workspace_size(n, hq, hkv, D, B, T, max_kv_len)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().pa_chunked_prefill(
        _cuda(q, "q", dt), T, _cuda(cu_q_lens, "cu_q_lens", torch.int32), _cuda(k_cache, "k_cache", dt),
        _cuda(v_cache, "v_cache", dt), _cuda(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _cuda(ctx_lens, "ctx_lens", torch.int32), n, int(max_q_len), int(max_kv_len), hq, hkv, D, B, P,
        float(scale), _cuda(out, "out", dt), ws_ptr, ws_bytes, _DT[dt], _stream(stream))
    _check(rc, "pa_chunked_prefill")
    return out


def pa_decode_shared_prefix_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                                           block_size: int, max_seq_len: int, partition_size: int,
                                           num_groups: int) -> int:
    return int(load().pa_decode_shared_prefix_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                             block_size, max_seq_len, partition_size, num_groups))


def pa_decode_shared_prefix(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                            group_starts: torch.Tensor, prefix_lens: torch.Tensor, scale: float,
                            out: torch.Tensor | None = None, partition_size: int = 0,
                            workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    N, hq, D = q.shape
    P, hkv, B, _ = k_cache.shape
    G = group_starts.shape[0] - 1
    dt = q.dtype
    if out is None:
        out = torch.empty_like(q)
    need = pa_decode_shared_prefix_workspace_size(N, hq, hkv, D, B, max_seq_len, partition_size, G)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().pa_decode_shared_prefix(
        _cuda(q, "q", dt), _cuda(k_cache, "k_cache", dt), _cuda(v_cache, "v_cache", dt),
        _cuda(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _cuda(seq_lens, "seq_lens", torch.int32), N, int(max_seq_len),
        _cuda(group_starts, "group_starts", torch.int32), _cuda(prefix_lens, "prefix_lens", torch.int32), G,
        hq, hkv, D, B, P, float(scale), _cuda(out, "out", dt), int(partition_size), ws_ptr, ws_bytes, _DT[dt],
        _stream(stream))
    _check(rc, "pa_decode_shared_prefix")
    return out


def pa_decode_step(cow_pairs, new_seq_ids: torch.Tensor, new_positions: torch.Tensor, k_new: torch.Tensor,
                   v_new: torch.Tensor, slot_mapping: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                   scale: float, out: torch.Tensor | None = None, partition_size: int = 0,
                   workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One decode step in one call: pa_copy_blocks(cow_pairs), pa_slot_mapping,
    pa_reshape_and_cache, pa_decode. cow_pairs: HOST int64 [n, 2]."""
    pairs = np.ascontiguousarray(np.asarray(cow_pairs, dtype=np.int64).reshape(-1, 2))
    N, hq, D = q.shape
    P, hkv, B, _ = k_cache.shape
    dt = q.dtype
    T = new_seq_ids.shape[0]
    if out is None:
        out = torch.empty_like(q)
    need = pa_decode_workspace_size(N, hq, hkv, D, B, max_seq_len, partition_size)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().pa_decode_step(
        pairs.ctypes.data_as(ctypes.c_void_p) if pairs.shape[0] else None, pairs.shape[0],
        _cuda(new_seq_ids, "new_seq_ids", torch.int32), _cuda(new_positions, "new_positions", torch.int32),
        _cuda(k_new, "k_new", dt), _cuda(v_new, "v_new", dt), T, _cuda(slot_mapping, "slot_mapping", torch.int64),
        _cuda(q, "q", dt), _cuda(k_cache, "k_cache", dt), _cuda(v_cache, "v_cache", dt),
        _cuda(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _cuda(seq_lens, "seq_lens", torch.int32), N, int(max_seq_len), hq, hkv, D, B, P, float(scale),
        _cuda(out, "out", dt), int(partition_size), ws_ptr, ws_bytes, _DT[dt], _stream(stream))
    _check(rc, "pa_decode_step")
    return out


def pa_decode_step_shared_prefix(cow_pairs, new_seq_ids: torch.Tensor, new_positions: torch.Tensor,
                                 k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                                 q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                 block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                                 group_starts: torch.Tensor, prefix_lens: torch.Tensor, scale: float,
                                 out: torch.Tensor | None = None, partition_size: int = 0,
                                 workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One decode step in one call: pa_copy_blocks(cow_pairs), pa_slot_mapping,
    pa_reshape_and_cache, pa_decode_shared_prefix. cow_pairs: HOST int64
    [n, 2] (numpy array, list or CPU tensor)."""
    pairs = np.ascontiguousarray(np.asarray(cow_pairs, dtype=np.int64).reshape(-1, 2))
    N, hq, D = q.shape
    P, hkv, B, _ = k_cache.shape
    G = group_starts.shape[0] - 1
    dt = q.dtype
    T = new_seq_ids.shape[0]
    if out is None:
        out = torch.empty_like(q)
    need = pa_decode_shared_prefix_workspace_size(N, hq, hkv, D, B, max_seq_len, partition_size, G)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().pa_decode_step_shared_prefix(
        pairs.ctypes.data_as(ctypes.c_void_p) if pairs.shape[0] else None, pairs.shape[0],
        _cuda(new_seq_ids, "new_seq_ids", torch.int32), _cuda(new_positions, "new_positions", torch.int32),
        _cuda(k_new, "k_new", dt), _cuda(v_new, "v_new", dt), T, _cuda(slot_mapping, "slot_mapping", torch.int64),
        _cuda(q, "q", dt), _cuda(k_cache, "k_cache", dt), _cuda(v_cache, "v_cache", dt),
        _cuda(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _cuda(seq_lens, "seq_lens", torch.int32), N, int(max_seq_len),
        _cuda(group_starts, "group_starts", torch.int32), _cuda(prefix_lens, "prefix_lens", torch.int32), G,
        hq, hkv, D, B, P, float(scale), _cuda(out, "out", dt), int(partition_size), ws_ptr, ws_bytes, _DT[dt],
        _stream(stream))
    _check(rc, "pa_decode_step_shared_prefix")
    return out


def pa_selftest_bounded_wait(limit_ns: int, stream=None) -> None:
    """Launch a wait that nothing completes: it gives up after limit_ns and
    records PA_ERR_TIMEOUT (read it with pa_get_status)."""
    _check(load().pa_selftest_bounded_wait(int(limit_ns), _stream(stream)), "pa_selftest_bounded_wait")


def pa_decode_noalloc_scratch_limit() -> int:
    return int(load().pa_decode_noalloc_scratch_limit())


def pa_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                      seq_lens: torch.Tensor, max_seq_len: int, scale: float, out: torch.Tensor,
                      partition_size: int = 0, stream=None) -> torch.Tensor:
    """pa_decode with the library's fixed scratch instead of a workspace.
    `out` must be given: this path allocates nothing."""
    N, hq, D = q.shape
    P, hkv, B, _ = k_cache.shape
    dt = q.dtype
    rc = load().pa_decode_noalloc(
        _cuda(q, "q", dt), _cuda(k_cache, "k_cache", dt), _cuda(v_cache, "v_cache", dt),
        _cuda(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _cuda(seq_lens, "seq_lens", torch.int32), N, int(max_seq_len), hq, hkv, D, B, P, float(scale),
        _cuda(out, "out", dt), int(partition_size), _DT[dt], _stream(stream))
    _check(rc, "pa_decode_noalloc")
    return out


# ---------------------------------------------------------------------------
# 8-bit KV cache: uint8 code pools [P, Hkv, B, D] and float32 scales
# [P, Hkv, 2] (K, V) per (block, KV head). The *_fp8 calls hold e4m3 codes,
# the *_e5m2 calls e5m2 codes; pa_copy_blocks_fp8 serves both.
# ---------------------------------------------------------------------------

def pa_reshape_and_cache_fp8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                             k_cache: torch.Tensor, v_cache: torch.Tensor, kv_scales: torch.Tensor,
                             stream=None) -> None:
    _reshape_and_cache_8bit("pa_reshape_and_cache_fp8", k, v, slot_mapping, k_cache, v_cache, kv_scales, stream)


def pa_reshape_and_cache_e5m2(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                              k_cache: torch.Tensor, v_cache: torch.Tensor, kv_scales: torch.Tensor,
                              stream=None) -> None:
    _reshape_and_cache_8bit("pa_reshape_and_cache_e5m2", k, v, slot_mapping, k_cache, v_cache, kv_scales, stream)


def _reshape_and_cache_8bit(sym, k, v, slot_mapping, k_cache, v_cache, kv_scales, stream) -> None:
    P, hkv, B, D = k_cache.shape
    dt = k.dtype
    rc = getattr(load(), sym)(
        _cuda(k, "k", dt), _cuda(v, "v", dt), _cuda(slot_mapping, "slot_mapping", torch.int64), k.shape[0],
        _cuda(k_cache, "k_cache", torch.uint8), _cuda(v_cache, "v_cache", torch.uint8),
        _cuda(kv_scales, "kv_scales", torch.float32), P, B, hkv, D, _DT[dt], _stream(stream))
    _check(rc, sym)


def pa_copy_blocks_fp8(k_cache: torch.Tensor, v_cache: torch.Tensor, kv_scales: torch.Tensor, src_dst_pairs,
                       stream=None) -> None:
    """src_dst_pairs: HOST int64 [n, 2] (numpy array, list or CPU tensor)."""
    pairs = np.ascontiguousarray(np.asarray(src_dst_pairs, dtype=np.int64).reshape(-1, 2))
    P, hkv, B, D = k_cache.shape
    rc = load().pa_copy_blocks_fp8(
        _cuda(k_cache, "k_cache", torch.uint8), _cuda(v_cache, "v_cache", torch.uint8),
        _cuda(kv_scales, "kv_scales", torch.float32), pairs.ctypes.data_as(ctypes.c_void_p), pairs.shape[0], P, B,
        hkv, D, _stream(stream))
    _check(rc, "pa_copy_blocks_fp8")


def pa_decode_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, kv_scales: torch.Tensor,
                  block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int, scale: float,
                  out: torch.Tensor | None = None, partition_size: int = 0, workspace: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    return _decode_8bit("pa_decode_fp8", q, k_cache, v_cache, kv_scales, block_tables, seq_lens, max_seq_len, scale,
                        out, partition_size, workspace, stream)


def pa_decode_e5m2(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, kv_scales: torch.Tensor,
                   block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int, scale: float,
                   out: torch.Tensor | None = None, partition_size: int = 0, workspace: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    return _decode_8bit("pa_decode_e5m2", q, k_cache, v_cache, kv_scales, block_tables, seq_lens, max_seq_len,
                        scale, out, partition_size, workspace, stream)


def _decode_8bit(sym, q, k_cache, v_cache, kv_scales, block_tables, seq_lens, max_seq_len, scale, out,
                 partition_size, workspace, stream) -> torch.Tensor:
    N, hq, D = q.shape
    P, hkv, B, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("q and k_cache head_dim differ")
    dt = q.dtype
    if out is None:
        out = torch.empty_like(q)
    need = pa_decode_workspace_size(N, hq, hkv, D, B, max_seq_len, partition_size)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = getattr(load(), sym)(
        _cuda(q, "q", dt), _cuda(k_cache, "k_cache", torch.uint8), _cuda(v_cache, "v_cache", torch.uint8),
        _cuda(kv_scales, "kv_scales", torch.float32), _cuda(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _cuda(seq_lens, "seq_lens", torch.int32), N, int(max_seq_len), hq, hkv, D, B, P,
        float(scale), _cuda(out, "out", dt), int(partition_size), ws_ptr, ws_bytes, _DT[dt], _stream(stream))
    _check(rc, sym)
    return out


def pa_decode_shared_prefix_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                kv_scales: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                                max_seq_len: int, group_starts: torch.Tensor, prefix_lens: torch.Tensor, scale: float,
                                out: torch.Tensor | None = None, partition_size: int = 0,
                                workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    return _shared_prefix_8bit("pa_decode_shared_prefix_fp8", q, k_cache, v_cache, kv_scales, block_tables,
                               seq_lens, max_seq_len, group_starts, prefix_lens, scale, out, partition_size,
                               workspace, stream)


def pa_decode_shared_prefix_e5m2(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                 kv_scales: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                                 max_seq_len: int, group_starts: torch.Tensor, prefix_lens: torch.Tensor, scale: float,
                                 out: torch.Tensor | None = None, partition_size: int = 0,
                                 workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    return _shared_prefix_8bit("pa_decode_shared_prefix_e5m2", q, k_cache, v_cache, kv_scales, block_tables,
                               seq_lens, max_seq_len, group_starts, prefix_lens, scale, out, partition_size,
                               workspace, stream)


def _shared_prefix_8bit(sym, q, k_cache, v_cache, kv_scales, block_tables, seq_lens, max_seq_len, group_starts,
                        prefix_lens, scale, out, partition_size, workspace, stream) -> torch.Tensor:
    N, hq, D = q.shape
    P, hkv, B, _ = k_cache.shape
    G = group_starts.shape[0] - 1
    dt = q.dtype
    if out is None:
        out = torch.empty_like(q)
    need = pa_decode_shared_prefix_workspace_size(N, hq, hkv, D, B, max_seq_len, partition_size, G)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = getattr(load(), sym)(
        _cuda(q, "q", dt), _cuda(k_cache, "k_cache", torch.uint8), _cuda(v_cache, "v_cache", torch.uint8),
        _cuda(kv_scales, "kv_scales", torch.float32), _cuda(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _cuda(seq_lens, "seq_lens", torch.int32), N, int(max_seq_len),
        _cuda(group_starts, "group_starts", torch.int32), _cuda(prefix_lens, "prefix_lens", torch.int32), G,
        hq, hkv, D, B, P, float(scale), _cuda(out, "out", dt), int(partition_size), ws_ptr, ws_bytes, _DT[dt],
        _stream(stream))
    _check(rc, sym)
    return out


def pa_chunked_prefill_fp8(q: torch.Tensor, cu_q_lens: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           kv_scales: torch.Tensor, block_tables: torch.Tensor, ctx_lens: torch.Tensor,
                           max_q_len: int, max_kv_len: int, scale: float, out: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    return _prefill_8bit("pa_chunked_prefill_fp8", q, cu_q_lens, k_cache, v_cache, kv_scales, block_tables, ctx_lens,
                         max_q_len, max_kv_len, scale, out, workspace, stream)


def pa_chunked_prefill_e5m2(q: torch.Tensor, cu_q_lens: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            kv_scales: torch.Tensor, block_tables: torch.Tensor, ctx_lens: torch.Tensor,
                            max_q_len: int, max_kv_len: int, scale: float, out: torch.Tensor | None = None,
                            workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    return _prefill_8bit("pa_chunked_prefill_e5m2", q, cu_q_lens, k_cache, v_cache, kv_scales, block_tables,
                         ctx_lens, max_q_len, max_kv_len, scale, out, workspace, stream)


def _prefill_8bit(sym, q, cu_q_lens, k_cache, v_cache, kv_scales, block_tables, ctx_lens, max_q_len, max_kv_len,
                  scale, out, workspace, stream) -> torch.Tensor:
    T, hq, D = q.shape
    P, hkv, B, _ = k_cache.shape
    n = ctx_lens.shape[0]
    dt = q.dtype
    if out is None:
        out = torch.empty_like(q)
    need = pa_chunked_prefill_workspace_size(n, hq, hkv, D, B, T, max_kv_len)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = getattr(load(), sym)(
        _cuda(q, "q", dt), T, _cuda(cu_q_lens, "cu_q_lens", torch.int32), _cuda(k_cache, "k_cache", torch.uint8),
        _cuda(v_cache, "v_cache", torch.uint8), _cuda(kv_scales, "kv_scales", torch.float32),
        _cuda(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _cuda(ctx_lens, "ctx_lens", torch.int32), n, int(max_q_len), int(max_kv_len), hq, hkv, D, B, P,
        float(scale), _cuda(out, "out", dt), ws_ptr, ws_bytes, _DT[dt], _stream(stream))
    _check(rc, sym)
    return out


def _pool_ptr(t: torch.Tensor | None, name: str) -> int | None:
    """Pointer of a pool for pa_swap_blocks: a contiguous CUDA tensor or a
    pinned CPU tensor."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or t.is_pinned()):
        raise TypeError(f"{name} must be a CUDA tensor or a pinned CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def pa_swap_blocks(src_k: torch.Tensor, src_v: torch.Tensor | None, dst_k: torch.Tensor,
                   dst_v: torch.Tensor | None, src_dst_pairs, stream=None) -> None:
    """Whole blocks dst[dst] <- src[src] between two pools (CUDA or pinned CPU
    tensors, leading dimension = blocks). src_dst_pairs: HOST int64 [n, 2]."""
    pairs = np.ascontiguousarray(np.asarray(src_dst_pairs, dtype=np.int64).reshape(-1, 2))
    if src_k.dtype != dst_k.dtype or src_k.shape[1:] != dst_k.shape[1:]:
        raise ValueError("source and destination pools differ in block layout")
    block_bytes = src_k[0].numel() * src_k.element_size()
    rc = load().pa_swap_blocks(
        _pool_ptr(src_k, "src_k"), _pool_ptr(src_v, "src_v"), _pool_ptr(dst_k, "dst_k"), _pool_ptr(dst_v, "dst_v"),
        pairs.ctypes.data_as(ctypes.c_void_p), pairs.shape[0], src_k.shape[0], dst_k.shape[0], block_bytes,
        _stream(stream))
    _check(rc, "pa_swap_blocks")
