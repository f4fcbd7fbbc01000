"""One pass of the paged-attention hot path on device tensors.

A step is what a serving engine runs per layer per iteration on the KV side:
  1. copy-on-write block copies (pa_copy_blocks) for blocks about to be
     written while shared,
  2. slot derivation for the new tokens (pa_slot_mapping),
  3. the cache write of their K/V (pa_reshape_and_cache),
  4. attention over the paged context: pa_decode when every sequence has one
     new query token (pa_decode_shared_prefix when sequences share prefix
     blocks), pa_chunked_prefill otherwise.
With an e4m3 cache the same step runs pa_copy_blocks_fp8,
pa_reshape_and_cache_fp8 and pa_decode_fp8 (pa_decode_shared_prefix_fp8,
pa_chunked_prefill_fp8); with an e5m2 cache the *_e5m2 calls
(pa_copy_blocks_fp8 moves either format).
This module only sequences library calls on one stream and owns the device
buffers the calls need (slot mapping, output, split-KV workspace), allocated
once with PyTorch.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _binding as pa


class PagedStep:
    def __init__(self, *, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_tables: torch.Tensor, kv_lens: torch.Tensor, q_lens_host: np.ndarray,
                 kv_lens_host: np.ndarray, k_new: torch.Tensor, v_new: torch.Tensor,
                 new_seq_ids: torch.Tensor, new_positions: torch.Tensor, cow_pairs_host: np.ndarray,
                 scale: float, partition_size: int = 0, cu_q_lens: torch.Tensor | None = None,
                 ctx_lens: torch.Tensor | None = None, group_starts: torch.Tensor | None = None,
                 prefix_lens: torch.Tensor | None = None, kv_scales: torch.Tensor | None = None,
                 kv_format: str = "e4m3"):
        self.q, self.k_cache, self.v_cache = q, k_cache, v_cache
        # e4m3 cache: k_cache / v_cache hold uint8 codes, kv_scales the
        # float32 (K, V) scale of every (block, KV head).
        self.kv_scales = kv_scales
        if kv_format not in ("e4m3", "e5m2"):
            raise ValueError(f"kv_format {kv_format!r}: e4m3 or e5m2")
        self.kv_format = kv_format
        # Suffix of the library's 8-bit calls for this format: pa_decode_fp8
        # and friends hold e4m3 codes, the *_e5m2 calls e5m2 codes.
        self.kv_call_suffix = "fp8" if kv_format == "e4m3" else "e5m2"
        self.block_tables, self.kv_lens = block_tables, kv_lens
        self.k_new, self.v_new = k_new, v_new
        self.new_seq_ids, self.new_positions = new_seq_ids, new_positions
        self.cow_pairs = np.ascontiguousarray(np.asarray(cow_pairs_host, dtype=np.int64).reshape(-1, 2))
        self.scale = float(scale)
        self.partition_size = int(partition_size)
        q_lens_host = np.asarray(q_lens_host)
        kv_lens_host = np.asarray(kv_lens_host)
        self.is_decode = bool(np.all(q_lens_host == 1))
        self.max_seq_len = int(kv_lens_host.max())
        self.max_q_len = int(q_lens_host.max())
        self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim = k_cache.shape
        dev = q.device
        self.slot_mapping = torch.empty(new_positions.shape[0], dtype=torch.int64, device=dev)
        self.out = torch.empty_like(q)
        n = kv_lens_host.shape[0]
        hq = q.shape[1]
        if self.is_decode:
            need = pa.pa_decode_workspace_size(n, hq, self.num_kv_heads, self.head_dim, self.block_size,
                                               self.max_seq_len, self.partition_size)
        else:
            need = pa.pa_chunked_prefill_workspace_size(n, hq, self.num_kv_heads, self.head_dim,
                                                        self.block_size, q.shape[0], self.max_seq_len)
            self.cu_q_lens = cu_q_lens
            self.ctx_lens = ctx_lens
        # Shared-prefix decode when the batch names groups that share blocks.
        self.group_starts, self.prefix_lens = group_starts, prefix_lens
        self.shared_prefix = bool(self.is_decode and group_starts is not None and prefix_lens is not None
                                  and group_starts.shape[0] - 1 < n)
        if self.shared_prefix:
            need = max(need, pa.pa_decode_shared_prefix_workspace_size(
                n, hq, self.num_kv_heads, self.head_dim, self.block_size, self.max_seq_len, self.partition_size,
                group_starts.shape[0] - 1))
        self.workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)

    # Per-step inputs a serving loop refreshes (attribute names).
    INPUTS = ("q", "k_new", "v_new", "block_tables", "kv_lens", "new_seq_ids", "new_positions",
              "group_starts", "prefix_lens", "cu_q_lens", "ctx_lens")

    def twin(self) -> "PagedStep":
        """A step over the same KV pools (and scales) with its own input,
        output, slot-mapping and workspace buffers (same shapes)."""
        t = PagedStep.__new__(PagedStep)
        t.__dict__.update(self.__dict__)
        for name in self.INPUTS:
            v = getattr(self, name, None)
            if isinstance(v, torch.Tensor):
                setattr(t, name, v.clone())
        t.slot_mapping = torch.empty_like(self.slot_mapping)
        t.out = torch.empty_like(self.out)
        t.workspace = torch.empty_like(self.workspace)
        return t

    @property
    def launches(self) -> int:
        """Kernel launches of one step (the library's own kernels)."""
        n = 0
        if self.cow_pairs.shape[0]:
            n += -(-self.cow_pairs.shape[0] // 1024) * (2 if self.kv_scales is not None else 1)
        n += 2  # slot mapping, cache write
        part = pa.pa_decode_partition_size(self.kv_lens.shape[0], self.q.shape[1], self.num_kv_heads,
                                           self.block_size, self.max_seq_len,
                                           self.partition_size if self.is_decode else 0)
        if self.shared_prefix:
            # prefix check (which also plans the suffixes), prefix pass,
            # suffix decode, merge (the prefix partial makes it always run)
            return n + 4
        merge = 1 if -(-self.max_seq_len // part) > 1 else 0
        if not self.is_decode and self.max_q_len > 1:
            return n + 3 + merge  # one plan for both lists, chunk kernel, decode rows, merge
        return n + 2 + merge  # plan, decode, split-KV merge

    @property
    def step_calls(self) -> str:
        """The library calls one run() makes."""
        if self.shared_prefix and self.kv_scales is None:
            return ("pa_decode_step_shared_prefix (copy_blocks + slot_mapping + reshape_and_cache + "
                    "pa_decode_shared_prefix in one call)")
        if self.is_decode and self.kv_scales is None and self.q.dtype != torch.float32:
            return "pa_decode_step (copy_blocks + slot_mapping + reshape_and_cache + pa_decode in one call)"
        if self.kv_scales is not None:
            f = self.kv_call_suffix
            return f"pa_copy_blocks_fp8 + pa_slot_mapping + pa_reshape_and_cache_{f} + " + (
                f"pa_decode_shared_prefix_{f}" if self.shared_prefix else
                f"pa_decode_{f}" if self.is_decode else f"pa_chunked_prefill_{f}")
        return "pa_copy_blocks + pa_slot_mapping + pa_reshape_and_cache + " + (
            "pa_decode" if self.is_decode else "pa_chunked_prefill")

    @property
    def attention_kernels(self) -> str:
        """What the step's attention call (attend()) runs on the device."""
        f, fmt = self.kv_call_suffix, self.kv_format
        if self.kv_scales is not None and self.shared_prefix:
            return (f"pa_decode_shared_prefix_{f}: prefix check + tcgen05 prefix pass (codes widened in shared "
                    f"memory) + {fmt} split-KV suffix decode + merge")
        if self.kv_scales is not None and not self.is_decode:
            return (f"pa_chunked_prefill_{f}: {fmt} decode rows (decode + merge) beside the tcgen05 chunk kernel "
                    "(codes widened in shared memory), one plan")
        if self.kv_scales is not None:
            return f"pa_decode_{f}: plan + persistent {fmt} decode + split-KV merge"
        if self.shared_prefix:
            return ("pa_decode_shared_prefix: prefix check + tcgen05 prefix pass + split-KV suffix decode "
                    "+ merge")
        if self.is_decode:
            return "pa_decode: plan + persistent decode + split-KV merge"
        return "pa_chunked_prefill: decode rows (plan + decode + merge) and tcgen05 chunk kernel (plan + main)"

    def run(self, stream=None) -> torch.Tensor:
        if self.shared_prefix and self.kv_scales is None:
            # One call: the shared-prefix check runs beside the copies,
            # slots and cache write (same results as prepare() + attend()).
            pa.pa_decode_step_shared_prefix(self.cow_pairs, self.new_seq_ids, self.new_positions, self.k_new,
                                            self.v_new, self.slot_mapping, self.q, self.k_cache, self.v_cache,
                                            self.block_tables, self.kv_lens, self.max_seq_len, self.group_starts,
                                            self.prefix_lens, self.scale, out=self.out,
                                            partition_size=self.partition_size, workspace=self.workspace,
                                            stream=stream)
            return self.out
        if self.is_decode and self.kv_scales is None and self.q.dtype != torch.float32:
            # One call: the decode plan runs beside the cache side.
            pa.pa_decode_step(self.cow_pairs, self.new_seq_ids, self.new_positions, self.k_new, self.v_new,
                              self.slot_mapping, self.q, self.k_cache, self.v_cache, self.block_tables,
                              self.kv_lens, self.max_seq_len, self.scale, out=self.out,
                              partition_size=self.partition_size, workspace=self.workspace, stream=stream)
            return self.out
        self.prepare(stream)
        self.attend(stream)
        return self.out

    def prepare(self, stream=None) -> None:
        """The step's cache side: copy-on-write copies, slots, cache write."""
        fp8 = self.kv_scales is not None
        if self.cow_pairs.shape[0]:
            if fp8:
                pa.pa_copy_blocks_fp8(self.k_cache, self.v_cache, self.kv_scales, self.cow_pairs, stream=stream)
            else:
                pa.pa_copy_blocks(self.k_cache, self.v_cache, self.cow_pairs, stream=stream)
        pa.pa_slot_mapping(self.block_tables, self.new_seq_ids, self.new_positions, self.block_size,
                           self.num_blocks, slot_mapping=self.slot_mapping, stream=stream)
        if fp8:
            write_8bit = self.call_8bit("pa_reshape_and_cache")
            write_8bit(self.k_new, self.v_new, self.slot_mapping, self.k_cache, self.v_cache, self.kv_scales,
                       stream=stream)
        else:
            pa.pa_reshape_and_cache(self.k_new, self.v_new, self.slot_mapping, self.k_cache, self.v_cache,
                                    stream=stream)

    def call_8bit(self, name: str):
        """The binding's 8-bit form of a call for this cache's format."""
        return getattr(pa, f"{name}_{self.kv_call_suffix}")

    def attend(self, stream=None) -> torch.Tensor:
        """The attention call of the step alone."""
        if self.kv_scales is not None and self.shared_prefix:
            self.call_8bit("pa_decode_shared_prefix")(
                self.q, self.k_cache, self.v_cache, self.kv_scales, self.block_tables, self.kv_lens, self.max_seq_len,
                self.group_starts, self.prefix_lens, self.scale, out=self.out, partition_size=self.partition_size,
                workspace=self.workspace, stream=stream)
        elif self.kv_scales is not None and not self.is_decode:
            self.call_8bit("pa_chunked_prefill")(
                self.q, self.cu_q_lens, self.k_cache, self.v_cache, self.kv_scales, self.block_tables, self.ctx_lens,
                self.max_q_len, self.max_seq_len, self.scale, out=self.out, workspace=self.workspace, stream=stream)
        elif self.kv_scales is not None:
            self.call_8bit("pa_decode")(
                self.q, self.k_cache, self.v_cache, self.kv_scales, self.block_tables, self.kv_lens, self.max_seq_len,
                self.scale, out=self.out, partition_size=self.partition_size, workspace=self.workspace, stream=stream)
        elif self.shared_prefix:
            pa.pa_decode_shared_prefix(self.q, self.k_cache, self.v_cache, self.block_tables, self.kv_lens,
                                       self.max_seq_len, self.group_starts, self.prefix_lens, self.scale,
                                       out=self.out, partition_size=self.partition_size, workspace=self.workspace,
                                       stream=stream)
        elif self.is_decode:
            pa.pa_decode(self.q, self.k_cache, self.v_cache, self.block_tables, self.kv_lens, self.max_seq_len,
                         self.scale, out=self.out, partition_size=self.partition_size, workspace=self.workspace,
                         stream=stream)
        else:
            pa.pa_chunked_prefill(self.q, self.cu_q_lens, self.k_cache, self.v_cache, self.block_tables,
                                  self.ctx_lens, self.max_q_len, self.max_seq_len, self.scale, out=self.out,
                                  workspace=self.workspace, stream=stream)
        return self.out


def step_from_host(batch, device="cuda", partition_size: int = 0, shared_prefix: bool = False,
                   fp8_pool=None, kv_format: str = "e4m3") -> PagedStep:
    """Build a PagedStep from a host-side batch object exposing the fields of
    a seeded workload (q, caches, tables, lengths, new tokens, CoW pairs).
    With shared_prefix, decode uses the batch's prefix-sharing groups. With
    fp8_pool = (k_codes, v_codes, kv_scales) the step runs on an 8-bit cache
    (kv_format "e4m3" or "e5m2") holding those codes instead of the batch's
    16-bit pools."""
    def dev(x, dtype=None):
        t = torch.as_tensor(x)
        if dtype is not None:
            t = t.to(dtype)
        return t.to(device, non_blocking=False).contiguous()

    cu = np.zeros(batch.num_seqs + 1, dtype=np.int32)
    np.cumsum(batch.q_lens, out=cu[1:])
    kc, vc, sc = (batch.k_cache, batch.v_cache, None) if fp8_pool is None else fp8_pool
    return PagedStep(
        q=dev(batch.q), k_cache=dev(kc), v_cache=dev(vc), kv_scales=None if sc is None else dev(sc),
        block_tables=dev(batch.block_tables, torch.int32), kv_lens=dev(batch.kv_lens, torch.int32),
        q_lens_host=batch.q_lens, kv_lens_host=batch.kv_lens,
        k_new=dev(batch.k_new), v_new=dev(batch.v_new),
        new_seq_ids=dev(batch.new_seq_ids, torch.int32), new_positions=dev(batch.new_positions, torch.int32),
        cow_pairs_host=batch.cow_pairs, scale=batch.scale, partition_size=partition_size,
        cu_q_lens=dev(cu, torch.int32), ctx_lens=dev(batch.kv_lens - batch.q_lens, torch.int32),
        group_starts=dev(batch.group_starts, torch.int32) if shared_prefix else None,
        prefix_lens=dev(batch.prefix_lens, torch.int32) if shared_prefix else None,
        kv_format=kv_format,
    )


class HostPipeline:
    """Steps fed from the host with the transfers overlapped with compute.

    A serving loop that receives every step's inputs in (pinned) host memory
    and wants the attention output back on the host submits steps here. Two
    device buffer sets (a step and its twin over the same KV pools) alternate:
    step i's inputs are copied in on a copy stream while step i-1 computes,
    and its output is copied out on a second copy stream while step i+1
    computes. Events order every buffer's reuse; the steps themselves run in
    submission order on the compute stream, so the cache updates keep their
    order.
    """

    def __init__(self, step: PagedStep, compute_stream: torch.cuda.Stream | None = None):
        self.steps = (step, step.twin())
        self.compute = compute_stream or torch.cuda.current_stream()
        self.h2d = torch.cuda.Stream()
        self.d2h = torch.cuda.Stream()
        self.ev_in = [torch.cuda.Event(), torch.cuda.Event()]     # inputs of buffer k copied in
        self.ev_done = [torch.cuda.Event(), torch.cuda.Event()]   # step on buffer k computed
        self.ev_out = [torch.cuda.Event(), torch.cuda.Event()]    # output of buffer k copied out
        self.n = 0

    def submit(self, host_inputs: dict, host_out: torch.Tensor) -> None:
        """Enqueue one step: host_inputs maps PagedStep input names to pinned
        host tensors; host_out (pinned) receives the step's output."""
        k = self.n & 1
        st = self.steps[k]
        self.h2d.wait_event(self.ev_done[k])          # buffer k's previous step has read its inputs
        with torch.cuda.stream(self.h2d):
            for name, t in host_inputs.items():
                getattr(st, name).copy_(t, non_blocking=True)
        self.ev_in[k].record(self.h2d)
        self.compute.wait_event(self.ev_in[k])
        self.compute.wait_event(self.ev_out[k])      # buffer k's previous output has been copied out
        st.run(stream=self.compute)
        self.ev_done[k].record(self.compute)
        self.d2h.wait_event(self.ev_done[k])
        with torch.cuda.stream(self.d2h):
            host_out.copy_(st.out, non_blocking=True)
        self.ev_out[k].record(self.d2h)
        self.n += 1

    def drain(self) -> None:
        """Make the compute stream wait for every submitted copy."""
        self.compute.wait_stream(self.d2h)
