// Shared-prefix (cascade) decode, preparation step. Sequences that share
// leading blocks through refcounted block tables ("High-Throughput Local LLM
// Infrastructure...", section 1.2, "Reference Counting & Copy-on-Write";
// "Inside vLLM...", section "Zero-Copy Branching and Parallel Sampling")
// attend to those blocks in one tensor-core pass for the whole group; this
// kernel checks the caller's hints and lists that pass's work.
//
// For every sequence, the requested shared-prefix length is kept only if it
// is a positive multiple of the block size, shorter than the sequence, and
// its first prefix/B block-table entries equal those of the group member with
// the longest requested prefix (the reference, whose table then covers the
// group's whole shared prefix). Anything else is ignored for that sequence
// (prefix 0: its suffix pass covers all its keys), so a wrong hint costs
// speed, never correctness.
#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_plan.cuh"

namespace pa {

__device__ __forceinline__ int group_of(const int32_t* group_starts, int num_groups, int s) {
  int lo = 0, hi = num_groups - 1;  // last g with group_starts[g] <= s
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (group_starts[mid] <= s) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <typename T>
__global__ void __launch_bounds__(1024) cascade_prep_kernel(const DecodeParams p, const int32_t* group_starts,
                                                            const int32_t* prefix_in, int32_t num_groups,
                                                            int32_t members_per_tile, int32_t* prefix_out,
                                                            int32_t* group_ref, int32_t* group_of_seq,
                                                            int32_t* work, int32_t* pairs, int32_t* pair_keys) {
  pdl_trigger();  // the prefix pass may start its set-up now; it waits for this kernel
  __shared__ int count;
  const int N = p.num_seqs, B = p.block_size;
  const int tid = threadIdx.x, nt = blockDim.x;
  if (tid == 0) count = 0;
  // 1. Requested prefix, sanitised; every sequence's group.
  for (int s = tid; s < N; s += nt) {
    const int len = p.lens[s];
    const int q = prefix_in[s];
    const bool ok = len >= 1 && len <= p.len_cap && len <= p.max_blocks_per_seq * B && q > 0 && q % B == 0 && q < len;
    prefix_out[s] = ok ? q : 0;
    group_of_seq[s] = group_of(group_starts, num_groups, s);
  }
  for (int g = tid; g < num_groups; g += nt) group_ref[g] = 0;
  // Groups must tile the batch in order: group_starts[0] = 0, non-decreasing,
  // group_starts[num_groups] = num_seqs. Otherwise every hint is dropped.
  __shared__ int bad_groups;
  if (tid == 0) bad_groups = group_starts[0] != 0 || group_starts[num_groups] != N;
  __syncthreads();
  for (int g = tid; g < num_groups; g += nt)
    if (group_starts[g + 1] < group_starts[g]) bad_groups = 1;
  __syncthreads();
  if (bad_groups) {
    if (tid == 0) record_error(p.status, PA_ERR_ARG);
    for (int s = tid; s < N; s += nt) prefix_out[s] = 0;
    for (int s = tid; s < N; s += nt) group_of_seq[s] = 0;
  }
  __syncthreads();
  // 2. Reference member of every group: the longest requested prefix.
  for (int s = tid; s < N; s += nt) {
    const int g = group_of_seq[s];
    atomicMax(&group_ref[g], ((prefix_out[s] / B) << 16) | (s - group_starts[g]));
  }
  __syncthreads();
  for (int g = tid; g < num_groups; g += nt) group_ref[g] = group_starts[g] + (group_ref[g] & 0xffff);
  __syncthreads();
  // 3. Verify every member's shared blocks against the reference's table; a
  //    mismatch drops that member's hint (the reference always matches).
  for (int idx = tid; idx < N * 4; idx += nt) {
    const int s = idx >> 2, c = idx & 3;
    const int r = group_ref[group_of_seq[s]];
    const int nb = prefix_out[s] / B;
    const int32_t* a = p.block_tables + (int64_t)s * p.max_blocks_per_seq;
    const int32_t* b = p.block_tables + (int64_t)r * p.max_blocks_per_seq;
    bool mismatch = false;  // no early exit: the loads stay independent
#pragma unroll 8
    for (int j = c; j < nb; j += 4) mismatch |= a[j] != b[j];
    if (mismatch) prefix_out[s] = 0;
  }
  __syncthreads();
  // 4. Prefix-pass work: one pair per (group, tile of consecutive members)
  //    whose members share anything; its key count is their longest prefix.
  for (int s = tid; s < N; s += nt) {
    const int g = group_of_seq[s];
    const int m = s - group_starts[g];
    if (m % members_per_tile) continue;  // the tile's first member speaks for it
    const int end = min(group_starts[g + 1], s + members_per_tile);
    int keys = 0;
    for (int t = s; t < end; ++t) keys = max(keys, prefix_out[t]);
    if (keys > 0) {
      const int slot = atomicAdd(&count, 1);
      pairs[slot] = (g << 16) | (m / members_per_tile);
      pair_keys[slot] = keys;
    }
  }
  __syncthreads();
  if (tid == 0) {
    work[0] = 0;
    work[1] = count * p.num_kv_heads;
  }
  // 5. The suffix decode's work list, from the verified prefixes.
  decode_plan_body<T>(p);
}

int launch_cascade_prep(const DecodeParams& dp, pa_dtype dt, const int32_t* group_starts, const int32_t* prefix_in,
                        int32_t num_groups, int32_t members_per_tile, int32_t* prefix_out, int32_t* group_ref,
                        int32_t* group_of_seq, int32_t* work, int32_t* pairs, int32_t* pair_keys,
                        cudaStream_t stream) {
  if (dt == PA_BF16)
    cascade_prep_kernel<__nv_bfloat16><<<1, 1024, 0, stream>>>(dp, group_starts, prefix_in, num_groups,
                                                               members_per_tile, prefix_out, group_ref, group_of_seq,
                                                               work, pairs, pair_keys);
  else
    cascade_prep_kernel<__half><<<1, 1024, 0, stream>>>(dp, group_starts, prefix_in, num_groups, members_per_tile,
                                                        prefix_out, group_ref, group_of_seq, work, pairs, pair_keys);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
