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

// Last g with gs[g] <= s (gs non-decreasing, gs[0] <= s).
__device__ __forceinline__ int group_of(const int32_t* gs, int num_groups, int s) {
  int lo = 0, hi = num_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (gs[mid] <= s) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Shared memory of the staged preparation (32-bit words): group starts,
// reference members, then per sequence the length, the prefix and the group.
inline size_t cascade_prep_smem(int64_t num_seqs, int64_t num_groups) {
  return (size_t)(2 * num_groups + 1 + 3 * num_seqs) * 4;
}
constexpr size_t kCascadePrepSmemMax = 192 * 1024;

// One CTA of 1024 threads. staged = 1: the group starts, lengths, hints and
// per-group state live in shared memory (one pass of global loads up front,
// then only the block-table check reads global memory); staged = 0 (batches
// too large for shared memory): the same steps on the workspace arrays.
template <typename T>
__global__ void __launch_bounds__(1024) cascade_prep_kernel(const DecodeParams p, const int32_t* group_starts,
                                                            const int32_t* prefix_in, int32_t num_groups,
                                                            int32_t members_per_tile, int32_t staged,
                                                            int32_t* prefix_out, int32_t* group_ref,
                                                            int32_t* group_of_seq, int32_t* work, int32_t* pairs,
                                                            int32_t* pair_keys) {
  pdl_trigger();  // the prefix pass may start its set-up now; it waits for this kernel
  extern __shared__ int32_t sm[];
  __shared__ int count, bad_groups;
  const int N = p.num_seqs, B = p.block_size;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int32_t* gs = staged ? sm : group_starts;
  int32_t* ref = staged ? sm + num_groups + 1 : group_ref;
  int32_t* lens = staged ? ref + num_groups : nullptr;
  int32_t* pfx = staged ? lens + N : prefix_out;
  int32_t* gof = staged ? pfx + N : group_of_seq;
  // 0. Inputs (independent loads, one round trip when staged).
  if (tid == 0) count = 0;
  for (int s = tid; s < N; s += nt) {
    const int q = prefix_in[s];
    if (staged) {
      lens[s] = p.lens[s];
      pfx[s] = q;
    }
    // Pull the table entries the check in step 3 may compare into L2 now,
    // while the other steps run (128-byte lines of 32 entries).
    const int nbq = q > 0 ? min(q / B, p.max_blocks_per_seq) : 0;
    const int32_t* row = p.block_tables + (int64_t)s * p.max_blocks_per_seq;
    for (int j = 0; j < nbq; j += 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + j));
  }
  if (staged)
    for (int g = tid; g <= num_groups; g += nt) sm[g] = group_starts[g];
  for (int g = tid; g < num_groups; g += nt) ref[g] = 0;
  __syncthreads();
  // Groups must tile the batch in order: group_starts[0] = 0, non-decreasing,
  // group_starts[num_groups] = num_seqs. Otherwise every hint is dropped.
  if (tid == 0) bad_groups = gs[0] != 0 || gs[num_groups] != N;
  __syncthreads();
  for (int g = tid; g < num_groups; g += nt)
    if (gs[g + 1] < gs[g]) bad_groups = 1;
  __syncthreads();
  if (bad_groups && tid == 0) record_error(p.status, PA_ERR_ARG);
  // 1. Requested prefix, sanitised; every sequence's group.
  for (int s = tid; s < N; s += nt) {
    const int len = staged ? lens[s] : p.lens[s];
    const int q = staged ? pfx[s] : prefix_in[s];
    const bool ok = !bad_groups && len >= 1 && len <= p.len_cap && len <= p.max_blocks_per_seq * B && q > 0 &&
                    q % B == 0 && q < len;
    pfx[s] = ok ? q : 0;
    gof[s] = bad_groups ? 0 : group_of(gs, num_groups, s);
  }
  __syncthreads();
  // With invalid groups no hint survives: no reference, no prefix work.
  const bool groups_ok = !bad_groups;
  // 2. Reference member of every group: the longest requested prefix.
  for (int s = tid; s < N && groups_ok; s += nt) {
    const int g = gof[s];
    // Key: prefix blocks (clamped to 16 bits; beyond that a tie, which can
    // only drop hints) above the member index, compared as unsigned.
    const uint32_t key = ((uint32_t)min(pfx[s] / B, 65535) << 16) | (uint32_t)(s - gs[g]);
    atomicMax(reinterpret_cast<unsigned int*>(&ref[g]), key);
  }
  __syncthreads();
  for (int g = tid; g < num_groups && groups_ok; g += nt) ref[g] = gs[g] + (ref[g] & 0xffff);
  __syncthreads();
  // 3. Verify every member's shared blocks against the reference's table; a
  //    mismatch drops that member's hint (the reference always matches).
  //    Four threads per member, each over a contiguous quarter of the shared
  //    entries (16-byte loads when rows are 16-byte aligned), so one warp
  //    load covers whole row segments and all loads are in flight at once.
  const bool vec = (reinterpret_cast<uintptr_t>(p.block_tables) & 15) == 0 && (p.max_blocks_per_seq & 3) == 0;
  for (int idx = tid; idx < N * 4 && groups_ok; idx += nt) {
    const int s = idx >> 2, c = idx & 3;
    const int r = ref[gof[s]];
    const int nb = pfx[s] / B;
    const int q = ((nb + 3) / 4 + 3) & ~3;  // entries per quarter, a multiple of 4
    const int j0 = min(nb, c * q), j1 = min(nb, j0 + q);
    const int32_t* a = p.block_tables + (int64_t)s * p.max_blocks_per_seq;
    const int32_t* b = p.block_tables + (int64_t)r * p.max_blocks_per_seq;
    bool mismatch = false;  // no early exit: the loads stay independent
    int j = j0;
    if (vec) {
#pragma unroll 4
      for (; j + 4 <= j1; j += 4) {
        const int4 x = *reinterpret_cast<const int4*>(a + j), y = *reinterpret_cast<const int4*>(b + j);
        mismatch |= (x.x != y.x) | (x.y != y.y) | (x.z != y.z) | (x.w != y.w);
      }
    }
#pragma unroll 4
    for (; j < j1; ++j) mismatch |= a[j] != b[j];
    if (mismatch) pfx[s] = 0;
  }
  __syncthreads();
  // 4. Prefix-pass work: one pair per (group, tile of consecutive members)
  //    whose members share anything; its key count is their longest prefix.
  for (int s = tid; s < N && groups_ok; s += nt) {
    const int g = gof[s];
    const int m = s - gs[g];
    if (m % members_per_tile) continue;  // the tile's first member speaks for it
    const int end = min(min(gs[g + 1], s + members_per_tile), N);
    int keys = 0;
    for (int t = s; t < end; ++t) keys = max(keys, pfx[t]);
    if (keys > 0) {
      const int slot = atomicAdd(&count, 1);
      pairs[slot] = pack_pair(g, m / members_per_tile);
      pair_keys[slot] = keys;
    }
  }
  if (staged) {
    for (int s = tid; s < N; s += nt) prefix_out[s] = pfx[s];
    for (int g = tid; g < num_groups; g += nt) group_ref[g] = ref[g];
  }
  __syncthreads();
  if (tid == 0) {
    work[0] = 0;
    work[1] = count * p.num_kv_heads;
  }
  // 5. The suffix decode's work list, from the verified prefixes.
  decode_plan_body<T>(p, staged ? lens : nullptr, staged ? pfx : nullptr);
}

int launch_cascade_prep(const DecodeParams& dp, pa_dtype dt, const int32_t* group_starts, const int32_t* prefix_in,
                        int32_t num_groups, int32_t members_per_tile, int32_t* prefix_out, int32_t* group_ref,
                        int32_t* group_of_seq, int32_t* work, int32_t* pairs, int32_t* pair_keys,
                        cudaStream_t stream) {
  const size_t smem = cascade_prep_smem(dp.num_seqs, num_groups);
  const int staged = smem <= kCascadePrepSmemMax && !dp.cu_q_lens;
  auto kern = dt == PA_BF16 ? cascade_prep_kernel<__nv_bfloat16> : cascade_prep_kernel<__half>;
  if (staged && smem > 48 * 1024 &&
      set_max_dynamic_smem(reinterpret_cast<const void*>(kern), (int)kCascadePrepSmemMax) != PA_OK)
    return PA_ERR_CUDA;
  kern<<<1, 1024, staged ? smem : 0, stream>>>(dp, group_starts, prefix_in, num_groups, members_per_tile, staged,
                                               prefix_out, group_ref, group_of_seq, work, pairs, pair_keys);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
