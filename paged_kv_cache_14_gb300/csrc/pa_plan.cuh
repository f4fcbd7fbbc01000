// Decode work planning shared by the decode and shared-prefix translation
// units: which rows are decode rows, the legal key count, and the plan body
// that lists (sequence, partition) work pairs.
#pragma once

#include "pa_common.cuh"
#include "pa_internal.h"

// Work order of the decode plan: 1 = first partitions sequence-major, then
// the rest longest first; 0 = all partitions sequence-major.
#ifndef PA_DECODE_PLAN_ORDER
#define PA_DECODE_PLAN_ORDER 1
#endif

namespace pa {

// Row of q / out and key count of sequence `seq`; false when the sequence
// is not a decode row of this launch (a prefill chunk in a mixed batch).
__device__ __forceinline__ bool decode_row(const DecodeParams& p, int seq, int& qrow, int& len) {
  if (p.cu_q_lens) {
    const int q0 = p.cu_q_lens[seq], q1 = p.cu_q_lens[seq + 1];
    if (q1 - q0 != 1) return false;
    qrow = q0;
    len = p.lens[seq] + 1;
  } else {
    qrow = seq;
    len = p.lens[seq];
  }
  return true;
}

__device__ __forceinline__ bool len_ok(const DecodeParams& p, int len) {
  return len >= 1 && len <= p.len_cap && len <= p.max_blocks_per_seq * p.block_size;
}

// ---------------------------------------------------------------------------
// Plan: list the (sequence, partition) pairs that exist, reset the counters.
// One CTA of 1024 threads. Sequences with an illegal length get zero output
// rows and PA_ERR_SEQLEN.
// ---------------------------------------------------------------------------
// Body of the plan, run by all 1024 threads of one CTA (also called from the
// shared-prefix preparation kernel once the verified prefixes are written).
// lens_s / prefix_s, when given, are shared-memory copies of p.lens and
// p.prefix (plain decode rows only) read instead of global memory.
template <typename T>
__device__ __forceinline__ void decode_plan_body(const DecodeParams& p, const int32_t* lens_s = nullptr,
                                                 const int32_t* prefix_s = nullptr) {
  // Work order: the first partition of every sequence in sequence order
  // (the sequences of a prefix-sharing group are adjacent, so the CTAs that
  // read a shared prefix run at the same time and hit in L2), then every
  // other partition from the longest to the shortest, so the last items
  // pulled from the counter are short and the tail is short.
  constexpr int kBins = 1024;  // later partitions binned by length, 16 tokens per bin, longest first
  __shared__ int32_t scan[33];
  __shared__ int32_t hist[kBins];
  __shared__ int32_t n_merge;  // sequences whose partitions the merge kernel combines
  const int N = p.num_seqs;
  const int P = p.partition;
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) hist[i] = 0;
  if (threadIdx.x == 0) n_merge = 0;
  __syncthreads();
  auto bin_of = [&](int len, int part) {
    if (!PA_DECODE_PLAN_ORDER) return 0;
    const int plen = min(P, len - part * P);
    return min((P - plen) >> 4, kBins - 1);
  };
  const int per = (N + 1023) / 1024;
  const int s0 = min(N, (int)threadIdx.x * per), s1 = min(N, s0 + per);
  auto row = [&](int s, int& qrow, int& len) -> bool {
    if (lens_s && !p.cu_q_lens) {
      qrow = s;
      len = lens_s[s];
      return true;
    }
    return decode_row(p, s, qrow, len);
  };
  auto prefix_of = [&](int s) -> int { return prefix_s ? prefix_s[s] : (p.prefix ? p.prefix[s] : 0); };
  int cnt0 = 0;
  for (int s = s0; s < s1; ++s) {
    int qrow, len;
    if (!row(s, qrow, len)) continue;
    if (!len_ok(p, len)) {
      if (p.static_first) ++cnt0;  // keeps its place in the first section; the kernel skips it
      record_error(p.status, PA_ERR_SEQLEN);
      T* out = static_cast<T*>(p.out) + (int64_t)qrow * p.num_q_heads * p.head_dim;
      for (int i = 0; i < p.num_q_heads * p.head_dim; ++i) out[i] = T(0.0f);
      continue;
    }
    const int sl = len - prefix_of(s);  // keys left to the suffix pass
    const int n = (sl + P - 1) / P;
    // With shared-prefix decode the prefix pass reads the shared blocks, so
    // there is no L2 locality to keep: every partition goes longest first.
    const int first_binned = p.prefix ? 0 : 1;
    if (!p.prefix) ++cnt0;
    for (int part = first_binned; part < n; ++part) atomicAdd(&hist[bin_of(sl, part)], 1);
  }
  int total0;
  int base0 = block_exclusive_scan_1024(cnt0, scan, &total0);
  // Bins in ascending order (longest partitions first), after the first
  // partitions: one bin per thread.
  int nbin_total;
  const int bin_off = block_exclusive_scan_1024(hist[threadIdx.x], scan, &nbin_total);
  hist[threadIdx.x] = total0 + bin_off;
  __syncthreads();
  const int total = total0 + nbin_total;
  for (int s = s0; s < s1; ++s) {
    int qrow, len;
    if (!row(s, qrow, len)) continue;
    if (!len_ok(p, len)) {
      if (p.static_first) p.pairs[base0++] = pack_pair(s, 0);
      continue;
    }
    const int sl = len - prefix_of(s);
    const int n = (sl + P - 1) / P;
    const int first_binned = p.prefix ? 0 : 1;
    if (!p.prefix) p.pairs[base0++] = pack_pair(s, 0);
    for (int part = first_binned; part < n; ++part)
      p.pairs[atomicAdd(&hist[bin_of(sl, part)], 1)] = pack_pair(s, part);
    // One suffix partition: written by the decode kernel (alone, or merged
    // there with the prefix partial); more: listed for the merge kernel.
    if (n > 1 && p.merge_list) {
      const int first = prefix_of(s) > 0 ? 0 : p.slot0;  // slot 0 holds the prefix pass's partial
      p.merge_list[atomicAdd(&n_merge, 1)] = make_int4(s, qrow, first, p.slot0 + n - first);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    p.work[0] = p.static_first ? p.first_static : 0;  // items below first_static are taken already
    p.work[1] = total * p.num_kv_heads * p.row_groups;
    p.work[2] = n_merge;
  }
}

}  // namespace pa
