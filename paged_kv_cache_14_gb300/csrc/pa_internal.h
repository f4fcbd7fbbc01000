// Internal launch interface between the C-ABI layer (pa_api.cu) and the
// kernel translation units. Not part of the public API.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedattn.h"

namespace pa {

// 8-bit cache formats (with kv_scales): OCP FP8 E4M3 or E5M2.
enum KvFormat : int32_t { PA_KV_E4M3 = 0, PA_KV_E5M2 = 1 };

// Work-list entries: a sequence (or sharing group) index below 65536 in the
// upper 16 bits and a partition or tile index below 65536 in the lower 16,
// packed and unpacked as unsigned so that indices from 32768 up stay
// positive.
__host__ __device__ __forceinline__ int32_t pack_pair(int hi, int lo) {
  return (int32_t)(((uint32_t)hi << 16) | ((uint32_t)lo & 0xffffu));
}
__host__ __device__ __forceinline__ int pair_hi(int32_t v) { return (int)((uint32_t)v >> 16); }
__host__ __device__ __forceinline__ int pair_lo(int32_t v) { return (int)((uint32_t)v & 0xffffu); }

// Largest partition (tokens) one decode CTA walks; bounds the shared-memory
// copy of the partition's block ids.
constexpr int kMaxPartition = 16384;
// Pairs handed to one copy_blocks launch by value (kernel parameter space).
constexpr int kCopyPairsPerLaunch = 1024;

struct DecodeParams {
  const void* q;
  void* out;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* lens;       // seq_lens (decode) or ctx_lens (decode rows of a prefill batch)
  const int32_t* cu_q_lens;  // nullptr for plain decode; else only rows with q_len == 1 run
  int32_t max_blocks_per_seq;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t num_blocks;
  int32_t group;         // num_q_heads / num_kv_heads
  int32_t rows_per_cta;  // query heads of one group handled by one CTA
  int32_t row_groups;    // ceil(group / rows_per_cta)
  int32_t partition;     // tokens per split-KV partition (multiple of block_size)
  int32_t max_parts;     // grid.x; ceil(len_cap / partition)
  int32_t len_cap;       // largest legal length (host bound)
  float scale_log2;      // scale * log2(e)
  float* part_o;         // [num_seqs][num_q_heads][max_parts][head_dim]
  float* part_ml;        // [num_seqs][num_q_heads][max_parts][2] (m, l)
  // [num_seqs] x {sequence, output row, first partial slot, slots}: the
  // sequences with more than one split-KV partition (written by the plan).
  int4* merge_list;
  int32_t* work;         // [0] next work item, [1] number of work items, [2] sequences to merge (plan)
  int32_t* pairs;        // [num_seqs * max_parts] pack_pair(seq, partition), in work order
  // Shared-prefix (cascade) decode: tokens [0, prefix[i]) of sequence i were
  // attended by the prefix pass, whose partial sits in slot 0; the suffix
  // partitions use slots 1.. . nullptr / 0 for plain decode.
  const int32_t* prefix;
  int32_t slot0;
  int32_t planned;       // the work list is already built (by the shared-prefix preparation)
  // The decode rows of a mixed batch: launched behind the chunk kernel,
  // which waited for the plan that built this work list before letting this
  // kernel start; the decode streams at once, beside it, and waits for it
  // only before exiting.
  int32_t beside;
  // Standalone plain decode: the plan lists every row's first partition
  // first, in row order (rows with an illegal length too, as items the
  // kernel skips), so work item i < num_seqs * heads_per_row is known
  // without the plan: CTA c < first_static runs item c while the plan runs,
  // and the plan starts the work counter at first_static.
  int32_t static_first;
  int32_t first_static;
  // 8-bit KV cache: (K, V) scale per (block, KV head), float32
  // [num_blocks][num_kv_heads][2]; nullptr when the pools hold q's dtype.
  const float* kv_scales;
  int32_t kv_fmt;  // KvFormat of the codes when kv_scales is given
  int* status;
};

// Rows of a query-head group handled per decode work item (depends on dtype).
void decode_set_rows(DecodeParams& p, pa_dtype dt);


// Split-KV workspace layout shared by the size query and the launch. Every
// region starts on a 256-byte boundary.
struct DecodeWorkspace {
  size_t work, pairs, part_o, part_ml, merge, total;
};
inline DecodeWorkspace decode_workspace_layout(int64_t num_seqs, int64_t num_q_heads, int64_t head_dim,
                                               int64_t max_parts) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  DecodeWorkspace w{};
  w.work = 0;
  w.pairs = up(w.work + 16);
  w.part_o = up(w.pairs + (size_t)num_seqs * max_parts * 4);
  const size_t po = max_parts > 1 ? (size_t)num_seqs * num_q_heads * max_parts * head_dim * 4 : 0;
  w.part_ml = up(w.part_o + po);
  const size_t pm = max_parts > 1 ? (size_t)num_seqs * num_q_heads * max_parts * 2 * 4 : 0;
  w.merge = up(w.part_ml + pm);
  w.total = up(w.merge + (max_parts > 1 ? (size_t)num_seqs * 16 : 0));
  return w;
}

// Packed (position, GQA head) rows per work item of the tcgen05 prefill
// kernel (chunks and the shared-prefix pass).
constexpr int kPrefillRowsPerItem = 256;
// Query positions (chunked prefill) or group members (prefix pass) of one
// tcgen05 work item: two Q tiles of floor(128 / group) positions, each
// position's `group` query heads adjacent.
inline int prefill_positions_per_item(int group) { return 2 * (128 / group); }

struct PrefillParams {
  const void* q;
  void* out;
  const int32_t* block_tables;
  const int32_t* cu_q_lens;
  const int32_t* ctx_lens;
  int32_t max_blocks_per_seq;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t num_blocks;
  int32_t group;
  int32_t max_q_len;
  int32_t max_kv_len;
  int32_t total_q;   // rows of q / out
  int32_t tile_pos;  // query positions (or group members) per 128-row Q tile: floor(128 / group)
  float scale_log2;
  int32_t* work;     // [0] next work item, [1] number of work items, [2] CTAs that run items (chunks)
  int32_t* pairs;    // pack_pair(seq, row tile), longest first; prefix pass: pack_pair(group, member tile)
  int32_t ctas;      // grid of the chunk kernel
  int32_t num_sms;
  // Mixed batches: KV bytes of one decode-row token (K and V, all KV heads)
  // and the SM-time of one chunk (item, KV tile) unit in decode KV bytes.
  int32_t decode_token_bytes;
  float decode_bytes_per_tile;
  // 8-bit cache: (K, V) scale per (block, KV head), float32
  // [num_blocks][num_kv_heads][2]; nullptr when the pools hold q's dtype.
  const float* kv_scales;
  int32_t kv_fmt;  // KvFormat of the codes when kv_scales is given
  // Prefix pass of shared-prefix decode (null for chunked prefill): rows are
  // (group member, GQA head); keys are the group's shared blocks, read
  // through the table of the member with the longest verified prefix; the
  // result is a partial (m, l, o~) in slot 0 of every member.
  const int32_t* group_starts;  // [num_groups + 1]
  const int32_t* prefix;        // [num_seqs] verified shared-prefix lengths
  const int32_t* group_ref;     // [num_groups] member whose table covers the group prefix
  const int32_t* pair_keys;     // [pairs] keys of the pair's tile (max prefix of its members)
  float* part_o;
  float* part_ml;
  int32_t max_parts;
  int* status;
};

// Workspace of shared-prefix decode, after the decode workspace (which is
// laid out with max_parts + 1 partial slots).
struct CascadeWorkspace {
  size_t prefix, group_of, group_ref, work, pairs, pair_keys, total;
};
inline CascadeWorkspace cascade_workspace_layout(int64_t num_seqs, int64_t num_groups) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  CascadeWorkspace w{};
  w.prefix = 0;
  w.group_of = up(w.prefix + (size_t)num_seqs * 4);
  w.group_ref = up(w.group_of + (size_t)num_seqs * 4);
  w.work = up(w.group_ref + (size_t)num_groups * 4);
  w.pairs = up(w.work + 16);
  w.pair_keys = up(w.pairs + (size_t)num_seqs * 4);
  w.total = up(w.pair_keys + (size_t)num_seqs * 4);
  return w;
}

// Returns the device status word of the current device (nullptr on error).
int* device_status_ptr();
int num_sms_current_device();
// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device); thread-safe. PA_OK or PA_ERR_CUDA.
int set_max_dynamic_smem(const void* kernel, int bytes);

// Encode a 2-D tensor map over a KV pool seen as [num_blocks*num_kv_heads*block_size rows][head_dim],
// box = [box_rows rows][64 elements] with 128-byte swizzle (16-bit dtypes only).
int make_kv_tensor_map(CUtensorMap* map, const void* base, int64_t rows, int32_t head_dim, pa_dtype dt,
                       int32_t box_rows);
// Same view of an e4m3 (one byte per element) pool: box = [box_rows rows][128 bytes].
int make_u8_tensor_map(CUtensorMap* map, const void* base, int64_t rows, int32_t head_dim, int32_t box_rows);
// 3-D map over a [d2][d1][d0] tensor (d0 contiguous), box [b2][b1][b0], 128-byte swizzle.
int make_3d_tensor_map(CUtensorMap* map, const void* base, int64_t d2, int64_t d1, int64_t d0, pa_dtype dt,
                       int32_t b2, int32_t b1, int32_t b0);
// Same view, generic box (inner box_cols elements), 128-byte swizzle.
int make_2d_tensor_map(CUtensorMap* map, const void* base, int64_t rows, int32_t cols, int64_t row_stride_elems,
                       pa_dtype dt, int32_t box_rows, int32_t box_cols);

int launch_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq, int32_t num_seqs,
                        const int32_t* seq_ids, const int32_t* positions, int64_t num_tokens, int32_t block_size,
                        int32_t num_blocks, int64_t* slot_mapping, int* status, cudaStream_t stream,
                        bool chained = false);
int launch_reshape_and_cache(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                             void* k_cache, void* v_cache, int32_t num_blocks, int32_t block_size,
                             int32_t num_kv_heads, int32_t row_bytes, int* status, cudaStream_t stream,
                             bool chained = false);
// chained = true: launched as programmatic dependents of the previous kernel
// (a step whose kernels are all this library's, see launch_dependent).
int launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int32_t num_pairs,
                       int64_t block_bytes, cudaStream_t stream, bool chained = false);
// e4m3 cache write: per (run of consecutive tokens in one block, KV head,
// pool) one warp computes the block's new scale and encodes the rows.
int launch_reshape_and_cache_fp8(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                                 uint8_t* k_cache, uint8_t* v_cache, float* kv_scales, int32_t num_blocks,
                                 int32_t block_size, int32_t num_kv_heads, int32_t head_dim, pa_dtype dt,
                                 int kv_fmt, int* status, cudaStream_t stream);
// Whole blocks between two pools (device or pinned host memory; device-usable pointers).
int launch_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v, const int32_t* src,
                       const int32_t* dst, int32_t num_pairs, int64_t block_bytes, int vec16, cudaStream_t stream);
// The (K, V) scales of whole blocks, dst <- src.
int launch_copy_scales(float* kv_scales, const int32_t* src, const int32_t* dst, int32_t num_pairs,
                       int32_t num_kv_heads, cudaStream_t stream);

// Decode: split-KV main pass (+ merge pass when max_parts > 1).
int launch_decode(const DecodeParams& p, pa_dtype dt, cudaStream_t stream);
// fp32 I/O chunk rows (q_len > 1) of a mixed batch on CUDA cores (exact
// fp32); the decode rows are launched separately (launch_decode).
int launch_prefill_simt(const DecodeParams& p, int32_t total_q, cudaStream_t stream);
// The decode plan alone (fp16/bf16), for a step that launches other kernels
// between the plan and the decode: launch_decode then runs with
// planned = 1 and its first kernel waits for the ones before it.
int launch_decode_plan(const DecodeParams& p, pa_dtype dt, cudaStream_t stream);
// Prefill chunks (q_len > 1) on the tensor-core path. With `beside` (the
// decode rows of the same batch), the plan also builds their work list and
// splits the SMs; the caller then launches the decode (planned, beside)
// right after.
int launch_prefill(const PrefillParams& p, const void* k_cache, const void* v_cache, pa_dtype dt,
                   cudaStream_t stream, const DecodeParams* beside = nullptr);
// Prefix pass of shared-prefix decode on the same tensor-core kernel.
int launch_prefix_pass(const PrefillParams& p, const void* k_cache, const void* v_cache, pa_dtype dt,
                       cudaStream_t stream);
// Shared-prefix verification and the prefix pass's work list (one CTA).
// Also builds the suffix decode's work list (dp.prefix must point at
// prefix_out); the caller then launches the decode with dp.planned = 1.
int launch_cascade_prep(const DecodeParams& dp, pa_dtype dt, const int32_t* group_starts, const int32_t* prefix_in,
                        int32_t num_groups, int32_t members_per_tile, int32_t* prefix_out, int32_t* group_ref,
                        int32_t* group_of_seq, int32_t* work, int32_t* pairs, int32_t* pair_keys,
                        cudaStream_t stream);

}  // namespace pa
