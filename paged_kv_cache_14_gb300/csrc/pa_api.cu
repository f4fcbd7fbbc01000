// C-ABI entry points of libpagedattn: host-side argument checks, tensor-map
// encoding, split-KV planning and dispatch to the kernel launchers.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <set>
#include <utility>
#include <unordered_set>
#include <vector>

#include "pa_common.cuh"
#include "pa_internal.h"

// First device-side error since the last pa_get_status() (one word per device).
__device__ int g_pa_status;

namespace pa {

namespace {
constexpr int kMaxDevices = 64;
// Decode-row KV bytes one SM streams in the time it runs one (item, KV tile)
// unit of the chunk kernel (see mixed_plan_kernel); it sets how a mixed batch
// splits the SMs. On GB300 a unit takes about 1.6 us and the decode kernel
// streams about 90-100 GB/s per SM when only a few SMs run it. A sweep of the
// mixed 70B-shaped batch (8 chunks of 512 rows, 96 decode rows) gave the
// call 1.27 / 1.01 / 0.98 / 0.935 / 0.99 / 1.00 ms at 40K / 80K / 120K /
// 160K / 240K / 400K bytes, and 1.03 ms with all SMs to the chunks.
#ifndef PA_DECODE_BYTES_PER_CHUNK_TILE
#define PA_DECODE_BYTES_PER_CHUNK_TILE 160000.0f
#endif
constexpr float kDecodeBytesPerChunkTile = PA_DECODE_BYTES_PER_CHUNK_TILE;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_tried = false;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(pa_dtype dt) {
  switch (dt) {
    case PA_F32: return 4;
    case PA_F16: return 2;
    case PA_BF16: return 2;
  }
  return 0;
}

bool head_dim_supported(pa_dtype dt, int32_t d) {
  if (dt == PA_F32) return d >= 32 && d <= 256 && d % 32 == 0;
  return d == 64 || d == 128;
}
}  // namespace

int* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

int num_sms_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_num_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

int set_max_dynamic_smem(const void* kernel, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  std::lock_guard<std::mutex> lk(mu);
  if (done.count({kernel, dev})) return PA_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return PA_ERR_CUDA;
  done.insert({kernel, dev});
  return PA_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode_tried) {
    g_encode_tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

int make_2d_tensor_map(CUtensorMap* map, const void* base, int64_t rows, int32_t cols, int64_t row_stride_elems,
                       pa_dtype dt, int32_t box_rows, int32_t box_cols) {
  auto fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  if (dt == PA_F32) return PA_ERR_DTYPE;
  const CUtensorMapDataType t = dt == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)row_stride_elems * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, t, 2, const_cast<void*>(base), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int make_3d_tensor_map(CUtensorMap* map, const void* base, int64_t d2, int64_t d1, int64_t d0, pa_dtype dt,
                       int32_t b2, int32_t b1, int32_t b0) {
  auto fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  if (dt == PA_F32) return PA_ERR_DTYPE;
  const CUtensorMapDataType t = dt == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint64_t gdim[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  cuuint64_t gstride[2] = {(cuuint64_t)d0 * 2, (cuuint64_t)(d1 * d0 * 2)};
  cuuint32_t box[3] = {(cuuint32_t)b0, (cuuint32_t)b1, (cuuint32_t)b2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, t, 3, const_cast<void*>(base), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int make_u8_tensor_map(CUtensorMap* map, const void* base, int64_t rows, int32_t head_dim, int32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  // The copy moves bytes unchanged, so the rows are described as 16-bit
  // elements (half as many per row): the same 128-byte box rows and swizzle.
  cuuint64_t gdim[2] = {(cuuint64_t)head_dim / 2, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)head_dim};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), gdim, gstride, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int make_kv_tensor_map(CUtensorMap* map, const void* base, int64_t rows, int32_t head_dim, pa_dtype dt,
                       int32_t box_rows) {
  return make_2d_tensor_map(map, base, rows, head_dim, head_dim, dt, box_rows, 64);
}

static int32_t auto_partition(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t max_seq_len) {
  // Work items are (sequence, partition, KV head group); the persistent
  // decode kernel (two CTAs per SM) pulls them from a counter. Use the
  // longest partition (at most 4096 tokens, and at most half the longest
  // sequence so long sequences still split) that gives about four items per
  // SM, assuming an average length of half the maximum. Longer partitions
  // mean fewer per-item epilogues and partials; more items, a shorter tail.
  const int32_t group = num_q_heads / num_kv_heads;
  const int64_t hr = (int64_t)num_kv_heads * ((group + 15) / 16);
  const int64_t target = 4LL * num_sms_current_device();
  const int64_t half = (max_seq_len + 1) / 2;
  int32_t part = 4096;
  while (part > 256 && (part > half || (int64_t)num_seqs * hr * ((half + part - 1) / part) < target)) part /= 2;
  return part;
}

// Host check of copy-on-write pairs: every block in range, no destination
// repeated or also a source. On success src / dst hold the pairs.
static int check_copy_pairs(const int64_t* src_dst_pairs, int32_t num_pairs, int32_t num_blocks,
                            std::vector<int32_t>& src, std::vector<int32_t>& dst) {
  src.resize(num_pairs);
  dst.resize(num_pairs);
  std::unordered_set<int64_t> dsts;
  dsts.reserve(num_pairs * 2);
  for (int32_t i = 0; i < num_pairs; ++i) {
    const int64_t s = src_dst_pairs[2 * i], d = src_dst_pairs[2 * i + 1];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) return PA_ERR_BLOCK_OOB;
    if (!dsts.insert(d).second) return PA_ERR_ALIAS;
    src[i] = (int32_t)s;
    dst[i] = (int32_t)d;
  }
  for (int32_t i = 0; i < num_pairs; ++i)
    if (dsts.count(src[i])) return PA_ERR_ALIAS;
  return PA_OK;
}

// The cache side of a one-call decode step: copy-on-write copies, slots and
// the cache write of the step's new tokens. check() makes every host check
// of pa_copy_blocks, pa_slot_mapping and pa_reshape_and_cache before
// anything is launched; launch() issues the kernels, as programmatic
// dependents of the previous kernel when chained.
struct StepCacheSide {
  const int64_t* cow_pairs;
  int32_t num_cow_pairs;
  const int32_t* new_seq_ids;
  const int32_t* new_positions;
  const void* k_new;
  const void* v_new;
  int64_t num_new_tokens;
  int64_t* slot_mapping;
  void* k_cache;
  void* v_cache;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  int32_t num_seqs;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t num_blocks;
  pa_dtype dtype;
  std::vector<int32_t> src, dst;
  int64_t row_bytes = 0;
  int* status = nullptr;

  int check() {
    if (num_cow_pairs < 0 || num_new_tokens < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 1 ||
        max_blocks_per_seq < 1 || num_seqs < 0)
      return PA_ERR_ARG;
    if (block_size != 16 && block_size != 32) return PA_ERR_BLOCKSIZE;
    const int eb = elem_bytes(dtype);
    if (!eb || dtype == PA_F32) return PA_ERR_DTYPE;
    row_bytes = (int64_t)head_dim * eb;
    if (row_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (!k_cache || !v_cache) return PA_ERR_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;
    if (num_cow_pairs > 0) {
      if (!cow_pairs) return PA_ERR_ARG;
      const int rc = check_copy_pairs(cow_pairs, num_cow_pairs, num_blocks, src, dst);
      if (rc != PA_OK) return rc;
    }
    if (num_new_tokens > 0) {
      if (!new_seq_ids || !new_positions || !k_new || !v_new || !slot_mapping || !block_tables) return PA_ERR_ARG;
      if (!aligned16(k_new) || !aligned16(v_new)) return PA_ERR_ALIGN;
    }
    status = device_status_ptr();
    return status ? PA_OK : PA_ERR_CUDA;
  }

  int launch(cudaStream_t s, bool chained) {
    int rc = PA_OK;
    if (num_cow_pairs > 0)
      rc = launch_copy_blocks(k_cache, v_cache, src.data(), dst.data(), num_cow_pairs,
                              (int64_t)num_kv_heads * block_size * row_bytes, s, chained);
    if (rc == PA_OK && num_new_tokens > 0)
      rc = launch_slot_mapping(block_tables, max_blocks_per_seq, num_seqs, new_seq_ids, new_positions,
                               num_new_tokens, block_size, num_blocks, slot_mapping, status, s, chained);
    if (rc == PA_OK && num_new_tokens > 0)
      rc = launch_reshape_and_cache(k_new, v_new, slot_mapping, num_new_tokens, k_cache, v_cache, num_blocks,
                                    block_size, num_kv_heads, (int32_t)row_bytes, status, s, chained);
    return rc;
  }
};

// Checks and parameter block of a decode launch. extra_slots = 1 reserves a
// partial slot per (sequence, head) for the prefix pass of shared-prefix
// decode. On success *wl is the decode workspace layout.
static int decode_prepare(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                          int32_t max_blocks_per_seq, const int32_t* lens, const int32_t* cu_q_lens,
                          int32_t num_seqs, int32_t max_len, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale, void* out,
                          int32_t partition_size, int32_t extra_slots, void* workspace, size_t workspace_bytes,
                          pa_dtype dtype, DecodeParams* dp, DecodeWorkspace* wl) {
  if (num_seqs < 0 || max_blocks_per_seq < 1 || num_blocks < 1 || head_dim < 1) return PA_ERR_ARG;
  if (num_q_heads < 1 || num_kv_heads < 1) return PA_ERR_ARG;
  if (num_q_heads % num_kv_heads) return PA_ERR_HEADS;
  if (block_size != 16 && block_size != 32) return PA_ERR_BLOCKSIZE;
  if (!elem_bytes(dtype)) return PA_ERR_DTYPE;
  if (!head_dim_supported(dtype, head_dim)) return PA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return PA_ERR_ARG;
  if (num_seqs == 0) return PA_OK;
  if (max_len < 1) return PA_ERR_ARG;
  if (num_seqs > 65535) return PA_ERR_UNSUPPORTED;
  if (!q || !k_cache || !v_cache || !block_tables || !lens || !out) return PA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PA_ERR_ALIGN;
  if ((int64_t)num_blocks * num_kv_heads * block_size >= (1LL << 31)) return PA_ERR_UNSUPPORTED;
  const int32_t part =
      pa_decode_partition_size(num_seqs, num_q_heads, num_kv_heads, block_size, max_len, partition_size);
  if (part < 0) return part;
  const int64_t max_parts = (max_len + part - 1) / part + extra_slots;
  if (max_parts > 12288) return PA_ERR_ARG;
  *wl = decode_workspace_layout(num_seqs, num_q_heads, head_dim, max_parts);
  if (!workspace || workspace_bytes < wl->total) return PA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return PA_ERR_ALIGN;
  int* st = device_status_ptr();
  if (!st) return PA_ERR_CUDA;

  DecodeParams p{};
  p.q = q;
  p.out = out;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.lens = lens;
  p.cu_q_lens = cu_q_lens;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.group = num_q_heads / num_kv_heads;
  p.partition = part;
  p.max_parts = (int32_t)max_parts;
  p.len_cap = max_len;
  p.scale_log2 = scale * 1.4426950408889634f;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.work = reinterpret_cast<int32_t*>(ws + wl->work);
  p.pairs = reinterpret_cast<int32_t*>(ws + wl->pairs);
  p.part_o = max_parts > 1 ? reinterpret_cast<float*>(ws + wl->part_o) : nullptr;
  p.part_ml = max_parts > 1 ? reinterpret_cast<float*>(ws + wl->part_ml) : nullptr;
  p.merge_list = max_parts > 1 ? reinterpret_cast<int4*>(ws + wl->merge) : nullptr;
  p.prefix = nullptr;
  p.slot0 = extra_slots;
  p.status = st;
  *dp = p;
  return PA_OK;
}

static int decode_common(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* lens, const int32_t* cu_q_lens,
                         int32_t num_seqs, int32_t max_len, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale, void* out,
                         int32_t partition_size, void* workspace, size_t workspace_bytes, pa_dtype dtype,
                         cudaStream_t stream) {
  DecodeParams p;
  DecodeWorkspace wl;
  const int rc = decode_prepare(q, k_cache, v_cache, block_tables, max_blocks_per_seq, lens, cu_q_lens, num_seqs,
                                max_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, out,
                                partition_size, 0, workspace, workspace_bytes, dtype, &p, &wl);
  if (rc != PA_OK || num_seqs == 0) return rc;
  return launch_decode(p, dtype, stream);
}

template <typename Between>
static int shared_prefix_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                            int32_t max_seq_len, const int32_t* group_starts, const int32_t* prefix_lens,
                            int32_t num_groups, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_blocks, float scale, void* out, int32_t partition_size,
                            void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream,
                            const float* kv_scales, int32_t kv_fmt, Between&& between) {
  if (num_seqs < 0 || num_groups < 0) return PA_ERR_ARG;
  if (num_seqs == 0) return between(false);
  if (num_groups < 1 || num_groups > num_seqs || !group_starts || !prefix_lens) return PA_ERR_ARG;
  if (dtype == PA_F32) return PA_ERR_DTYPE;
  if (!(scale > 0.f)) return PA_ERR_ARG;  // the prefix pass needs scale > 0
  if (head_dim != 128 && !(head_dim == 64 && !kv_scales)) return PA_ERR_UNSUPPORTED;
  if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads) return PA_ERR_HEADS;
  const int32_t g = num_q_heads / num_kv_heads;
  if (g > 128) return PA_ERR_UNSUPPORTED;
  const size_t need = pa_decode_shared_prefix_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                            block_size, max_seq_len, partition_size, num_groups);
  if (!workspace || workspace_bytes < need) return PA_ERR_WORKSPACE;
  DecodeParams dp;
  DecodeWorkspace wl;
  int rc = decode_prepare(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, nullptr, num_seqs,
                          max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, out,
                          partition_size, 1, workspace, workspace_bytes, dtype, &dp, &wl);
  if (rc != PA_OK) return rc;
  if (kv_scales && !aligned16(kv_scales)) return PA_ERR_ALIGN;
  dp.kv_scales = kv_scales;  // 8-bit cache (nullptr: the pools hold q's dtype)
  dp.kv_fmt = kv_fmt;
  const CascadeWorkspace cw = cascade_workspace_layout(num_seqs, num_groups);
  uint8_t* cbase = static_cast<uint8_t*>(workspace) + wl.total;
  int32_t* prefix = reinterpret_cast<int32_t*>(cbase + cw.prefix);
  int32_t* group_ref = reinterpret_cast<int32_t*>(cbase + cw.group_ref);
  int32_t* group_of_seq = reinterpret_cast<int32_t*>(cbase + cw.group_of);
  int32_t* pwork = reinterpret_cast<int32_t*>(cbase + cw.work);
  int32_t* ppairs = reinterpret_cast<int32_t*>(cbase + cw.pairs);
  int32_t* pkeys = reinterpret_cast<int32_t*>(cbase + cw.pair_keys);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dp.prefix = prefix;
  decode_set_rows(dp, dtype);
  // 1. Verify the hints, list the prefix pass's work and the suffix decode's.
  rc = launch_cascade_prep(dp, dtype, group_starts, prefix_lens, num_groups, prefill_positions_per_item(g), prefix,
                           group_ref, group_of_seq, pwork, ppairs, pkeys, s);
  dp.planned = 1;
  if (rc != PA_OK) return rc;
  // Whatever the caller launches here runs beside the check: it must not
  // write what the check reads (tables, lengths, hints, groups).
  rc = between(true);
  if (rc != PA_OK) return rc;
  // 2. Prefix pass (tcgen05): every group's shared blocks once for all its
  //    members, partials into slot 0.
  PrefillParams pp{};
  pp.q = q;
  pp.out = out;
  pp.block_tables = block_tables;
  pp.max_blocks_per_seq = max_blocks_per_seq;
  pp.num_seqs = num_seqs;
  pp.num_q_heads = num_q_heads;
  pp.num_kv_heads = num_kv_heads;
  pp.head_dim = head_dim;
  pp.block_size = block_size;
  pp.num_blocks = num_blocks;
  pp.group = g;
  pp.total_q = num_seqs;
  pp.scale_log2 = dp.scale_log2;
  pp.work = pwork;
  pp.pairs = ppairs;
  pp.group_starts = group_starts;
  pp.prefix = prefix;
  pp.group_ref = group_ref;
  pp.pair_keys = pkeys;
  pp.part_o = dp.part_o;
  pp.part_ml = dp.part_ml;
  pp.max_parts = dp.max_parts;
  pp.status = dp.status;
  pp.kv_scales = kv_scales;
  pp.kv_fmt = kv_fmt;
  rc = launch_prefix_pass(pp, k_cache, v_cache, dtype, s);
  if (rc != PA_OK) return rc;
  // 3. Suffix decode (split-KV over the private keys) and the merge.
  return launch_decode(dp, dtype, s);
}

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_strerror(int s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_ARG: return "PA_ERR_ARG: invalid argument";
    case PA_ERR_DTYPE: return "PA_ERR_DTYPE: dtype not supported here";
    case PA_ERR_HEADS: return "PA_ERR_HEADS: num_q_heads is not a multiple of num_kv_heads";
    case PA_ERR_BLOCKSIZE: return "PA_ERR_BLOCKSIZE: block_size must be 16 or 32";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing or too small";
    case PA_ERR_ALIAS: return "PA_ERR_ALIAS: copy_blocks destination repeated or also a source";
    case PA_ERR_BLOCK_OOB: return "PA_ERR_BLOCK_OOB: block id or slot outside the pool";
    case PA_ERR_SEQLEN: return "PA_ERR_SEQLEN: sequence length out of range";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA runtime error";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: shape not supported";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT: a bounded device wait ran out";
    case PA_ERR_ALIGN: return "PA_ERR_ALIGN: pointer not 16-byte aligned";
    case PA_ERR_SCRATCH: return "PA_ERR_SCRATCH: the call needs more than pa_decode_noalloc's fixed scratch";
  }
  return "unknown status";
}

int pa_version(void) { return 100; }

int pa_get_status(void* stream) {
  int* p = device_status_ptr();
  if (!p) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return PA_ERR_CUDA;
  const int zero = 0;
  if (v != 0 && cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return PA_ERR_CUDA;
  return v;
}

int pa_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq, int32_t num_seqs,
                    const int32_t* seq_ids, const int32_t* positions, int64_t num_tokens, int32_t block_size,
                    int32_t num_blocks, int64_t* slot_mapping, void* stream) {
  if (num_tokens < 0 || num_seqs < 0 || max_blocks_per_seq < 1 || num_blocks < 1) return PA_ERR_ARG;
  if (block_size != 16 && block_size != 32) return PA_ERR_BLOCKSIZE;
  if (num_tokens == 0) return PA_OK;
  if (!block_tables || !seq_ids || !positions || !slot_mapping) return PA_ERR_ARG;
  int* st = device_status_ptr();
  if (!st) return PA_ERR_CUDA;
  return launch_slot_mapping(block_tables, max_blocks_per_seq, num_seqs, seq_ids, positions, num_tokens, block_size,
                             num_blocks, slot_mapping, st, static_cast<cudaStream_t>(stream));
}

int pa_reshape_and_cache(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                         void* k_cache, void* v_cache, int32_t num_blocks, int32_t block_size,
                         int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype, void* stream) {
  if (num_tokens < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 1) return PA_ERR_ARG;
  if (block_size != 16 && block_size != 32) return PA_ERR_BLOCKSIZE;
  const int eb = elem_bytes(dtype);
  if (!eb) return PA_ERR_DTYPE;
  const int64_t row_bytes = (int64_t)head_dim * eb;
  if (row_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;
  int* st = device_status_ptr();
  if (!st) return PA_ERR_CUDA;
  return launch_reshape_and_cache(k, v, slot_mapping, num_tokens, k_cache, v_cache, num_blocks, block_size,
                                  num_kv_heads, (int32_t)row_bytes, st, static_cast<cudaStream_t>(stream));
}

int pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* src_dst_pairs, int32_t num_pairs,
                   int32_t num_blocks, int64_t block_bytes, void* stream) {
  if (num_pairs < 0 || num_blocks < 1 || block_bytes <= 0) return PA_ERR_ARG;
  if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !src_dst_pairs) return PA_ERR_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;
  std::vector<int32_t> src, dst;
  const int rc = check_copy_pairs(src_dst_pairs, num_pairs, num_blocks, src, dst);
  if (rc != PA_OK) return rc;
  return launch_copy_blocks(k_cache, v_cache, src.data(), dst.data(), num_pairs, block_bytes,
                            static_cast<cudaStream_t>(stream));
}

int32_t pa_decode_partition_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t block_size,
                                 int32_t max_seq_len, int32_t partition_size) {
  if (num_seqs < 0 || num_q_heads < 1 || num_kv_heads < 1 || max_seq_len < 0) return PA_ERR_ARG;
  if (num_q_heads % num_kv_heads) return PA_ERR_HEADS;
  if (block_size != 16 && block_size != 32) return PA_ERR_BLOCKSIZE;
  if (partition_size < 0) return PA_ERR_ARG;
  if (partition_size > 0) {
    if (partition_size % block_size || partition_size > kMaxPartition) return PA_ERR_ARG;
    return partition_size;
  }
  return auto_partition(num_seqs, num_q_heads, num_kv_heads, max_seq_len < 1 ? 1 : max_seq_len);
}

size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t block_size, int32_t max_seq_len, int32_t partition_size) {
  const int32_t part =
      pa_decode_partition_size(num_seqs, num_q_heads, num_kv_heads, block_size, max_seq_len, partition_size);
  if (part <= 0 || head_dim < 1 || num_seqs < 1) return 0;
  const int64_t max_parts = ((max_seq_len < 1 ? 1 : max_seq_len) + part - 1) / part;
  return decode_workspace_layout(num_seqs, num_q_heads, head_dim, max_parts).total;
}

int pa_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
              int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
              float scale, void* out, int32_t partition_size, void* workspace, size_t workspace_bytes,
              pa_dtype dtype, void* stream) {
  return decode_common(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, nullptr, num_seqs,
                       max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, out,
                       partition_size, workspace, workspace_bytes, dtype, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace pa {
static int decode_fp8(const void* q, const void* k_cache, const void* v_cache, const float* kv_scales,
                      const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                      int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale, void* out,
                      int32_t partition_size, void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream,
                      int32_t kv_fmt) {
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_DTYPE;
  if (head_dim != 128) return PA_ERR_UNSUPPORTED;
  DecodeParams p;
  DecodeWorkspace wl;
  const int rc = decode_prepare(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, nullptr, num_seqs,
                                max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, out,
                                partition_size, 0, workspace, workspace_bytes, dtype, &p, &wl);
  if (rc != PA_OK || num_seqs == 0) return rc;
  if (!kv_scales) return PA_ERR_ARG;
  if (!aligned16(kv_scales)) return PA_ERR_ALIGN;
  p.kv_scales = kv_scales;
  p.kv_fmt = kv_fmt;
  return launch_decode(p, dtype, static_cast<cudaStream_t>(stream));
}

static int reshape_and_cache_fp8(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                                 void* k_cache, void* v_cache, float* kv_scales, int32_t num_blocks,
                                 int32_t block_size, int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype,
                                 void* stream, int32_t kv_fmt) {
  if (num_tokens < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 1) return PA_ERR_ARG;
  if (block_size != 16 && block_size != 32) return PA_ERR_BLOCKSIZE;
  if (!elem_bytes(dtype)) return PA_ERR_DTYPE;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache || !kv_scales) return PA_ERR_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(kv_scales))
    return PA_ERR_ALIGN;
  int* st = device_status_ptr();
  if (!st) return PA_ERR_CUDA;
  return launch_reshape_and_cache_fp8(k, v, slot_mapping, num_tokens, static_cast<uint8_t*>(k_cache),
                                      static_cast<uint8_t*>(v_cache), kv_scales, num_blocks, block_size,
                                      num_kv_heads, head_dim, dtype, kv_fmt, st, static_cast<cudaStream_t>(stream));
}
}  // namespace pa

extern "C" {

int pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache, const float* kv_scales,
                  const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                  int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t block_size, int32_t num_blocks, float scale, void* out, int32_t partition_size,
                  void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream) {
  return decode_fp8(q, k_cache, v_cache, kv_scales, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                    max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, out,
                    partition_size, workspace, workspace_bytes, dtype, stream, PA_KV_E4M3);
}

int pa_decode_e5m2(const void* q, const void* k_cache, const void* v_cache, const float* kv_scales,
                   const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                   int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                   int32_t block_size, int32_t num_blocks, float scale, void* out, int32_t partition_size,
                   void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream) {
  return decode_fp8(q, k_cache, v_cache, kv_scales, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                    max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, out,
                    partition_size, workspace, workspace_bytes, dtype, stream, PA_KV_E5M2);
}

int pa_reshape_and_cache_fp8(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                             void* k_cache, void* v_cache, float* kv_scales, int32_t num_blocks, int32_t block_size,
                             int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype, void* stream) {
  return reshape_and_cache_fp8(k, v, slot_mapping, num_tokens, k_cache, v_cache, kv_scales, num_blocks, block_size,
                               num_kv_heads, head_dim, dtype, stream, PA_KV_E4M3);
}

int pa_reshape_and_cache_e5m2(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                              void* k_cache, void* v_cache, float* kv_scales, int32_t num_blocks, int32_t block_size,
                              int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype, void* stream) {
  return reshape_and_cache_fp8(k, v, slot_mapping, num_tokens, k_cache, v_cache, kv_scales, num_blocks, block_size,
                               num_kv_heads, head_dim, dtype, stream, PA_KV_E5M2);
}

int pa_copy_blocks_fp8(void* k_cache, void* v_cache, float* kv_scales, const int64_t* src_dst_pairs,
                       int32_t num_pairs, int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                       int32_t head_dim, void* stream) {
  if (num_pairs < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 1) return PA_ERR_ARG;
  if (block_size != 16 && block_size != 32) return PA_ERR_BLOCKSIZE;
  if (num_pairs == 0) return PA_OK;
  if (!kv_scales) return PA_ERR_ARG;
  const int64_t block_bytes = (int64_t)num_kv_heads * block_size * head_dim;
  // Codes first (validates the pairs), then the scales of the same pairs.
  const int rc = pa_copy_blocks(k_cache, v_cache, src_dst_pairs, num_pairs, num_blocks, block_bytes, stream);
  if (rc != PA_OK) return rc;
  std::vector<int32_t> src(num_pairs), dst(num_pairs);
  for (int32_t i = 0; i < num_pairs; ++i) {
    src[i] = (int32_t)src_dst_pairs[2 * i];
    dst[i] = (int32_t)src_dst_pairs[2 * i + 1];
  }
  return launch_copy_scales(kv_scales, src.data(), dst.data(), num_pairs, num_kv_heads,
                            static_cast<cudaStream_t>(stream));
}

// A pointer the GPU can dereference for this pool (device, managed or pinned
// host memory), or nullptr if it cannot (pageable host memory).
static const void* device_usable(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of the query
    return nullptr;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged: return p;
    case cudaMemoryTypeHost: return a.devicePointer;
    default: return nullptr;
  }
}

int pa_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v, const int64_t* src_dst_pairs,
                   int32_t num_pairs, int32_t src_num_blocks, int32_t dst_num_blocks, int64_t block_bytes,
                   void* stream) {
  if (num_pairs < 0 || src_num_blocks < 1 || dst_num_blocks < 1 || block_bytes <= 0) return PA_ERR_ARG;
  if (block_bytes % 4 != 0) return PA_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PA_OK;
  if (!src_k || !dst_k || !src_dst_pairs || (src_v == nullptr) != (dst_v == nullptr)) return PA_ERR_ARG;
  const bool same_pool = src_k == dst_k;
  std::vector<int32_t> src(num_pairs), dst(num_pairs);
  std::unordered_set<int64_t> dsts;
  dsts.reserve(num_pairs * 2);
  for (int32_t i = 0; i < num_pairs; ++i) {
    const int64_t s = src_dst_pairs[2 * i], d = src_dst_pairs[2 * i + 1];
    if (s < 0 || s >= src_num_blocks || d < 0 || d >= dst_num_blocks) return PA_ERR_BLOCK_OOB;
    if (!dsts.insert(d).second) return PA_ERR_ALIAS;
    src[i] = (int32_t)s;
    dst[i] = (int32_t)d;
  }
  if (same_pool)
    for (int32_t i = 0; i < num_pairs; ++i)
      if (dsts.count(src[i])) return PA_ERR_ALIAS;
  const void* sk = device_usable(src_k);
  const void* dk = device_usable(dst_k);
  const void* sv = src_v ? device_usable(src_v) : nullptr;
  const void* dv = dst_v ? device_usable(dst_v) : nullptr;
  if (!sk || !dk || (src_v && (!sv || !dv))) return PA_ERR_ARG;
  const int vec16 = block_bytes % 16 == 0 && aligned16(sk) && aligned16(dk) && (!sv || (aligned16(sv) && aligned16(dv)));
  return launch_swap_blocks(sk, sv, const_cast<void*>(dk), const_cast<void*>(dv), src.data(), dst.data(), num_pairs,
                            block_bytes, vec16, static_cast<cudaStream_t>(stream));
}

size_t pa_decode_shared_prefix_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                              int32_t head_dim, int32_t block_size, int32_t max_seq_len,
                                              int32_t partition_size, int32_t num_groups) {
  const int32_t part =
      pa_decode_partition_size(num_seqs, num_q_heads, num_kv_heads, block_size, max_seq_len, partition_size);
  if (part <= 0 || head_dim < 1 || num_seqs < 1 || num_groups < 1) return 0;
  const int64_t max_parts = ((max_seq_len < 1 ? 1 : max_seq_len) + part - 1) / part + 1;
  return decode_workspace_layout(num_seqs, num_q_heads, head_dim, max_parts).total +
         cascade_workspace_layout(num_seqs, num_groups).total;
}

int pa_decode_shared_prefix(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                            int32_t max_seq_len, const int32_t* group_starts, const int32_t* prefix_lens,
                            int32_t num_groups, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_blocks, float scale, void* out, int32_t partition_size,
                            void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream) {
  return shared_prefix_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                              group_starts, prefix_lens, num_groups, num_q_heads, num_kv_heads, head_dim, block_size,
                              num_blocks, scale, out, partition_size, workspace, workspace_bytes, dtype, stream,
                              nullptr, PA_KV_E4M3, [](bool) { return PA_OK; });
}

int pa_decode_shared_prefix_fp8(const void* q, const void* k_cache, const void* v_cache, const float* kv_scales,
                                const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                int32_t num_seqs, int32_t max_seq_len, const int32_t* group_starts,
                                const int32_t* prefix_lens, int32_t num_groups, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                float scale, void* out, int32_t partition_size, void* workspace,
                                size_t workspace_bytes, pa_dtype dtype, void* stream) {
  if (num_seqs > 0 && !kv_scales) return PA_ERR_ARG;
  return shared_prefix_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                              group_starts, prefix_lens, num_groups, num_q_heads, num_kv_heads, head_dim, block_size,
                              num_blocks, scale, out, partition_size, workspace, workspace_bytes, dtype, stream,
                              kv_scales, PA_KV_E4M3, [](bool) { return PA_OK; });
}

int pa_decode_shared_prefix_e5m2(const void* q, const void* k_cache, const void* v_cache, const float* kv_scales,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                 int32_t num_seqs, int32_t max_seq_len, const int32_t* group_starts,
                                 const int32_t* prefix_lens, int32_t num_groups, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                 float scale, void* out, int32_t partition_size, void* workspace,
                                 size_t workspace_bytes, pa_dtype dtype, void* stream) {
  if (num_seqs > 0 && !kv_scales) return PA_ERR_ARG;
  return shared_prefix_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                              group_starts, prefix_lens, num_groups, num_q_heads, num_kv_heads, head_dim, block_size,
                              num_blocks, scale, out, partition_size, workspace, workspace_bytes, dtype, stream,
                              kv_scales, PA_KV_E5M2, [](bool) { return PA_OK; });
}

int pa_decode_step_shared_prefix(const int64_t* cow_pairs, int32_t num_cow_pairs, const int32_t* new_seq_ids,
                                 const int32_t* new_positions, const void* k_new, const void* v_new,
                                 int64_t num_new_tokens, int64_t* slot_mapping, const void* q, void* k_cache,
                                 void* v_cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                                 const int32_t* group_starts, const int32_t* prefix_lens, int32_t num_groups,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int32_t num_blocks, float scale, void* out, int32_t partition_size, void* workspace,
                                 size_t workspace_bytes, pa_dtype dtype, void* stream) {
  // Host checks of the cache side, as the separate calls make them; the
  // decode's own checks run inside shared_prefix_decode before any launch,
  // so a rejected call launches nothing.
  StepCacheSide cs{cow_pairs,    num_cow_pairs, new_seq_ids,        new_positions, k_new,      v_new,
                   num_new_tokens, slot_mapping, k_cache,           v_cache,       block_tables, max_blocks_per_seq,
                   num_seqs,     num_kv_heads,  head_dim,           block_size,    num_blocks, dtype};
  int rc = cs.check();
  if (rc != PA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The cache side runs after the prefix check is launched, chained
  // (programmatic dependents) when it runs beside it; none of its kernels
  // writes what the check reads.
  auto cache_side = [&](bool chained) -> int { return cs.launch(s, chained); };
  return shared_prefix_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                              group_starts, prefix_lens, num_groups, num_q_heads, num_kv_heads, head_dim, block_size,
                              num_blocks, scale, out, partition_size, workspace, workspace_bytes, dtype, stream,
                              nullptr, PA_KV_E4M3, cache_side);
}

int pa_decode_step(const int64_t* cow_pairs, int32_t num_cow_pairs, const int32_t* new_seq_ids,
                   const int32_t* new_positions, const void* k_new, const void* v_new, int64_t num_new_tokens,
                   int64_t* slot_mapping, const void* q, void* k_cache, void* v_cache, const int32_t* block_tables,
                   int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                   int32_t num_blocks, float scale, void* out, int32_t partition_size, void* workspace,
                   size_t workspace_bytes, pa_dtype dtype, void* stream) {
  StepCacheSide cs{cow_pairs,    num_cow_pairs, new_seq_ids,        new_positions, k_new,      v_new,
                   num_new_tokens, slot_mapping, k_cache,           v_cache,       block_tables, max_blocks_per_seq,
                   num_seqs,     num_kv_heads,  head_dim,           block_size,    num_blocks, dtype};
  int rc = cs.check();
  if (rc != PA_OK) return rc;
  DecodeParams p;
  DecodeWorkspace wl;
  rc = decode_prepare(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, nullptr, num_seqs,
                      max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, out,
                      partition_size, 0, workspace, workspace_bytes, dtype, &p, &wl);
  if (rc != PA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (num_seqs == 0) return cs.launch(s, false);
  // The plan reads only the tables and lengths, which the cache side does
  // not write: it goes first and the cache side runs beside it, chained; the
  // decode kernel waits for the cache write (hence for all of them).
  rc = launch_decode_plan(p, dtype, s);
  if (rc != PA_OK) return rc;
  rc = cs.launch(s, true);
  if (rc != PA_OK) return rc;
  p.planned = 1;
  return launch_decode(p, dtype, s);
}

size_t pa_chunked_prefill_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t block_size, int32_t total_q, int32_t max_kv_len) {
  const size_t dec =
      pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_kv_len, 0);
  if (dec == 0) return 0;
  // + the chunk-tile work list: a counter pair and at most total_q tiles.
  return dec + (((size_t)16 + (size_t)(total_q > 0 ? total_q : 0) * 4 + 255) & ~size_t(255));
}

}  // extern "C"

namespace pa {
// Mixed batch (chunks and decode rows) over 16-bit pools, or over 8-bit
// pools (format kv_fmt) when kv_scales is given.
static int chunked_prefill(const void* q, int32_t total_q, const int32_t* cu_q_lens, const void* k_cache,
                           const void* v_cache, const float* kv_scales, int32_t kv_fmt, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* ctx_lens, int32_t num_seqs, int32_t max_q_len,
                           int32_t max_kv_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int32_t num_blocks, float scale, void* out, void* workspace,
                           size_t workspace_bytes, pa_dtype dtype, void* stream) {
  if (num_seqs < 0 || max_q_len < 0 || max_kv_len < 0 || total_q < 0) return PA_ERR_ARG;
  if (num_seqs == 0 || max_q_len == 0 || total_q == 0) return PA_OK;
  if (!cu_q_lens || !ctx_lens) return PA_ERR_ARG;
  // Chunks (q_len > 1): fp16 / bf16 on the tensor-core kernel, fp32 on the
  // CUDA-core kernel (exact fp32; any scale and decode head_dim).
  if (max_q_len > 1 && dtype != PA_F32) {
    if (!(scale > 0.f)) return PA_ERR_ARG;  // the tensor-core chunk kernel needs scale > 0
    if (head_dim != 128 && !(head_dim == 64 && !kv_scales)) return PA_ERR_UNSUPPORTED;
    if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads) return PA_ERR_HEADS;
    const int32_t g = num_q_heads / num_kv_heads;
    if (g > 128) return PA_ERR_UNSUPPORTED;
  }
  if (max_q_len > 1 && max_q_len > total_q) return PA_ERR_ARG;
  const size_t dec_ws =
      pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_kv_len, 0);
  if (!workspace ||
      workspace_bytes < pa_chunked_prefill_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                          block_size, total_q, max_kv_len))
    return PA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Decode rows (q_len == 1): the split-KV decode path, key count ctx + 1.
  DecodeParams dp;
  DecodeWorkspace wl;
  int rc = decode_prepare(q, k_cache, v_cache, block_tables, max_blocks_per_seq, ctx_lens, cu_q_lens, num_seqs,
                          max_kv_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, out, 0, 0,
                          workspace, dec_ws, dtype, &dp, &wl);
  if (rc != PA_OK) return rc;
  if (kv_scales) {
    if (!aligned16(kv_scales)) return PA_ERR_ALIGN;
    dp.kv_scales = kv_scales;
    dp.kv_fmt = kv_fmt;
  }
  if (max_q_len <= 1) return launch_decode(dp, dtype, s);
  if (dtype == PA_F32) {
    // Decode rows on the fp32 decode path, then the chunk rows.
    rc = launch_decode(dp, dtype, s);
    if (rc != PA_OK) return rc;
    return launch_prefill_simt(dp, total_q, s);
  }
  // Chunks (q_len > 1): tcgen05 tiles. One plan lists the chunk items and
  // the decode rows' partitions and splits the SMs between them; the chunk
  // kernel runs on its share and the decode kernel beside it on the rest.
  PrefillParams p{};
  p.q = q;
  p.out = out;
  p.block_tables = block_tables;
  p.cu_q_lens = cu_q_lens;
  p.ctx_lens = ctx_lens;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.group = num_q_heads / num_kv_heads;
  p.max_q_len = max_q_len;
  p.max_kv_len = max_kv_len;
  p.total_q = total_q;
  p.scale_log2 = scale * 1.4426950408889634f;
  uint8_t* pw = static_cast<uint8_t*>(workspace) + dec_ws;
  p.work = reinterpret_cast<int32_t*>(pw);
  p.pairs = reinterpret_cast<int32_t*>(pw + 16);
  p.status = dp.status;
  p.decode_token_bytes = 2 * num_kv_heads * head_dim * elem_bytes(dtype);
  p.decode_bytes_per_tile = kDecodeBytesPerChunkTile;
  p.kv_scales = kv_scales;
  p.kv_fmt = kv_fmt;
  rc = launch_prefill(p, k_cache, v_cache, dtype, s, &dp);
  if (rc != PA_OK) return rc;
  dp.planned = 1;
  dp.beside = 1;
  return launch_decode(dp, dtype, s);
}
}  // namespace pa

extern "C" {

int pa_chunked_prefill(const void* q, int32_t total_q, const int32_t* cu_q_lens, const void* k_cache,
                       const void* v_cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* ctx_lens, int32_t num_seqs, int32_t max_q_len, int32_t max_kv_len,
                       int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                       int32_t num_blocks, float scale, void* out, void* workspace, size_t workspace_bytes,
                       pa_dtype dtype, void* stream) {
  return chunked_prefill(q, total_q, cu_q_lens, k_cache, v_cache, nullptr, PA_KV_E4M3, block_tables, max_blocks_per_seq,
                         ctx_lens, num_seqs, max_q_len, max_kv_len, num_q_heads, num_kv_heads, head_dim, block_size,
                         num_blocks, scale, out, workspace, workspace_bytes, dtype, stream);
}

int pa_chunked_prefill_fp8(const void* q, int32_t total_q, const int32_t* cu_q_lens, const void* k_cache,
                           const void* v_cache, const float* kv_scales, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* ctx_lens, int32_t num_seqs, int32_t max_q_len,
                           int32_t max_kv_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int32_t num_blocks, float scale, void* out, void* workspace,
                           size_t workspace_bytes, pa_dtype dtype, void* stream) {
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_DTYPE;
  if (head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (num_seqs > 0 && total_q > 0 && !kv_scales) return PA_ERR_ARG;
  return chunked_prefill(q, total_q, cu_q_lens, k_cache, v_cache, kv_scales, PA_KV_E4M3, block_tables,
                         max_blocks_per_seq, ctx_lens, num_seqs, max_q_len, max_kv_len, num_q_heads, num_kv_heads,
                         head_dim, block_size, num_blocks, scale, out, workspace, workspace_bytes, dtype, stream);
}

int pa_chunked_prefill_e5m2(const void* q, int32_t total_q, const int32_t* cu_q_lens, const void* k_cache,
                            const void* v_cache, const float* kv_scales, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* ctx_lens, int32_t num_seqs, int32_t max_q_len,
                            int32_t max_kv_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_blocks, float scale, void* out, void* workspace,
                            size_t workspace_bytes, pa_dtype dtype, void* stream) {
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_DTYPE;
  if (head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (num_seqs > 0 && total_q > 0 && !kv_scales) return PA_ERR_ARG;
  return chunked_prefill(q, total_q, cu_q_lens, k_cache, v_cache, kv_scales, PA_KV_E5M2, block_tables,
                         max_blocks_per_seq, ctx_lens, num_seqs, max_q_len, max_kv_len, num_q_heads, num_kv_heads,
                         head_dim, block_size, num_blocks, scale, out, workspace, workspace_bytes, dtype, stream);
}

}  // extern "C"
