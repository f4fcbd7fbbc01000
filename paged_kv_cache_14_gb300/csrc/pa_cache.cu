// Cache-side kernels: slot derivation, the paged KV write (reshape_and_cache)
// and whole-block copy-on-write copies. All three are bandwidth-trivial,
// bit-exact moves of 16-byte vectors.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

// slot = block_tables[seq][pos / B] * B + pos % B (logical block index and
// block offset, section 1.2 of the "High-Throughput Local LLM
// Infrastructure" page).
__global__ void slot_mapping_kernel(const int32_t* __restrict__ block_tables, int32_t max_blocks_per_seq,
                                    int32_t num_seqs, const int32_t* __restrict__ seq_ids,
                                    const int32_t* __restrict__ positions, int64_t num_tokens, int32_t block_size,
                                    int32_t num_blocks, int64_t* __restrict__ slot_mapping, int* status) {
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < num_tokens;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int32_t s = seq_ids[t];
    const int32_t pos = positions[t];
    int64_t slot = -1;
    if (s >= 0 && s < num_seqs && pos >= 0 && pos / block_size < max_blocks_per_seq) {
      const int32_t phys = block_tables[(int64_t)s * max_blocks_per_seq + pos / block_size];
      if (phys >= 0 && phys < num_blocks) slot = (int64_t)phys * block_size + pos % block_size;
    }
    if (slot < 0) record_error(status, PA_ERR_BLOCK_OOB);
    slot_mapping[t] = slot;
  }
}

// One warp per (token, KV head) row of row_bytes bytes; lanes move 16-byte
// vectors. cache[slot / B][h][slot % B][:] = new[t][h][:].
__global__ void reshape_and_cache_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
                                         const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
                                         uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                                         int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                         int32_t row_bytes, int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t total_rows = num_tokens * num_kv_heads;
  const int vec_per_row = row_bytes >> 4;
  for (int64_t r = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); r < total_rows; r += warps) {
    const int64_t t = r / num_kv_heads;
    const int32_t h = (int32_t)(r - t * num_kv_heads);
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;  // padding token
    if (slot >= (int64_t)num_blocks * block_size) {
      if (lane == 0) record_error(status, PA_ERR_BLOCK_OOB);
      continue;
    }
    const int64_t blk = slot / block_size;
    const int64_t off = slot - blk * block_size;
    const int64_t dst_row = (blk * num_kv_heads + h) * block_size + off;
    const int4* ks = reinterpret_cast<const int4*>(k + r * row_bytes);
    const int4* vs = reinterpret_cast<const int4*>(v + r * row_bytes);
    int4* kd = reinterpret_cast<int4*>(k_cache + dst_row * row_bytes);
    int4* vd = reinterpret_cast<int4*>(v_cache + dst_row * row_bytes);
    for (int i = lane; i < vec_per_row; i += 32) {
      kd[i] = ks[i];
      vd[i] = vs[i];
    }
  }
}

struct CopyPairs {
  int32_t src[kCopyPairsPerLaunch];
  int32_t dst[kCopyPairsPerLaunch];
};

// grid = (num_pairs, 2): y selects the K or the V pool. Each CTA copies one
// whole block (all KV heads) with 16-byte vectors.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint8_t* __restrict__ k_cache,
                                                          uint8_t* __restrict__ v_cache,
                                                          const __grid_constant__ CopyPairs pairs,
                                                          int64_t block_bytes) {
  uint8_t* pool = blockIdx.y == 0 ? k_cache : v_cache;
  const int4* src = reinterpret_cast<const int4*>(pool + (int64_t)pairs.src[blockIdx.x] * block_bytes);
  int4* dst = reinterpret_cast<int4*>(pool + (int64_t)pairs.dst[blockIdx.x] * block_bytes);
  const int64_t n = block_bytes >> 4;
  int64_t i = threadIdx.x;
  // Four independent 16-byte loads in flight per thread.
  for (; i + 3 * 256 < n; i += 4 * 256) {
    int4 a = src[i], b = src[i + 256], c = src[i + 512], d = src[i + 768];
    dst[i] = a;
    dst[i + 256] = b;
    dst[i + 512] = c;
    dst[i + 768] = d;
  }
  for (; i < n; i += 256) dst[i] = src[i];
}

static int grid_for(int64_t work, int per_block) {
  int64_t g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > 65535LL * 32) g = 65535LL * 32;
  return (int)g;
}

int launch_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq, int32_t num_seqs,
                        const int32_t* seq_ids, const int32_t* positions, int64_t num_tokens, int32_t block_size,
                        int32_t num_blocks, int64_t* slot_mapping, int* status, cudaStream_t stream) {
  slot_mapping_kernel<<<grid_for(num_tokens, 256), 256, 0, stream>>>(
      block_tables, max_blocks_per_seq, num_seqs, seq_ids, positions, num_tokens, block_size, num_blocks,
      slot_mapping, status);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_reshape_and_cache(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                             void* k_cache, void* v_cache, int32_t num_blocks, int32_t block_size,
                             int32_t num_kv_heads, int32_t row_bytes, int* status, cudaStream_t stream) {
  const int64_t rows = num_tokens * num_kv_heads;
  reshape_and_cache_kernel<<<grid_for(rows, 8), 256, 0, stream>>>(
      static_cast<const uint8_t*>(k), static_cast<const uint8_t*>(v), slot_mapping, num_tokens,
      static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), num_blocks, block_size, num_kv_heads,
      row_bytes, status);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int32_t num_pairs,
                       int64_t block_bytes, cudaStream_t stream) {
  for (int32_t base = 0; base < num_pairs; base += kCopyPairsPerLaunch) {
    const int32_t n = num_pairs - base < kCopyPairsPerLaunch ? num_pairs - base : kCopyPairsPerLaunch;
    CopyPairs pairs;
    for (int32_t i = 0; i < n; ++i) {
      pairs.src[i] = src[base + i];
      pairs.dst[i] = dst[base + i];
    }
    copy_blocks_kernel<<<dim3(n, 2), 256, 0, stream>>>(static_cast<uint8_t*>(k_cache),
                                                       static_cast<uint8_t*>(v_cache), pairs, block_bytes);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

}  // namespace pa
