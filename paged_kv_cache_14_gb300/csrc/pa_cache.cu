// Cache-side kernels: slot derivation, the paged KV write (reshape_and_cache)
// and whole-block copy-on-write copies. All three are bandwidth-trivial,
// bit-exact moves of 16-byte vectors.
//
// In a chained step (launched as programmatic dependents, see
// launch_dependent) slot derivation and block copies read nothing their
// predecessor writes: they let their successor start at once and wait for
// the predecessor only before exiting, so each one's completion still
// implies every earlier kernel's. The cache write reads the slots, so it
// waits first. Launched the ordinary way these calls are no-ops.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

struct CopyPairsScales {
  int32_t src[kCopyPairsPerLaunch];
  int32_t dst[kCopyPairsPerLaunch];
};

// slot = block_tables[seq][pos / B] * B + pos % B (logical block index and
// block offset, section 1.2 of the "High-Throughput Local LLM
// Infrastructure" page).
__global__ void slot_mapping_kernel(const int32_t* __restrict__ block_tables, int32_t max_blocks_per_seq,
                                    int32_t num_seqs, const int32_t* __restrict__ seq_ids,
                                    const int32_t* __restrict__ positions, int64_t num_tokens, int32_t block_size,
                                    int32_t num_blocks, int64_t* __restrict__ slot_mapping, int* status) {
  pdl_trigger();
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
  pdl_wait();
}

// One warp per (token, KV head) row of row_bytes bytes; lanes move 16-byte
// vectors. cache[slot / B][h][slot % B][:] = new[t][h][:].
__global__ void reshape_and_cache_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
                                         const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
                                         uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                                         int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                         int32_t row_bytes, int* status) {
  pdl_wait();  // the slots (and, in a chained step, every earlier kernel)
  pdl_trigger();
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

// ---------------------------------------------------------------------------
// 8-bit cache write (e4m3, or e5m2 with E5) with one scale per (block, KV
// head) and pool. The rows a
// call writes into one block are consecutive entries of the slot mapping
// (padding entries may sit between them); the first of them leads a warp
// per (KV head, pool) that
//   1. takes a = the largest |x| of the run's rows and the lowest written
//      offset o_min;
//   2. forms s_new = max(s_old, a / fmax), fmax = 448 (e4m3) or 57344
//      (e5m2), the format's largest finite value, with s_old = 0 when the run
//      touches offset 0 (the block starts afresh), else the stored scale;
//   3. if the scale grew (and s_old > 0), re-encodes the codes at offsets
//      below o_min (the tokens already in the block) with ratio s_old / s_new;
//   4. encodes every row of the run as fp8(x / s_new) and stores s_new.
// Each step is one IEEE single-precision operation (division and product
// rounded to nearest) followed by the round-to-nearest-even, saturating
// conversion to the 8-bit format, so the codes are reproducible bit for bit.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_c(uint16_t c) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(c));
  return d;
}

__device__ __forceinline__ uint32_t e5m2x2_to_f16x2_c(uint16_t c) {
  uint32_t d;
  asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(d) : "h"(c));
  return d;
}

// Two floats to two 8-bit codes (e4m3, or e5m2 with E5): lo in the low byte.
template <bool E5>
__device__ __forceinline__ uint32_t f32x2_to_fp8x2(float lo, float hi) {
  uint16_t r;
  if constexpr (E5)
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int VEC>
__device__ __forceinline__ void store_codes(uint8_t* dst, const uint32_t (&c)[VEC / 2]) {
  if constexpr (VEC == 2) {
    *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(c[0]);
  } else if constexpr (VEC == 4) {
    *reinterpret_cast<uint32_t*>(dst) = c[0] | (c[1] << 16);
  }
}

template <int VEC, bool E5>
__device__ __forceinline__ void load_codes(const uint8_t* src, float (&x)[VEC]) {
  uint32_t w;
  if constexpr (VEC == 2) w = *reinterpret_cast<const uint16_t*>(src);
  else w = *reinterpret_cast<const uint32_t*>(src);
#pragma unroll
  for (int i = 0; i < VEC; i += 2) {
    const uint16_t c2 = static_cast<uint16_t>(w >> (8 * i));
    const uint32_t h2 = E5 ? e5m2x2_to_f16x2_c(c2) : e4m3x2_to_f16x2_c(c2);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
    x[i] = f.x;
    x[i + 1] = f.y;
  }
}

template <typename TI, int VEC, bool E5>
__global__ void __launch_bounds__(256) reshape_and_cache_fp8_kernel(
    const TI* __restrict__ k, const TI* __restrict__ v, const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
    uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache, float* __restrict__ kv_scales, int32_t num_blocks,
    int32_t block_size, int32_t num_kv_heads, int* status) {
  constexpr int D = VEC * 32;
  constexpr unsigned kFull = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t cap = (int64_t)num_blocks * block_size;
  const int64_t total = num_tokens * num_kv_heads * 2;
  for (int64_t w = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); w < total; w += warps) {
    const int64_t t = w / (num_kv_heads * 2);
    const int rem = (int)(w - t * num_kv_heads * 2);
    const int h = rem >> 1, pool = rem & 1;
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;  // padding token
    if (slot >= cap) {
      if (lane == 0 && rem == 0) record_error(status, PA_ERR_BLOCK_OOB);
      continue;
    }
    const int64_t blk = slot / block_size;
    // Lead only if the nearest earlier token with a valid slot lies in
    // another block (or there is none).
    bool leader = true;
    for (int64_t base = t - 1; base >= 0; base -= 32) {
      const int64_t j = base - lane;
      const int64_t sj = j >= 0 ? slot_mapping[j] : -1;
      const unsigned ok = __ballot_sync(kFull, j >= 0 && sj >= 0 && sj < cap);
      if (ok) {
        const int64_t sf = __shfl_sync(kFull, sj, __ffs(ok) - 1);  // lowest lane = latest token
        leader = sf / block_size != blk;
        break;
      }
    }
    if (!leader) continue;
    const TI* src = pool == 0 ? k : v;
    uint8_t* codes = (pool == 0 ? k_cache : v_cache) + (blk * num_kv_heads + h) * (int64_t)block_size * D;
    // 1. The run's rows: amax and the lowest offset; `end` = one past the run.
    float amax = 0.f;
    int omin = block_size;
    int64_t end = num_tokens;
    for (int64_t base = t; base < num_tokens; base += 32) {
      const int64_t j = base + lane;
      const int64_t sj = j < num_tokens ? slot_mapping[j] : -1;
      const bool okj = j < num_tokens && sj >= 0 && sj < cap;
      const unsigned other = __ballot_sync(kFull, okj && sj / block_size != blk);
      const int lim = other ? __ffs(other) - 1 : 32;
      unsigned mem = __ballot_sync(kFull, okj && sj / block_size == blk && lane < lim);
      while (mem) {
        const int ln = __ffs(mem) - 1;
        mem &= mem - 1;
        const int64_t sm = __shfl_sync(kFull, sj, ln);
        omin = min(omin, (int)(sm - blk * block_size));
        const TI* row = src + ((base + ln) * num_kv_heads + h) * D + lane * VEC;
#pragma unroll
        for (int i = 0; i < VEC; ++i) amax = fmaxf(amax, fabsf(to_f32(row[i])));
      }
      if (other) {
        end = base + lim;
        break;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
    // 2. The block's new scale.
    float* sp = kv_scales + (blk * num_kv_heads + h) * 2 + pool;
    const float s_old = omin == 0 ? 0.f : *sp;
    const float s_new = fmaxf(s_old, __fdiv_rn(amax, E5 ? 57344.f : 448.f));
    // 3. Re-encode the tokens already in the block if the scale grew.
    if (s_new > s_old && s_old > 0.f && omin > 0) {
      const float r = __fdiv_rn(s_old, s_new);
      for (int o = 0; o < omin; ++o) {
        uint8_t* cp = codes + (int64_t)o * D + lane * VEC;
        float x[VEC];
        load_codes<VEC, E5>(cp, x);
        uint32_t c[VEC / 2];
#pragma unroll
        for (int i = 0; i < VEC; i += 2) c[i / 2] = f32x2_to_fp8x2<E5>(__fmul_rn(x[i], r), __fmul_rn(x[i + 1], r));
        store_codes<VEC>(cp, c);
      }
    }
    // 4. Encode the run's rows.
    for (int64_t base = t; base < end; base += 32) {
      const int64_t j = base + lane;
      const int64_t sj = j < end ? slot_mapping[j] : -1;
      unsigned mem = __ballot_sync(kFull, j < end && sj >= 0 && sj < cap && sj / block_size == blk);
      while (mem) {
        const int ln = __ffs(mem) - 1;
        mem &= mem - 1;
        const int64_t sm = __shfl_sync(kFull, sj, ln);
        const TI* row = src + ((base + ln) * num_kv_heads + h) * D + lane * VEC;
        uint32_t c[VEC / 2];
#pragma unroll
        for (int i = 0; i < VEC; i += 2) {
          const float x0 = to_f32(row[i]), x1 = to_f32(row[i + 1]);
          c[i / 2] = s_new > 0.f ? f32x2_to_fp8x2<E5>(__fdiv_rn(x0, s_new), __fdiv_rn(x1, s_new)) : 0u;
        }
        store_codes<VEC>(codes + (sm - blk * block_size) * D + lane * VEC, c);
      }
    }
    if (lane == 0) *sp = s_new;
  }
}

// grid = num_pairs: the 2 * num_kv_heads scales of block dst <- those of src.
__global__ void __launch_bounds__(256) copy_scales_kernel(float* __restrict__ kv_scales,
                                                          const __grid_constant__ CopyPairsScales pairs,
                                                          int32_t per_block) {
  const float* src = kv_scales + (int64_t)pairs.src[blockIdx.x] * per_block;
  float* dst = kv_scales + (int64_t)pairs.dst[blockIdx.x] * per_block;
  for (int i = threadIdx.x; i < per_block; i += blockDim.x) dst[i] = src[i];
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
  pdl_trigger();
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
  pdl_wait();
}

// Swap preemption ("Inside vLLM...", section "Preemption Mechanics: Swapping
// vs. Recomputation"): whole blocks between two pools, either of which may be
// device memory or pinned host memory (the GPU reaches the latter directly,
// over NVLink-C2C on a Grace-Blackwell node). grid = (num_pairs, pools): y
// selects the K or the V pool; one CTA per block, four independent loads in
// flight per thread so remote host memory latency is covered.
__global__ void __launch_bounds__(256) swap_blocks_kernel(const uint8_t* __restrict__ src_k,
                                                          const uint8_t* __restrict__ src_v,
                                                          uint8_t* __restrict__ dst_k, uint8_t* __restrict__ dst_v,
                                                          const __grid_constant__ CopyPairs pairs,
                                                          int64_t block_bytes, int vec16) {
  const uint8_t* sp = (blockIdx.y == 0 ? src_k : src_v) + (int64_t)pairs.src[blockIdx.x] * block_bytes;
  uint8_t* dp = (blockIdx.y == 0 ? dst_k : dst_v) + (int64_t)pairs.dst[blockIdx.x] * block_bytes;
  if (vec16) {
    const int4* src = reinterpret_cast<const int4*>(sp);
    int4* dst = reinterpret_cast<int4*>(dp);
    const int64_t n = block_bytes >> 4;
    int64_t i = threadIdx.x;
    for (; i + 3 * 256 < n; i += 4 * 256) {
      int4 a = src[i], b = src[i + 256], c = src[i + 512], d = src[i + 768];
      dst[i] = a;
      dst[i + 256] = b;
      dst[i + 512] = c;
      dst[i + 768] = d;
    }
    for (; i < n; i += 256) dst[i] = src[i];
  } else {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(sp);
    uint32_t* dst = reinterpret_cast<uint32_t*>(dp);
    for (int64_t i = threadIdx.x; i < (block_bytes >> 2); i += 256) dst[i] = src[i];
  }
}

static int grid_for(int64_t work, int per_block) {
  int64_t g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > 65535LL * 32) g = 65535LL * 32;
  return (int)g;
}

int launch_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq, int32_t num_seqs,
                        const int32_t* seq_ids, const int32_t* positions, int64_t num_tokens, int32_t block_size,
                        int32_t num_blocks, int64_t* slot_mapping, int* status, cudaStream_t stream,
                        bool chained) {
  const dim3 grid(grid_for(num_tokens, 256));
  if (chained)
    return launch_dependent(slot_mapping_kernel, grid, dim3(256), 0, stream, block_tables, max_blocks_per_seq,
                            num_seqs, seq_ids, positions, num_tokens, block_size, num_blocks, slot_mapping,
                            status) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
  slot_mapping_kernel<<<grid, 256, 0, stream>>>(block_tables, max_blocks_per_seq, num_seqs, seq_ids, positions,
                                                num_tokens, block_size, num_blocks, slot_mapping, status);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_reshape_and_cache(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                             void* k_cache, void* v_cache, int32_t num_blocks, int32_t block_size,
                             int32_t num_kv_heads, int32_t row_bytes, int* status, cudaStream_t stream,
                             bool chained) {
  const int64_t rows = num_tokens * num_kv_heads;
  const dim3 grid(grid_for(rows, 8));
  const uint8_t* kp = static_cast<const uint8_t*>(k);
  const uint8_t* vp = static_cast<const uint8_t*>(v);
  uint8_t* kc = static_cast<uint8_t*>(k_cache);
  uint8_t* vc = static_cast<uint8_t*>(v_cache);
  if (chained)
    return launch_dependent(reshape_and_cache_kernel, grid, dim3(256), 0, stream, kp, vp, slot_mapping, num_tokens,
                            kc, vc, num_blocks, block_size, num_kv_heads, row_bytes, status) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
  reshape_and_cache_kernel<<<grid, 256, 0, stream>>>(kp, vp, slot_mapping, num_tokens, kc, vc, num_blocks,
                                                     block_size, num_kv_heads, row_bytes, status);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int32_t num_pairs,
                       int64_t block_bytes, cudaStream_t stream, bool chained) {
  for (int32_t base = 0; base < num_pairs; base += kCopyPairsPerLaunch) {
    const int32_t n = num_pairs - base < kCopyPairsPerLaunch ? num_pairs - base : kCopyPairsPerLaunch;
    CopyPairs pairs;
    for (int32_t i = 0; i < n; ++i) {
      pairs.src[i] = src[base + i];
      pairs.dst[i] = dst[base + i];
    }
    uint8_t* kc = static_cast<uint8_t*>(k_cache);
    uint8_t* vc = static_cast<uint8_t*>(v_cache);
    if (chained) {
      if (launch_dependent(copy_blocks_kernel, dim3(n, 2), dim3(256), 0, stream, kc, vc, pairs, block_bytes) !=
          cudaSuccess)
        return PA_ERR_CUDA;
      continue;
    }
    copy_blocks_kernel<<<dim3(n, 2), 256, 0, stream>>>(kc, vc, pairs, block_bytes);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

int launch_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v, const int32_t* src,
                       const int32_t* dst, int32_t num_pairs, int64_t block_bytes, int vec16, cudaStream_t stream) {
  const int pools = src_v ? 2 : 1;
  for (int32_t base = 0; base < num_pairs; base += kCopyPairsPerLaunch) {
    const int32_t n = num_pairs - base < kCopyPairsPerLaunch ? num_pairs - base : kCopyPairsPerLaunch;
    CopyPairs pairs;
    for (int32_t i = 0; i < n; ++i) {
      pairs.src[i] = src[base + i];
      pairs.dst[i] = dst[base + i];
    }
    swap_blocks_kernel<<<dim3(n, pools), 256, 0, stream>>>(
        static_cast<const uint8_t*>(src_k), static_cast<const uint8_t*>(src_v), static_cast<uint8_t*>(dst_k),
        static_cast<uint8_t*>(dst_v), pairs, block_bytes, vec16);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

int launch_reshape_and_cache_fp8(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                                 uint8_t* k_cache, uint8_t* v_cache, float* kv_scales, int32_t num_blocks,
                                 int32_t block_size, int32_t num_kv_heads, int32_t head_dim, pa_dtype dt,
                                 int kv_fmt, int* status, cudaStream_t stream) {
  const int64_t warps = num_tokens * num_kv_heads * 2;
  const int grid = grid_for(warps, 8);
#define PA_RC8_F(TI, VEC, E5)                                                                                    \
  reshape_and_cache_fp8_kernel<TI, VEC, E5><<<grid, 256, 0, stream>>>(                                           \
      static_cast<const TI*>(k), static_cast<const TI*>(v), slot_mapping, num_tokens, k_cache, v_cache, kv_scales, \
      num_blocks, block_size, num_kv_heads, status)
#define PA_RC8(TI, VEC)          \
  if (kv_fmt == PA_KV_E5M2)      \
    PA_RC8_F(TI, VEC, true);     \
  else                           \
    PA_RC8_F(TI, VEC, false)
  const bool d128 = head_dim == 128;
  if (dt == PA_BF16) {
    if (d128) PA_RC8(__nv_bfloat16, 4); else PA_RC8(__nv_bfloat16, 2);
  } else if (dt == PA_F16) {
    if (d128) PA_RC8(__half, 4); else PA_RC8(__half, 2);
  } else {
    if (d128) PA_RC8(float, 4); else PA_RC8(float, 2);
  }
#undef PA_RC8
#undef PA_RC8_F
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_copy_scales(float* kv_scales, const int32_t* src, const int32_t* dst, int32_t num_pairs,
                       int32_t num_kv_heads, cudaStream_t stream) {
  for (int32_t base = 0; base < num_pairs; base += kCopyPairsPerLaunch) {
    const int32_t n = num_pairs - base < kCopyPairsPerLaunch ? num_pairs - base : kCopyPairsPerLaunch;
    CopyPairsScales pairs;
    for (int32_t i = 0; i < n; ++i) {
      pairs.src[i] = src[base + i];
      pairs.dst[i] = dst[base + i];
    }
    copy_scales_kernel<<<n, 256, 0, stream>>>(kv_scales, pairs, 2 * num_kv_heads);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

}  // namespace pa
