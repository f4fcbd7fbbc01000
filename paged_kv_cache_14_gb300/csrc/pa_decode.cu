// Paged decode attention for sm_103a.
//
// One CTA handles one (split-KV partition, KV head [, query-row group],
// sequence). It walks the sequence's block table over the partition and, for
// every logical block, stages that block's K and V tiles for its KV head
// (each tile is block_size x head_dim contiguous elements of the pool) into
// shared memory with TMA. All query heads of the GQA group that share the KV
// head are packed as the rows of one 16-row MMA tile, so every KV block is
// read from HBM once per KV head ("03 - PagedAttention & the vLLM V1
// Architecture", section "The attention kernel side": look up the block
// table, fetch each block's K/V tiles, attend over the gathered tiles).
//
// Warp roles (160 threads): warp 4 is the producer (one lane issues the TMA
// copies, ring of kStages stages guarded by full/empty mbarriers); warps 0-3
// consume blocks round-robin, each keeping its own running max m, running
// sum l and unnormalised output o for the 16 rows (online softmax), with
// S = Q K^T and O += P V on warp-level tensor-core MMAs (m16n8k16, fp32
// accumulate). At the end the four warps are merged through shared memory.
// Decode is HBM-bound (about 8 flop per KV byte at GQA group 8), so the
// warp-level MMA has ample headroom and tcgen05 tiles (M >= 64) would only
// pad the 8 live rows.
//
// A partition writes the final output when it is the sequence's only one;
// otherwise it writes fp32 partials (m, l, o~) and a merge kernel combines
// them with log-sum-exp weights.
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

template <int D, int BS>
struct DecodeCfg {
  static constexpr int kHalves = D / 64;                  // 128-byte swizzle boxes across head_dim
  static constexpr int kTileBytes = BS * D * 2;           // one (block, KV head) tile of K or V
  static constexpr int kStageBytes = 2 * kTileBytes;      // K tile + V tile
  static constexpr int kStages = (65536 / kStageBytes) > 16 ? 16 : (65536 / kStageBytes);
  static constexpr int kConsumerWarps = 4;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int kRows = 16;
  static constexpr int kOStride = D + 4;  // fp32 merge-scratch row stride (bank spread)
  static constexpr int kMaxIds = kMaxPartition / BS;
  static constexpr size_t kStageRegion = (size_t)kStages * kStageBytes;
  static constexpr size_t kMergeBytes = (size_t)kConsumerWarps * kRows * kOStride * 4;
  static constexpr size_t kBarOff = kStageRegion;
  static constexpr size_t kMlOff = kBarOff + 2 * kStages * 8;
  static constexpr size_t kFlagOff = kMlOff + kConsumerWarps * kRows * 2 * 4;
  static constexpr size_t kIdsOff = kFlagOff + 16;
  static constexpr size_t kSmemBytes = kIdsOff + kMaxIds * 4 + 1024;  // + alignment slack
  static_assert(kStages % kConsumerWarps == 0, "a stage must always belong to the same consumer warp");
  static_assert(kMergeBytes <= kStageRegion, "merge scratch reuses the stage ring");
};

__device__ __forceinline__ uint32_t ld_u32(const void* p) { return *reinterpret_cast<const uint32_t*>(p); }

// Resolve the row of q / out and the key count of sequence `seq`.
// Returns false when this sequence is not a decode row of this launch.
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

template <typename T>
__device__ void write_zero_rows(const DecodeParams& p, int qrow, int h0, int nrows) {
  T* out = static_cast<T*>(p.out);
  for (int i = threadIdx.x; i < nrows * p.head_dim; i += blockDim.x) {
    const int r = i / p.head_dim, d = i - r * p.head_dim;
    out[((int64_t)qrow * p.num_q_heads + h0 + r) * p.head_dim + d] = T(0.0f);
  }
}

template <typename T, int D, int BS>
__global__ void __launch_bounds__(DecodeCfg<D, BS>::kThreads, 2)
    decode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                     const DecodeParams p) {
  using C = DecodeCfg<D, BS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int part = blockIdx.x;
  const int kvh = blockIdx.y / p.row_groups;
  const int rg = blockIdx.y - kvh * p.row_groups;
  const int seq = blockIdx.z;
  int qrow, len;
  if (!decode_row(p, seq, qrow, len)) return;
  const int h0 = kvh * p.group + rg * p.rows_per_cta;
  const int nrows = min(p.rows_per_cta, p.group - rg * p.rows_per_cta);
  if (len < 1 || len > p.len_cap || len > p.max_blocks_per_seq * BS) {
    if (part == 0) {
      if (threadIdx.x == 0) record_error(p.status, PA_ERR_SEQLEN);
      write_zero_rows<T>(p, qrow, h0, nrows);
    }
    return;
  }
  const int n_parts = (len + p.partition - 1) / p.partition;
  if (part >= n_parts) return;
  const int t_begin = part * p.partition;
  const int t_end = min(t_begin + p.partition, len);
  const int nblk = (t_end - t_begin + BS - 1) / BS;

  int32_t* ids = reinterpret_cast<int32_t*>(smem + C::kIdsOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + C::kStages;
  float* ml = reinterpret_cast<float*>(smem + C::kMlOff);
  int* abort_flag = reinterpret_cast<int*>(smem + C::kFlagOff);

  {
    const int32_t* bt = p.block_tables + (int64_t)seq * p.max_blocks_per_seq + t_begin / BS;
    for (int j = threadIdx.x; j < nblk; j += blockDim.x) {
      int id = bt[j];
      if (id < 0 || id >= p.num_blocks) {
        record_error(p.status, PA_ERR_BLOCK_OOB);
        id = -1;
      }
      ids[j] = id;
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    abort_flag[0] = 0;
    abort_flag[1] = 0;  // loads issued by the producer
    fence_barrier_init();
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t stage0 = smem_u32(smem);

  // Per-consumer state (rows r0 = lane/4 and r0 + 8 of the 16-row tile).
  const int r0 = lane >> 2;
  const int cq = (lane & 3) * 2;
  float o[D / 8][4];
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

  if (warp == C::kConsumerWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      int j = 0;
      for (; j < nblk; ++j) {
        const int s = j % C::kStages;
        if (j >= C::kStages && !mbar_wait(smem_u32(&empty[s]), ((j / C::kStages) & 1) ^ 1, p.status)) {
          atomicExch(&abort_flag[0], 1);
          break;
        }
        const int id = ids[j];
        const uint32_t fb = smem_u32(&full[s]);
        if (id >= 0) {
          mbar_arrive_expect_tx(fb, C::kStageBytes);
          const int32_t row = (id * p.num_kv_heads + kvh) * BS;
          const uint32_t kdst = stage0 + s * C::kStageBytes;
          const uint32_t vdst = kdst + C::kTileBytes;
#pragma unroll
          for (int hf = 0; hf < C::kHalves; ++hf) {
            tma_load_2d(kdst + hf * (BS * 128), &kmap, hf * 64, row, fb);
            tma_load_2d(vdst + hf * (BS * 128), &vmap, hf * 64, row, fb);
          }
        } else {
          mbar_arrive(fb);
        }
      }
      abort_flag[1] = j;
    }
  } else {
    // ---------------- consumers ----------------
    uint32_t qa[D / 16][4];
    {
      const T* qb = static_cast<const T*>(p.q) + ((int64_t)qrow * p.num_q_heads + h0) * D;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int c = kk * 16 + cq;
        qa[kk][0] = r0 < nrows ? ld_u32(qb + r0 * D + c) : 0u;
        qa[kk][1] = r0 + 8 < nrows ? ld_u32(qb + (r0 + 8) * D + c) : 0u;
        qa[kk][2] = r0 < nrows ? ld_u32(qb + r0 * D + c + 8) : 0u;
        qa[kk][3] = r0 + 8 < nrows ? ld_u32(qb + (r0 + 8) * D + c + 8) : 0u;
      }
    }
    const float sl2 = p.scale_log2;
    const int mi = lane >> 3, rr = lane & 7;
    for (int j = warp; j < nblk; j += C::kConsumerWarps) {
      const int s = j % C::kStages;
      if (!mbar_wait(smem_u32(&full[s]), (j / C::kStages) & 1, p.status)) {
        atomicExch(&abort_flag[0], 1);
        break;
      }
      if (ids[j] >= 0) {
        const uint32_t kb = stage0 + s * C::kStageBytes;
        const uint32_t vb = kb + C::kTileBytes;
#pragma unroll
        for (int sub = 0; sub < BS / 16; ++sub) {
          const int tok0 = t_begin + j * BS + sub * 16;
          if (tok0 >= t_end) break;
          float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          {
            const int tok = sub * 16 + (mi >> 1) * 8 + rr;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const int cg = kk * 2 + (mi & 1);
              const uint32_t addr = kb + (cg >> 3) * (BS * 128) + tok * 128 + (((cg & 7) ^ (tok & 7)) << 4);
              uint32_t b0, b1, b2, b3;
              ldsm_x4(addr, b0, b1, b2, b3);
              MmaOp<T>::run(sc[0], qa[kk], b0, b1);
              MmaOp<T>::run(sc[1], qa[kk], b2, b3);
            }
          }
          // Scale into log2 units and mask keys past the partition end.
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int tok = tok0 + nt * 8 + cq + (e & 1);
              sc[nt][e] = tok < t_end ? sc[nt][e] * sl2 : -CUDART_INF_F;
            }
          // Online softmax (row max over the quad of lanes that share a row).
          float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
          float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
          const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
          const bool dead0 = mn0 == -CUDART_INF_F, dead1 = mn1 == -CUDART_INF_F;
          const float a0 = dead0 ? 1.f : exp2f(m0 - mn0);
          const float a1 = dead1 ? 1.f : exp2f(m1 - mn1);
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            sc[nt][0] = dead0 ? 0.f : exp2f(sc[nt][0] - mn0);
            sc[nt][1] = dead0 ? 0.f : exp2f(sc[nt][1] - mn0);
            sc[nt][2] = dead1 ? 0.f : exp2f(sc[nt][2] - mn1);
            sc[nt][3] = dead1 ? 0.f : exp2f(sc[nt][3] - mn1);
          }
          l0 = l0 * a0 + (sc[0][0] + sc[0][1]) + (sc[1][0] + sc[1][1]);
          l1 = l1 * a1 + (sc[0][2] + sc[0][3]) + (sc[1][2] + sc[1][3]);
          m0 = mn0;
          m1 = mn1;
#pragma unroll
          for (int nt = 0; nt < D / 8; ++nt) {
            o[nt][0] *= a0;
            o[nt][1] *= a0;
            o[nt][2] *= a1;
            o[nt][3] *= a1;
          }
          // P as the A operand (the S accumulator layout is the A layout).
          const uint32_t pa[4] = {MmaOp<T>::pack(sc[0][0], sc[0][1]), MmaOp<T>::pack(sc[0][2], sc[0][3]),
                                  MmaOp<T>::pack(sc[1][0], sc[1][1]), MmaOp<T>::pack(sc[1][2], sc[1][3])};
          // Keys past the end carry p = 0, but their V slots may hold any
          // bits (NaN included): zero those V elements so 0 * V stays 0.
          const bool tail = tok0 + 16 > t_end;
          const int tlo = tok0 + cq;  // tokens held by the low / high halves of b0 (b1: +8)
          const uint32_t keep0 = (tlo < t_end ? 0x0000ffffu : 0u) | (tlo + 1 < t_end ? 0xffff0000u : 0u);
          const uint32_t keep1 = (tlo + 8 < t_end ? 0x0000ffffu : 0u) | (tlo + 9 < t_end ? 0xffff0000u : 0u);
          {
            const int tok = sub * 16 + (mi & 1) * 8 + rr;
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
              const int cg = np * 2 + (mi >> 1);
              const uint32_t addr = vb + (cg >> 3) * (BS * 128) + tok * 128 + (((cg & 7) ^ (tok & 7)) << 4);
              uint32_t b0, b1, b2, b3;
              ldsm_x4_t(addr, b0, b1, b2, b3);
              if (tail) {
                b0 &= keep0;
                b1 &= keep1;
                b2 &= keep0;
                b3 &= keep1;
              }
              MmaOp<T>::run(o[2 * np], pa, b0, b1);
              MmaOp<T>::run(o[2 * np + 1], pa, b2, b3);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  }
  __syncthreads();

  if (abort_flag[0]) {
    // A bounded wait ran out (recorded in the status word). Let every copy
    // still in flight land before the CTA's shared memory is released.
    if (threadIdx.x == 0) {
      const int issued = abort_flag[1];
      for (int s = 0; s < C::kStages && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / C::kStages) * C::kStages;
        mbar_wait(smem_u32(&full[s]), (last / C::kStages) & 1, nullptr);
      }
    }
    return;
  }

  // ---------------- merge the four consumer warps ----------------
  if (warp < C::kConsumerWarps && (lane & 3) == 0) {
    ml[(warp * 16 + r0) * 2 + 0] = m0;
    ml[(warp * 16 + r0) * 2 + 1] = l0;
    ml[(warp * 16 + r0 + 8) * 2 + 0] = m1;
    ml[(warp * 16 + r0 + 8) * 2 + 1] = l1;
  }
  __syncthreads();
  float* ob = reinterpret_cast<float*>(smem);
  if (warp < C::kConsumerWarps) {
    float M0 = -CUDART_INF_F, M1 = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < C::kConsumerWarps; ++w) {
      M0 = fmaxf(M0, ml[(w * 16 + r0) * 2]);
      M1 = fmaxf(M1, ml[(w * 16 + r0 + 8) * 2]);
    }
    const float f0 = m0 == -CUDART_INF_F ? 0.f : exp2f(m0 - M0);
    const float f1 = m1 == -CUDART_INF_F ? 0.f : exp2f(m1 - M1);
    float* wb = ob + warp * 16 * C::kOStride;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int col = nt * 8 + cq;
      *reinterpret_cast<float2*>(&wb[r0 * C::kOStride + col]) = make_float2(o[nt][0] * f0, o[nt][1] * f0);
      *reinterpret_cast<float2*>(&wb[(r0 + 8) * C::kOStride + col]) = make_float2(o[nt][2] * f1, o[nt][3] * f1);
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nrows * (D / 4); idx += blockDim.x) {
    const int row = idx / (D / 4);
    const int c4 = (idx - row * (D / 4)) * 4;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < C::kConsumerWarps; ++w) M = fmaxf(M, ml[(w * 16 + row) * 2]);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < C::kConsumerWarps; ++w) {
      const float mw = ml[(w * 16 + row) * 2];
      L += mw == -CUDART_INF_F ? 0.f : ml[(w * 16 + row) * 2 + 1] * exp2f(mw - M);
      const float4 v = *reinterpret_cast<const float4*>(&ob[(w * 16 + row) * C::kOStride + c4]);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    if (n_parts == 1) {
      const float inv = 1.f / L;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
      store4(static_cast<T*>(p.out) + ((int64_t)qrow * p.num_q_heads + h0 + row) * D + c4, acc);
    } else {
      const int64_t base = ((int64_t)seq * p.num_q_heads + h0 + row) * p.max_parts + part;
      store4(p.part_o + base * D + c4, acc);
      if (c4 == 0) {
        p.part_ml[base * 2 + 0] = M;
        p.part_ml[base * 2 + 1] = L;
      }
    }
  }
}

// fp32 I/O: CUDA-core path (exact fp32 FMAs, no TF32). Four warps take the
// partition's tokens round-robin; each lane holds head_dim/32 dimensions and
// the dot products are reduced across the warp.
template <int VEC>
__global__ void __launch_bounds__(128) decode_simt_kernel(const DecodeParams p) {
  constexpr int D = VEC * 32;
  constexpr int ROWS = 8;
  constexpr int NW = 4;
  __shared__ int32_t ids[kMaxPartition / 16];
  __shared__ float ml[NW][ROWS][2];
  __shared__ float ob[NW][ROWS][D];

  const int part = blockIdx.x;
  const int kvh = blockIdx.y / p.row_groups;
  const int rg = blockIdx.y - kvh * p.row_groups;
  const int seq = blockIdx.z;
  const int BS = p.block_size;
  int qrow, len;
  if (!decode_row(p, seq, qrow, len)) return;
  const int h0 = kvh * p.group + rg * p.rows_per_cta;
  const int nrows = min(p.rows_per_cta, p.group - rg * p.rows_per_cta);
  if (len < 1 || len > p.len_cap || len > p.max_blocks_per_seq * BS) {
    if (part == 0) {
      if (threadIdx.x == 0) record_error(p.status, PA_ERR_SEQLEN);
      write_zero_rows<float>(p, qrow, h0, nrows);
    }
    return;
  }
  const int n_parts = (len + p.partition - 1) / p.partition;
  if (part >= n_parts) return;
  const int t_begin = part * p.partition;
  const int t_end = min(t_begin + p.partition, len);
  const int nblk = (t_end - t_begin + BS - 1) / BS;
  {
    const int32_t* bt = p.block_tables + (int64_t)seq * p.max_blocks_per_seq + t_begin / BS;
    for (int j = threadIdx.x; j < nblk; j += blockDim.x) {
      int id = bt[j];
      if (id < 0 || id >= p.num_blocks) {
        record_error(p.status, PA_ERR_BLOCK_OOB);
        id = -1;
      }
      ids[j] = id;
    }
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* qb = static_cast<const float*>(p.q) + ((int64_t)qrow * p.num_q_heads + h0) * D;
  float q[ROWS][VEC], o[ROWS][VEC], m[ROWS], l[ROWS];
#pragma unroll
  for (int g = 0; g < ROWS; ++g) {
    m[g] = -CUDART_INF_F;
    l[g] = 0.f;
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      q[g][v] = g < nrows ? qb[g * D + lane + 32 * v] : 0.f;
      o[g][v] = 0.f;
    }
  }
  const float* kc = static_cast<const float*>(p.k_cache);
  const float* vc = static_cast<const float*>(p.v_cache);
  for (int t = t_begin + warp; t < t_end; t += NW) {
    const int id = ids[(t - t_begin) / BS];
    if (id < 0) continue;
    const int64_t row = ((int64_t)id * p.num_kv_heads + kvh) * BS + (t % BS);
    float kv[VEC], vv[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      kv[v] = kc[row * D + lane + 32 * v];
      vv[v] = vc[row * D + lane + 32 * v];
    }
#pragma unroll
    for (int g = 0; g < ROWS; ++g) {
      if (g >= nrows) break;
      float d = 0.f;
#pragma unroll
      for (int v = 0; v < VEC; ++v) d = fmaf(q[g][v], kv[v], d);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
      const float s = d * p.scale_log2;
      const float mn = fmaxf(m[g], s);
      const float a = exp2f(m[g] - mn);
      const float e = exp2f(s - mn);
      l[g] = l[g] * a + e;
#pragma unroll
      for (int v = 0; v < VEC; ++v) o[g][v] = fmaf(e, vv[v], o[g][v] * a);
      m[g] = mn;
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int g = 0; g < ROWS; ++g) {
      ml[warp][g][0] = m[g];
      ml[warp][g][1] = l[g];
    }
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < ROWS; ++g) {
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, ml[w][g][0]);
    const float f = m[g] == -CUDART_INF_F ? 0.f : exp2f(m[g] - M);
#pragma unroll
    for (int v = 0; v < VEC; ++v) ob[warp][g][lane + 32 * v] = o[g][v] * f;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nrows * D; idx += blockDim.x) {
    const int g = idx / D, d = idx - g * D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, ml[w][g][0]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = ml[w][g][0];
      L += mw == -CUDART_INF_F ? 0.f : ml[w][g][1] * exp2f(mw - M);
      acc += ob[w][g][d];
    }
    if (n_parts == 1) {
      static_cast<float*>(p.out)[((int64_t)qrow * p.num_q_heads + h0 + g) * D + d] = acc / L;
    } else {
      const int64_t base = ((int64_t)seq * p.num_q_heads + h0 + g) * p.max_parts + part;
      p.part_o[base * D + d] = acc;
      if (d == 0) {
        p.part_ml[base * 2 + 0] = M;
        p.part_ml[base * 2 + 1] = L;
      }
    }
  }
}

// Split-KV merge: out = sum_p 2^(m_p - M) o~_p / sum_p 2^(m_p - M) l_p with
// M = max_p m_p (scores are kept in log2 units). One CTA per (q head, seq).
template <typename T>
__global__ void __launch_bounds__(128) splitkv_merge_kernel(const DecodeParams p) {
  const int h = blockIdx.x;
  const int seq = blockIdx.y;
  int qrow, len;
  if (!decode_row(p, seq, qrow, len)) return;
  if (len < 1 || len > p.len_cap || len > p.max_blocks_per_seq * p.block_size) return;
  const int n = (len + p.partition - 1) / p.partition;
  if (n <= 1) return;
  const int64_t base = ((int64_t)seq * p.num_q_heads + h) * p.max_parts;
  extern __shared__ float wts[];  // [max_parts]
  __shared__ float red[2];
  if (threadIdx.x < 32) {
    float M = -CUDART_INF_F;
    for (int i = threadIdx.x; i < n; i += 32) M = fmaxf(M, p.part_ml[(base + i) * 2]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    for (int i = threadIdx.x; i < n; i += 32) {
      const float w = exp2f(p.part_ml[(base + i) * 2] - M);
      wts[i] = w;
      L += w * p.part_ml[(base + i) * 2 + 1];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (threadIdx.x == 0) red[0] = 1.f / L;
  }
  __syncthreads();
  const float invL = red[0];
  const int D = p.head_dim;
  T* out = static_cast<T*>(p.out) + ((int64_t)qrow * p.num_q_heads + h) * D;
  for (int d4 = threadIdx.x * 4; d4 < D; d4 += blockDim.x * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < n; ++i) {
      const float w = wts[i];
      const float4 v = *reinterpret_cast<const float4*>(p.part_o + (base + i) * D + d4);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    acc.x *= invL;
    acc.y *= invL;
    acc.z *= invL;
    acc.w *= invL;
    store4(out + d4, acc);
  }
}

template <typename T, int D, int BS>
static int launch_tc(const DecodeParams& p, cudaStream_t stream) {
  using C = DecodeCfg<D, BS>;
  const pa_dtype dt = sizeof(T) == 2 && std::is_same<T, __half>::value ? PA_F16 : PA_BF16;
  CUtensorMap kmap, vmap;
  const int64_t rows = (int64_t)p.num_blocks * p.num_kv_heads * BS;
  int rc = make_kv_tensor_map(&kmap, p.k_cache, rows, D, dt, BS);
  if (rc != PA_OK) return rc;
  rc = make_kv_tensor_map(&vmap, p.v_cache, rows, D, dt, BS);
  if (rc != PA_OK) return rc;
  auto kern = decode_tc_kernel<T, D, BS>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes) !=
        cudaSuccess)
      return PA_ERR_CUDA;
    attr_set[dev] = true;
  }
  dim3 grid(p.max_parts, p.num_kv_heads * p.row_groups, p.num_seqs);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(kmap, vmap, p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <int VEC>
static int launch_simt(const DecodeParams& p, cudaStream_t stream) {
  dim3 grid(p.max_parts, p.num_kv_heads * p.row_groups, p.num_seqs);
  decode_simt_kernel<VEC><<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_decode(const DecodeParams& p0, pa_dtype dt, cudaStream_t stream) {
  DecodeParams p = p0;
  const int rows_max = dt == PA_F32 ? 8 : 16;
  p.rows_per_cta = p.group < rows_max ? p.group : rows_max;
  p.row_groups = (p.group + p.rows_per_cta - 1) / p.rows_per_cta;
  if ((int64_t)p.num_kv_heads * p.row_groups > 65535) return PA_ERR_UNSUPPORTED;
  int rc = PA_ERR_UNSUPPORTED;
  if (dt == PA_F32) {
    switch (p.head_dim) {
      case 32: rc = launch_simt<1>(p, stream); break;
      case 64: rc = launch_simt<2>(p, stream); break;
      case 96: rc = launch_simt<3>(p, stream); break;
      case 128: rc = launch_simt<4>(p, stream); break;
      case 160: rc = launch_simt<5>(p, stream); break;
      case 192: rc = launch_simt<6>(p, stream); break;
      case 224: rc = launch_simt<7>(p, stream); break;
      case 256: rc = launch_simt<8>(p, stream); break;
      default: return PA_ERR_UNSUPPORTED;
    }
  } else {
    const bool bf = dt == PA_BF16;
    const int key = (p.head_dim == 64 ? 0 : p.head_dim == 128 ? 1 : 9) * 2 + (p.block_size == 16 ? 0 : 1);
    switch (key) {
      case 0: rc = bf ? launch_tc<__nv_bfloat16, 64, 16>(p, stream) : launch_tc<__half, 64, 16>(p, stream); break;
      case 1: rc = bf ? launch_tc<__nv_bfloat16, 64, 32>(p, stream) : launch_tc<__half, 64, 32>(p, stream); break;
      case 2: rc = bf ? launch_tc<__nv_bfloat16, 128, 16>(p, stream) : launch_tc<__half, 128, 16>(p, stream); break;
      case 3: rc = bf ? launch_tc<__nv_bfloat16, 128, 32>(p, stream) : launch_tc<__half, 128, 32>(p, stream); break;
      default: return PA_ERR_UNSUPPORTED;
    }
  }
  if (rc != PA_OK || p.max_parts <= 1) return rc;
  const size_t wbytes = (size_t)p.max_parts * sizeof(float);
  dim3 grid(p.num_q_heads, p.num_seqs);
  if (dt == PA_F32)
    splitkv_merge_kernel<float><<<grid, 128, wbytes, stream>>>(p);
  else if (dt == PA_BF16)
    splitkv_merge_kernel<__nv_bfloat16><<<grid, 128, wbytes, stream>>>(p);
  else
    splitkv_merge_kernel<__half><<<grid, 128, wbytes, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
