// Chunked-prefill attention over a paged context on tcgen05 tensor cores
// (sm_103a). Chunked prefill splits a prompt into chunks that run alongside
// decode rows ("Tech Radar: vLLM v1 Production Engine Architecture ...",
// section 3 "Dynamic Chunked Prefill"); prefill is the tensor-core-bound
// phase (same page, "The Prefill Phase (Compute-Bound)").
//
// Tiles. A chunk of q_len query rows of a sequence with ctx prior tokens is
// cut into work items of 256 packed (query position, GQA head) rows, two
// Q tiles of 128: all G query heads that share one KV head are consecutive
// rows, so every K/V tile is read once per KV head and item and feeds two
// full 128-row MMAs. Row r of the chunk sits at position ctx + r and attends
// to keys 0 .. ctx + r.
//
// One persistent CTA per SM (320 threads) loops over work items (chunk
// rows, KV head) listed by a plan kernel, longest first:
//   warp 0  producer: TMA of the two Q tiles (3-D tensor map over
//           [tokens][heads][head_dim], 128-byte swizzle), then for every
//           128-token KV tile the eight 16-token sub-tiles of K and of V
//           through the block table, into separate K and V rings;
//   warp 1  owns the tensor memory (all 512 columns: per Q tile an S tile
//           of 128x128 fp32 and O = 128x128 fp32) and one lane issues the
//           MMAs: S = Q K^T (K-major operands from shared memory), then
//           O += P V with P read from tensor memory and V an MN-major
//           shared-memory operand;
//   warps 2-5, 6-9  softmax of Q tile 0, 1: thread i of a warpgroup owns
//           row i (tensor-memory lane i): it loads its S row, applies the
//           causal mask, keeps the running max and sum in registers, writes P
//           (16-bit) back over its S row, rescales its O row in tensor memory
//           when the max moved, and at the end normalises O and stores it.
// While one warpgroup computes its softmax the tensor pipe runs the other
// Q tile's MMAs. Per SM and KV tile the MMAs read 192 KB of shared memory
// and the copies write 64 KB, against 2048 tensor-pipe cycles at
// 8192 flop per cycle.
// Every mbarrier wait is time-bounded: on a timeout the kernel records
// PA_ERR_TIMEOUT, lets outstanding copies and MMAs finish (bounded) and
// returns; no wait can spin forever.
#include <math_constants.h>

#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_plan.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

namespace pf {
constexpr int kM = 128;          // rows per Q tile (tensor-memory lanes)
constexpr int kQT = 2;           // Q tiles per work item, one softmax warpgroup each
constexpr int kRows = kM * kQT;  // packed rows per work item
constexpr int kD = 128;          // largest head_dim: the shared-memory tiles are laid out for it
constexpr int kN = 128;          // keys per KV tile
constexpr int kSubTiles = kN / 16;  // 16-token sub-tiles per KV tile
constexpr int kThreads = 64 + kQT * 128;  // producer, MMA, one softmax warpgroup per Q tile
constexpr int kSoftmaxWarp0 = 2;           // first softmax warp
constexpr int kQHalf = kM * 128;          // one 64-column half of a Q tile: 128 rows x 128 B
constexpr int kQBytes = 2 * kQHalf;       // one Q tile: 32 KB
constexpr int kKVHalf = kN * 128;         // kN rows x 128 B
constexpr int kKBytes = 2 * kKVHalf;      // one K (or V) tile: 32 KB
#ifndef PA_PREFILL_NV
#define PA_PREFILL_NV 2
#endif
constexpr int NK = 2;               // K stages
constexpr int NV = PA_PREFILL_NV;   // V stages (2 or 3)
constexpr int kVLead = NV - NK;     // V(t + kVLead) is issued right after K(t)
static_assert(kVLead == 0 || kVLead == 1, "two K stages, two or three V stages");
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQT * kQBytes;
constexpr int kOffV = kOffK + NK * kKBytes;
constexpr int kOffBar = kOffV + NV * kKBytes;
// bars: q_full, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], then per Q
// tile s_full, p_full, o_done
constexpr int kBarQ = 0;
constexpr int kBarKFull = 1;
constexpr int kBarKEmpty = kBarKFull + NK;
constexpr int kBarVFull = kBarKEmpty + NK;
constexpr int kBarVEmpty = kBarVFull + NV;
constexpr int kBarSFull = kBarVEmpty + NV;
constexpr int kBarPFull = kBarSFull + kQT;
constexpr int kBarODone = kBarPFull + kQT;
// e4m3 cache only: codes of K / V landed in a stage (TMA), Q tiles moved
// into fp16 (converter warps).
constexpr int kBarKCode = kBarODone + kQT;
constexpr int kBarVCode = kBarKCode + NK;
constexpr int kBarQConv = kBarVCode + NV;
constexpr int kNumBars = kBarQConv + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, item, abort
constexpr int kOffQExp = kOffMisc + 64;           // e4m3: per-row exponent of the fp16 Q rows [kQT][kM]
constexpr int kSmem = kOffQExp + kQT * kM * 4;
// 8-bit cache: converter warps widen the codes of each K / V stage (TMA puts
// them in the upper half of the stage) into the 16-bit stage layout, and
// move a bf16 Q tile into fp16. Two warps: one left the widening on the
// critical path (1.63 ms for the mixed 70B batch over e4m3 pools against
// 1.52 ms with two; four gave 1.60 ms).
constexpr int kConvWarp0 = kSoftmaxWarp0 + 4 * kQT;
#ifndef PA_PREFILL_CONV_WARPS
#define PA_PREFILL_CONV_WARPS 2
#endif
constexpr int kConvWarps = PA_PREFILL_CONV_WARPS;
template <bool KV8>
__host__ __device__ constexpr int threads() { return kThreads + (KV8 ? 32 * kConvWarps : 0); }
static_assert(kSmem <= 227 * 1024, "shared memory of one CTA");
// Tensor memory, per Q tile t: S (kN fp32 columns; P, 16-bit pairs, over its
// first kN/2) at t * 256, O (128 fp32 columns) at t * 256 + 128.
constexpr int kTmemCols = 512;
constexpr int kCtasPerSm = 1;
__host__ __device__ constexpr int col_s(int t) { return t * 256; }
__host__ __device__ constexpr int col_o(int t) { return t * 256 + kN; }
static_assert(kRows == kPrefillRowsPerItem, "work list granularity shared with the shared-prefix preparation");
}  // namespace pf

// Plan: list (sequence, 256-row item) pairs of every chunk with q_len > 1,
// ordered by decreasing number of KV tiles (longest items first), and reset
// the item counter. Run by the 1024 threads of one CTA. Returns (to every
// thread) the number of (item, KV tile) units the chunk kernel will run.
__device__ __forceinline__ int64_t prefill_plan_body(const PrefillParams& p) {
  constexpr int kBins = 2048;
  __shared__ int hist[kBins];
  __shared__ int total;
  __shared__ int scratch[33];
  const int pp = pf::kQT * p.tile_pos;  // query positions per work item
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) hist[i] = 0;
  if (threadIdx.x == 0) total = 0;
  __syncthreads();
  auto tiles_of = [&](int seq, int mt) -> int {
    const int q0 = p.cu_q_lens[seq], ql = p.cu_q_lens[seq + 1] - q0;
    const int ctx = p.ctx_lens[seq];
    const int pos_hi = min((mt + 1) * pp, ql);
    const int keys = ctx + pos_hi;
    const int t = (keys + pf::kN - 1) / pf::kN;
    return min(t, kBins - 1);
  };
  int my_tiles = 0;
  for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x) {
    const int ql = p.cu_q_lens[s + 1] - p.cu_q_lens[s];
    if (ql <= 1) continue;
    const int kv = p.ctx_lens[s] + ql;
    if (p.ctx_lens[s] < 0 || kv > p.max_kv_len || kv > p.max_blocks_per_seq * p.block_size || ql > p.max_q_len) {
      record_error(p.status, PA_ERR_SEQLEN);
      continue;
    }
    const int nm = (ql + pp - 1) / pp;
    for (int mt = 0; mt < nm; ++mt) {
      const int t = tiles_of(s, mt);
      my_tiles += t;
      atomicAdd(&hist[t], 1);
    }
  }
  int all_tiles;
  block_exclusive_scan_1024(my_tiles, scratch, &all_tiles);
  {
    // Exclusive scan from the longest bin down: thread t owns bins
    // kBins-1-2t and kBins-2-2t.
    const int b0 = kBins - 1 - 2 * threadIdx.x, b1 = b0 - 1;
    const int c0 = hist[b0], c1 = hist[b1];
    int tot;
    const int off = block_exclusive_scan_1024(c0 + c1, scratch, &tot);
    hist[b0] = off;
    hist[b1] = off + c0;
    if (threadIdx.x == 0) total = tot;
    __syncthreads();
  }
  for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x) {
    const int ql = p.cu_q_lens[s + 1] - p.cu_q_lens[s];
    if (ql <= 1) continue;
    const int kv = p.ctx_lens[s] + ql;
    if (p.ctx_lens[s] < 0 || kv > p.max_kv_len || kv > p.max_blocks_per_seq * p.block_size || ql > p.max_q_len)
      continue;
    const int nm = (ql + pp - 1) / pp;
    for (int mt = 0; mt < nm; ++mt) {
      const int slot = atomicAdd(&hist[tiles_of(s, mt)], 1);
      p.pairs[slot] = pack_pair(s, mt);
    }
  }
  if (threadIdx.x == 0) {
    p.work[0] = 0;
    p.work[1] = total * p.num_kv_heads;
  }
  return (int64_t)all_tiles * p.num_kv_heads;
}

// Plan of a batch of chunks only: every CTA of the chunk kernel runs items.
__global__ void __launch_bounds__(1024) prefill_plan_kernel(const PrefillParams p) {
  pdl_trigger();  // the chunk kernel may start its set-up now; it waits for this plan
  prefill_plan_body(p);
  if (threadIdx.x == 0) p.work[2] = p.ctas;
}

// Plan of a mixed batch (chunks and decode rows): the chunk list, the decode
// rows' work list (the decode kernel runs beside the chunk kernel and reads
// it without waiting: every chunk CTA lets the decode kernel start only
// after waiting for this plan), and the split of the SMs. The chunk kernel
// is bound by its tensor work, the decode rows by their KV reads, so the
// chunk kernel gets a share of the SMs in proportion to its estimated time
// on one SM: (item, KV tile) units at the measured per-SM rate against the
// decode rows' KV bytes at the measured per-SM streaming rate, expressed as
// decode_bytes_per_tile (KV bytes one SM streams in the time it runs one
// unit). Its surplus CTAs exit at once and the decode kernel takes their
// SMs; decode CTAs also take the SMs of chunk CTAs that run out of items.
template <typename T>
__global__ void __launch_bounds__(1024) mixed_plan_kernel(const PrefillParams p, const DecodeParams dp) {
  pdl_trigger();
  __shared__ int scratch2[33];
  const int64_t chunk_units = prefill_plan_body(p);
  __syncthreads();
  decode_plan_body<T>(dp);
  int64_t my_tokens = 0;
  for (int s = threadIdx.x; s < dp.num_seqs; s += blockDim.x) {
    int qrow, len;
    if (decode_row(dp, s, qrow, len) && len_ok(dp, len)) my_tokens += len;
  }
  // Tokens of one thread stay below 2^31 (at most num_seqs / 1024 rows of
  // at most 2^31 / 64 tokens each): the block sum is taken in units of 64.
  int total64;
  block_exclusive_scan_1024((int)((my_tokens + 63) >> 6), scratch2, &total64);
  if (threadIdx.x == 0) {
    const double decode_units = (double)total64 * 64.0 * p.decode_token_bytes / p.decode_bytes_per_tile;
    int n = p.ctas;
    if (chunk_units > 0 && decode_units > 0.0) {
      const double share = (double)chunk_units / ((double)chunk_units + decode_units);
      n = (int)lrint(share * p.num_sms);
      n = max(1, min(n, p.ctas));
    }
    p.work[2] = n;
  }
}

// PREFIX = false: chunked prefill (causal rows, normalised output).
// PREFIX = true: prefix pass of shared-prefix decode (rows = group members x
// GQA heads, each row masked to its own verified prefix, fp32 partial
// (m, l, o~) written to slot 0 of the member's partials).
//
// Pipeline of one item (KV tile g = tile_base + j, Q tiles 0 and 1):
//   producer:  K(g) into K stage g % NK once S1(g - NK) freed it, then V
//              into its stage once PV1 of the tile NV back freed it (the
//              stages free in the order K(g), V(g), K(g + 1), ...);
//   MMA:       S0(g), S1(g), then per tile PV0(g), S0(g + 1), PV1(g),
//              S1(g + 1). The tensor pipe executes one thread's MMAs in issue
//              order, so S_t(g + 1) cannot overwrite P_t(g) before PV_t(g)
//              has read it, and the commit that reports S_t(g + 1) also
//              covers PV_t(g): a softmax warpgroup that sees S_t ready may
//              rescale its O at once. The issue order also keeps the two Q
//              tiles half a step apart, so one tile's softmax overlaps the
//              other tile's MMAs;
//   softmax t: reads S_t(g), writes P_t(g) (16-bit) over the first kN/2
//              columns of S_t, signals p_full[t].
// Every barrier completes once per KV tile (s_full, p_full, stages) or once
// per item (q_full, o_done), those of Q tile 1 only on items whose second
// tile has rows, and is waited on in phase order.
//
// KV8 (8-bit cache, kv_scales given; e4m3 codes, or e5m2 with E5): the
// producer loads each 16-token sub-tile's codes into the upper half of its
// 16-bit stage; the converter warps widen them (exactly) to fp16 in the
// stage's swizzled layout and
// complete k_full / v_full. The MMAs run in fp16: a bf16 Q tile is moved into
// fp16 in place once per item, each row by its own power of two. The softmax
// multiplies a score by the K scale of its key's block (and the Q row's power
// of two) before the max, and weights P by the V scale of the key's block
// times 2^kap, kap the largest exponent keeping every weight of the item
// seen so far below 2^7 (P stays below 2^15 in fp16); O is rescaled exactly
// when kap drops and divided by 2^kap at the end. The row sum takes p alone.
// D = head_dim, 128 or 64 (16-bit caches): a tile is D / 64 swizzled
// 64-column halves of 128-byte rows (the layout is sized for 128).
template <typename T, int BS, bool PREFIX, bool KV8, bool E5 = false, int D = 128>
__global__ void __launch_bounds__(pf::threads<KV8>(), 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  using namespace pf;
  static_assert(D == 64 || D == kD, "head_dim 64 or 128");
  static_assert(!KV8 || D == 128, "8-bit caches at head_dim 128");
  constexpr int kH = D / 64;  // 64-column halves per row
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value && !KV8;  // the MMA's 16-bit type
  using MT = typename std::conditional<KV8, __half, T>::type;             // P's 16-bit type
  constexpr uint32_t kIdescS = idesc_f16(kM, kN, kBf16, false);  // S = Q K^T
  constexpr uint32_t kIdescO = idesc_f16(kM, D, kBf16, true);    // O += P V (V MN-major)
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  const uint32_t b_q = smem_u32(&bars[kBarQ]);
  const uint32_t b_kfull0 = smem_u32(&bars[kBarKFull]);    // + 8 * stage
  const uint32_t b_kempty0 = smem_u32(&bars[kBarKEmpty]);  // + 8 * stage
  const uint32_t b_vfull0 = smem_u32(&bars[kBarVFull]);    // + 8 * stage
  const uint32_t b_vempty0 = smem_u32(&bars[kBarVEmpty]);  // + 8 * stage
  const uint32_t b_sfull0 = smem_u32(&bars[kBarSFull]);    // + 8 * Q tile
  const uint32_t b_pfull0 = smem_u32(&bars[kBarPFull]);    // + 8 * Q tile
  const uint32_t b_odone0 = smem_u32(&bars[kBarODone]);    // + 8 * Q tile
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&misc[2]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);

  if (threadIdx.x == 0) {
    if ((sbase & 1023u) != 0) record_error(p.status, PA_ERR_ALIGN);
    mbar_init(b_q, 1);
    // A K / V stage is complete once its copies landed or, with an e4m3
    // cache, once both converter warps widened it.
    for (int i = 0; i < NK; ++i) {
      mbar_init(b_kfull0 + 8 * i, KV8 ? kConvWarps : 1);
      mbar_init(b_kempty0 + 8 * i, 1);
      mbar_init(smem_u32(&bars[kBarKCode + i]), 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(b_vfull0 + 8 * i, KV8 ? kConvWarps : 1);
      mbar_init(b_vempty0 + 8 * i, 1);
      mbar_init(smem_u32(&bars[kBarVCode + i]), 1);
    }
    mbar_init(smem_u32(&bars[kBarQConv]), kConvWarps);
    for (int i = 0; i < kQT; ++i) {
      mbar_init(b_sfull0 + 8 * i, 1);
      mbar_init(b_pfull0 + 8 * i, 4);  // one arrival per softmax warp
      mbar_init(b_odone0 + 8 * i, 1);
    }
    abort_flag[0] = (sbase & 1023u) != 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&misc[0]), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // the work list of the plan / preparation kernel
  pdl_trigger();
  const uint32_t tmem = misc[0];
  if constexpr (!PREFIX) {
    // CTAs beyond the plan's share of the SMs leave them to the decode rows
    // of a mixed batch at once.
    if ((int)blockIdx.x >= p.work[2]) {
      if (warp == 1) tmem_dealloc(tmem, kTmemCols);
      return;
    }
  }
  const int G = p.group;
  const int pp = p.tile_pos;  // query positions (or group members) per Q tile: pp * G <= 128 rows
  const int total = p.work[1];

  int tile_base = 0;  // KV tiles processed by this CTA before the current item
  // The barriers of Q tile 1 (s_full, p_full, o_done) only complete on items
  // whose second tile has rows: their phases count those items and tiles.
  int tile_base1 = 0, items1 = 0;
  for (int it = 0;; ++it) {
    if (threadIdx.x == 0) misc[1] = abort_flag[0] ? 0x7fffffff : atomicAdd(&p.work[0], 1);
    __syncthreads();
    const int item = (int)misc[1];
    if (item >= total) break;
    const int pi = item / p.num_kv_heads;
    const int pr = p.pairs[pi];
    const int kvh = item - pi * p.num_kv_heads;
    const int mt = pair_lo(pr);
    // Item geometry (kQT * pp positions from pos_lo). Chunk: rows are query
    // positions of sequence `seq`; prefix pass: rows are members of group
    // `grp`, keys are the group's shared prefix read through the reference
    // member's table.
    int seq, q_z, q0 = 0, ql = 0, ctx = 0, kv_len, keys, grp = 0, s0 = 0, m_hi = 0;
    const int pos_lo = mt * kQT * pp;
    if constexpr (!PREFIX) {
      seq = pair_hi(pr);
      q0 = p.cu_q_lens[seq];
      ql = p.cu_q_lens[seq + 1] - q0;
      ctx = p.ctx_lens[seq];
      kv_len = ctx + ql;
      keys = ctx + min(pos_lo + kQT * pp, ql);  // keys the item's last row needs
      q_z = q0 + pos_lo;
    } else {
      grp = pair_hi(pr);
      s0 = p.group_starts[grp];
      m_hi = min(pos_lo + kQT * pp, p.group_starts[grp + 1] - s0);
      seq = p.group_ref[grp];
      keys = p.pair_keys[pi];
      kv_len = keys;
      q_z = s0 + pos_lo;
    }
    const int ntiles = (keys + kN - 1) / kN;
    const int nblk_seq = (kv_len + BS - 1) / BS;
    // Q tiles with at least one row (the second is empty when the chunk or
    // group ends within the first): an empty tile gets no MMAs.
    const int nq = (PREFIX ? m_hi : ql) - pos_lo > pp ? 2 : 1;

    if (warp == 0) {
      // =========================== producer ===========================
      bool bad = false;
      int k_issued = 0, v_issued = 0;  // tiles of this item whose K / V copies were issued
      if (lane == 0) {
        // The box holds pp * G of the tile's 128 rows (all of them when G
        // divides 128); the rest of the tile is never read into an output.
        mbar_arrive_expect_tx(b_q, kQT * kH * pp * G * 128);
#pragma unroll
        for (int t = 0; t < kQT; ++t)
#pragma unroll
          for (int h = 0; h < kH; ++h)
            tma_load_3d(sbase + kOffQ + t * kQBytes + h * kQHalf, &qmap, h * 64, kvh * G, q_z + t * pp, b_q);
      }
      const int32_t* bt = p.block_tables + (int64_t)seq * p.max_blocks_per_seq;
      // Block ids are loaded 32 sub-tiles (kTB tiles) at a time, one per
      // lane, a batch ahead of use, so no copy waits on a table load. Lane
      // u < kSubTiles owns sub-tile u of every tile: it picks its id from the
      // batch with a shuffle and issues that sub-tile's copies (lane 0 first
      // waits for the stage and posts its byte count).
      constexpr int kTB = 32 / kSubTiles;
      auto load_batch = [&](int b0) -> int {
        const int j = b0 + lane / kSubTiles, u = lane % kSubTiles;
        int id = 0;
        if (j < ntiles) {
          const int bi = (j * kN + u * 16) / BS;
          if (bi < nblk_seq) {
            id = bt[bi];
            if (id < 0 || id >= p.num_blocks) {
              record_error(p.status, PA_ERR_BLOCK_OOB);
              id = 0;
            }
          }
        }
        return id;
      };
      int b_start = 0;
      int id_cur = load_batch(0), id_next = load_batch(kTB);
      const int su = lane % kSubTiles;
      // Block id of sub-tile su of tile x (x in the current or the next batch).
      auto id_of = [&](int x) -> int {
        const bool nxt = x >= b_start + kTB;
        const int src = ((x - b_start) % kTB) * kSubTiles + su;
        const int a = __shfl_sync(0xffffffffu, id_cur, src);
        const int b = __shfl_sync(0xffffffffu, id_next, src);
        return nxt ? b : a;
      };
      // One tile of K or V: wait for its stage, post the bytes, issue the
      // kSubTiles x 2 boxes.
      auto issue = [&](int x, bool is_v) {
        const int g = tile_base + x;
        const int ns = is_v ? NV : NK;
        const int st = g % ns;
        // e4m3: the copies complete the stage's code barrier; the converter
        // warps complete its full barrier.
        const uint32_t b_full = KV8 ? smem_u32(&bars[(is_v ? kBarVCode : kBarKCode) + st])
                                    : (is_v ? b_vfull0 : b_kfull0) + 8 * st;
        const uint32_t b_empty = (is_v ? b_vempty0 : b_kempty0) + 8 * st;
        const int id = id_of(x);
        if (lane == 0) {
          if (g >= ns && !mbar_wait(b_empty, ((g / ns) & 1) ^ 1, p.status)) bad = true;
          else mbar_arrive_expect_tx(b_full, KV8 ? kKVHalf : kH * kKVHalf);
        }
        bad = __shfl_sync(0xffffffffu, bad, 0);
        if (bad) return;
        if (lane < kSubTiles) {
          const int row = (id * p.num_kv_heads + kvh) * BS + ((x * kN + lane * 16) % BS);
          if constexpr (KV8) {
            // 16 tokens x 128 one-byte codes (2 KB) into the stage's upper half.
            const uint32_t dst = sbase + (is_v ? kOffV : kOffK) + st * kKBytes + kKVHalf + lane * 2048;
            tma_load_2d(dst, is_v ? &vmap : &kmap, 0, row, b_full);
          } else {
            const uint32_t dst = sbase + (is_v ? kOffV : kOffK) + st * kKBytes + lane * 2048;
#pragma unroll
            for (int h = 0; h < kH; ++h) tma_load_2d(dst + h * kKVHalf, is_v ? &vmap : &kmap, h * 64, row, b_full);
          }
        }
        if (is_v) v_issued = x + 1;
        else k_issued = x + 1;
      };
      for (int t = -kVLead; t < ntiles && !bad; ++t) {
        if (t == b_start + kTB) {
          id_cur = id_next;
          b_start += kTB;
          id_next = load_batch(b_start + kTB);
        }
        if (t >= 0) issue(t, false);
        if (!bad && t + kVLead < ntiles) issue(t + kVLead, true);
      }
      if (bad) {
        abort_flag[0] = 1;
        // Let the copies already issued land before the CTA moves on.
        if (lane == 0) {
          mbar_wait(b_q, it & 1, nullptr);
          const uint32_t kb0 = KV8 ? smem_u32(&bars[kBarKCode]) : b_kfull0;
          const uint32_t vb0 = KV8 ? smem_u32(&bars[kBarVCode]) : b_vfull0;
          for (int jj = max(0, k_issued - NK); jj < k_issued; ++jj)
            mbar_wait(kb0 + 8 * ((tile_base + jj) % NK), ((tile_base + jj) / NK) & 1, nullptr);
          for (int jj = max(0, v_issued - NV); jj < v_issued; ++jj)
            mbar_wait(vb0 + 8 * ((tile_base + jj) % NV), ((tile_base + jj) / NV) & 1, nullptr);
        }
      }
    } else if (warp == 1) {
      // ============================= MMA =============================
      if (lane == 0) {
        // e4m3: the converter warps complete q_conv once the Q tiles are in fp16.
        bool bad = !mbar_wait(KV8 ? smem_u32(&bars[kBarQConv]) : b_q, it & 1, p.status);
        uint32_t last_bar = 0, last_phase = 0;  // the last commit: it covers every MMA issued before it
        // Shared-memory descriptors differ only in the start-address field
        // (address >> 4, 14 bits; every operand lies below 256 KB), so each is
        // a base descriptor plus a constant: no per-MMA descriptor assembly.
        const uint64_t dq = sdesc_sw128(sbase + kOffQ, 16, 1024);
        const uint64_t dk = sdesc_sw128(sbase + kOffK, 16, 1024);
        const uint64_t dv = sdesc_sw128(sbase + kOffV, kKVHalf, 1024);
        // S_t(g) = Q_t K(g)^T into S_t (phase ph of s_full[t]).
        auto issue_s = [&](int t, int g, int ph) {
          const uint64_t ka = dk + (uint64_t)((g % NK) * (kKBytes >> 4));
          const uint64_t qa = dq + (uint64_t)(t * (kQBytes >> 4));
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            tc_mma_f16(tmem + col_s(t), qa + (((k >> 2) * kQHalf + (k & 3) * 32) >> 4),
                       ka + (((k >> 2) * kKVHalf + (k & 3) * 32) >> 4), kIdescS, k > 0);
          tc_commit(b_sfull0 + 8 * t);
          last_bar = b_sfull0 + 8 * t;
          last_phase = ph & 1;
        };
        // O_t += P_t(g) V(g), P_t read from tensor memory, once the softmax
        // has written P_t(g) (phase ph of p_full[t]).
        auto issue_pv = [&](int t, int g, int ph, bool acc) -> bool {
          if (!mbar_wait(b_pfull0 + 8 * t, ph & 1, p.status)) return false;
          tc_fence_after();
          const uint64_t va = dv + (uint64_t)((g % NV) * (kKBytes >> 4));
#pragma unroll
          for (int k = 0; k < kN / 16; ++k)
            tc_mma_f16_ta(tmem + col_o(t), tmem + col_s(t) + k * 8, va + ((k * 2048) >> 4), kIdescO,
                          (acc || k > 0) ? 1u : 0u);
          return true;
        };
        auto wait_k = [&](int g) -> bool {
          if (!mbar_wait(b_kfull0 + 8 * (g % NK), (g / NK) & 1, p.status)) return false;
          tc_fence_after();
          return true;
        };
        if (!bad && ntiles > 0) {
          if (!wait_k(tile_base)) {
            bad = true;
          } else {
            issue_s(0, tile_base, tile_base);
            if (nq == 2) issue_s(1, tile_base, tile_base1);
            tc_commit(b_kempty0 + 8 * (tile_base % NK));
          }
        }
        for (int j = 0; j < ntiles && !bad; ++j) {
          const int g = tile_base + j, g1 = tile_base1 + j;  // phases of Q tile 0 / 1
          const bool more = j + 1 < ntiles;
          if (!mbar_wait(b_vfull0 + 8 * (g % NV), (g / NV) & 1, p.status)) { bad = true; break; }
          if (!issue_pv(0, g, g, j > 0)) { bad = true; break; }
          if (!more) {
            tc_commit(b_odone0);
            last_bar = b_odone0;
            last_phase = it & 1;
          } else {
            if (!wait_k(g + 1)) { bad = true; break; }
            issue_s(0, g + 1, g + 1);
          }
          if (nq == 2 && !issue_pv(1, g, g1, j > 0)) { bad = true; break; }
          tc_commit(b_vempty0 + 8 * (g % NV));
          if (nq == 2 && !more) {
            tc_commit(b_odone0 + 8);
            last_bar = b_odone0 + 8;
            last_phase = items1 & 1;
          }
          if (more) {
            if (nq == 2) issue_s(1, g + 1, g1 + 1);
            tc_commit(b_kempty0 + 8 * ((g + 1) % NK));
          }
        }
        if (bad) {
          abort_flag[0] = 1;
          // Let issued MMAs finish before tensor memory is released.
          if (last_bar) mbar_wait(last_bar, last_phase, nullptr);
        }
      }
      __syncwarp();
    } else if (KV8 && warp >= kConvWarp0) {
      // ========================== converters ==========================
      if constexpr (KV8) {
        const int ct = threadIdx.x - 32 * kConvWarp0;  // lane of the converter warp(s)
        bool bad = !mbar_wait(b_q, it & 1, p.status);
        if (!bad && std::is_same<T, __nv_bfloat16>::value) {
          // bf16 Q rows into fp16 in place: x * 2^-e, e from the row's
          // largest magnitude (amax * 2^-e in [2^14, 2^15)), so every element
          // within 2^24 of the row's largest is an exact fp16 normal value.
          int* qexp = reinterpret_cast<int*>(smem + kOffQExp);
          for (int rr = ct; rr < nq * kM; rr += 32 * kConvWarps) {
            const int t = rr / kM, r = rr % kM;
            uint8_t* rb = smem + kOffQ + t * kQBytes + r * 128;
            auto chunk = [&](int c) -> uint4* {  // 16-byte chunk c (8 elements) of the row
              return reinterpret_cast<uint4*>(rb + (c >> 3) * kQHalf + (((c & 7) ^ (r & 7)) << 4));
            };
            float amax = 0.f;
#pragma unroll 4
            for (int c = 0; c < 16; ++c) {
              const uint4 raw = *chunk(c);
              const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
              for (int i = 0; i < 4; ++i)
                amax = fmax3(amax, fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xffff0000u)));
            }
            int ex = 0;
            frexpf(amax, &ex);
            const int sh = amax > 0.f ? ex - 15 : 0;
            const float mul = ldexpf(1.f, -sh);
#pragma unroll 4
            for (int c = 0; c < 16; ++c) {
              const uint4 raw = *chunk(c);
              uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
              for (int i = 0; i < 4; ++i)
                w[i] = MmaOp<__half>::pack(__uint_as_float(w[i] << 16) * mul, __uint_as_float(w[i] & 0xffff0000u) * mul);
              *chunk(c) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            qexp[t * kM + r] = sh;
          }
        }
        fence_async_shared();  // the MMAs read Q through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars[kBarQConv]));
        // K then V of every tile: wait for its codes, widen them in place,
        // one row per lane at a time. The codes of a row sit exactly where
        // the widened upper half (head_dim 64..127) of that same row goes, so
        // reading the whole row before writing it is all the ordering needed.
        for (int j = 0; j < ntiles && !bad; ++j) {
          const int g = tile_base + j;
#pragma unroll 1
          for (int kv = 0; kv < 2; ++kv) {
            const int ns = kv ? NV : NK, st = g % ns;
            if (!mbar_wait(smem_u32(&bars[(kv ? kBarVCode : kBarKCode) + st]), (g / ns) & 1, p.status)) {
              bad = true;
              break;
            }
            uint8_t* base = smem + (kv ? kOffV : kOffK) + st * kKBytes;
#pragma unroll 2
            for (int r = ct; r < kN; r += 32 * kConvWarps) {
              uint4 cr[8];
#pragma unroll
              for (int c = 0; c < 8; ++c)
                cr[c] = *reinterpret_cast<const uint4*>(base + kKVHalf + r * 128 + ((c ^ (r & 7)) << 4));
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                // Codes of head_dim 16c .. 16c + 15 -> two 16-byte chunks of
                // 16-bit values in half c / 4 of the row.
                uint32_t o[8];
                fp8x4_to_f16x4<E5>(cr[c].x, o[0], o[1]);
                fp8x4_to_f16x4<E5>(cr[c].y, o[2], o[3]);
                fp8x4_to_f16x4<E5>(cr[c].z, o[4], o[5]);
                fp8x4_to_f16x4<E5>(cr[c].w, o[6], o[7]);
                uint8_t* rb = base + (c >> 2) * kKVHalf + r * 128;
                const int cc = 2 * (c & 3);
                *reinterpret_cast<uint4*>(rb + ((cc ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                *reinterpret_cast<uint4*>(rb + (((cc + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
              }
            }
            fence_async_shared();  // the MMAs read the stage through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive((kv ? b_vfull0 : b_kfull0) + 8 * st);
          }
        }
        if (bad) abort_flag[0] = 1;
      }
    } else {
      // =========================== softmax ===========================
      const int t = (warp - kSoftmaxWarp0) >> 2;  // Q tile of this warpgroup
      const int q = warp & 3;             // tensor-memory lane quarter of this warp
      const int row = q * 32 + lane;      // packed row of Q tile t owned by this thread
      const uint32_t tl = (uint32_t)(q * 32) << 16;
      const uint32_t ts = tmem + tl + col_s(t), to = tmem + tl + col_o(t);
      const uint32_t b_sfull = b_sfull0 + 8 * t, b_pfull = b_pfull0 + 8 * t, b_odone = b_odone0 + 8 * t;
      const int pos = pos_lo + t * pp + row / G;  // query position (chunk) or group member (prefix)
      const int head = row - (row / G) * G;
      const bool row_used = row < pp * G;  // rows past pp * G hold no (position, head)
      int lim;  // last key this row may see (-1: none)
      if constexpr (!PREFIX) {
        lim = row_used ? min(ctx + pos, kv_len - 1) : -1;
      } else {
        lim = row_used && pos < m_hi ? p.prefix[s0 + pos] - 1 : -1;
      }
      // e4m3: scores are scaled to log2 units before the max (sl2 then 1).
      const float sl2 = KV8 ? 1.f : p.scale_log2;
      float m = -CUDART_INF_F, l = 0.f;
      bool bad = false;
      const bool live = t < nq;  // warpgroup 0 always: it also zeroes V rows past the keys
      const int ph0 = t == 0 ? tile_base : tile_base1;  // phase base of this tile's s_full / p_full
      // e4m3: rf = log2(e) * scale * 2^(this row's Q exponent); kap / pw =
      // 2^kap weight the V scales (see the kernel comment).
      float rf = p.scale_log2;
      constexpr int kKapUnset = 1 << 20;
      int kap = kKapUnset;
      float pw = 1.f;
      const int32_t* btab = p.block_tables + (int64_t)seq * p.max_blocks_per_seq;
      auto load_scales = [&](int jj) -> float2 {
        float2 r = make_float2(0.f, 0.f);
        if constexpr (KV8) {
          if (lane < kSubTiles && jj < ntiles) {
            const int bi = (jj * kN + lane * 16) / BS;
            if (bi < nblk_seq) {
              const int id = btab[bi];
              if (id >= 0 && id < p.num_blocks)
                r = __ldg(reinterpret_cast<const float2*>(p.kv_scales) + (int64_t)id * p.num_kv_heads + kvh);
            }
          }
        }
        return r;
      };
      if constexpr (KV8) {
        if (live) {
          if constexpr (std::is_same<T, __nv_bfloat16>::value) {
            if (!mbar_wait(smem_u32(&bars[kBarQConv]), it & 1, p.status)) bad = true;
            rf = ldexpf(p.scale_log2, reinterpret_cast<const int*>(smem + kOffQExp)[t * kM + row]);
          }
        }
      }
      for (int j = 0; j < ntiles && live && !bad; ++j) {
        const int g = tile_base + j;
        // e4m3: lane u < kSubTiles holds the (K, V) scale of sub-tile u;
        // every thread takes sub-tile u's score factor s_K(u) * rf and V
        // weight s_V(u) * 2^kap from it with a shuffle where it needs them.
        float2 csc = make_float2(0.f, 0.f);
        float kap_r = 1.f;    // e4m3: 2^(new kap - old kap) when kap dropped
        if constexpr (KV8) {
          // Requested before the wait for S, which covers their latency.
          csc = load_scales(j);
          float vmax = lane < kSubTiles ? csc.y : 0.f;
          vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 1));
          vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 2));
          vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 4));
          vmax = __shfl_sync(0xffffffffu, vmax, 0);  // lanes 0..7 hold the max: the same in every lane
          if (vmax > 0.f) {
            // vmax in [2^(ex-1), 2^ex) (a subnormal counts as ex = -126):
            // kap = 7 - ex keeps vmax * 2^kap below 2^7.
            const int ex = (int)((__float_as_uint(vmax) >> 23) & 0xffu) - 126;
            const int kmax = min(7 - ex, 127);
            if (kmax < kap) {
              if (kap != kKapUnset) kap_r = __uint_as_float((uint32_t)(max(kmax - kap, -126) + 127) << 23);
              kap = kmax;
              pw = __uint_as_float((uint32_t)(kmax + 127) << 23);
            }
          }
        }
        if (!mbar_wait(b_sfull, (ph0 + j) & 1, p.status)) { bad = true; break; }
        tc_fence_after();
        const int k0 = j * kN;
        // The causal / prefix mask is skipped when the whole tile is visible
        // to every row of the warp.
        const bool full_vis = __all_sync(0xffffffffu, k0 + kN - 1 <= lim);
        // Exponentials are taken against m. It only moves up when the row max
        // exceeds it by more than 2^8 in probability (then O and l are
        // rescaled); below that, p <= 256 stays exact enough in fp32 and
        // representable in the 16-bit P tile, and O / l is unchanged.
        float alpha = 1.f;
        auto update_max = [&](float mx) {
          if (m == -CUDART_INF_F) {
            m = mx;  // first keys of this row (still -inf for a row without keys)
          } else if ((mx - m) * sl2 > 8.f) {
            alpha = fast_exp2((m - mx) * sl2);
            m = mx;
          }
        };
        // Keys past the sequence end carry p = 0, but their V slots may hold
        // any bits (NaN included): zero those V rows before PV reads them
        // (warpgroup 0 does it before its p_full; PV1 is issued after PV0,
        // which waits for that). False if the wait for V ran out.
        auto zero_v_tail = [&]() -> bool {
          if (t == 0 && k0 + kN > kv_len) {
            const int sv = g % NV;
            if (!mbar_wait(b_vfull0 + 8 * sv, (g / NV) & 1, p.status)) return false;
            uint8_t* vst = smem + kOffV + sv * kKBytes;
            const int first = max(kv_len - k0, 0);
            for (int idx = threadIdx.x - 32 * kSoftmaxWarp0 - 128 * t; idx < (kN - first) * 8 * kH; idx += 128) {
              const int r = first + idx / (8 * kH), c = idx % (8 * kH);  // row, 16-byte chunk over the halves
              *reinterpret_cast<int4*>(vst + (c >> 3) * kKVHalf + r * 128 + (c & 7) * 16) = make_int4(0, 0, 0, 0);
            }
            fence_async_shared();
          }
          return true;
        };
        // Rescale the O row (warp-uniform), before PV of this tile
        // accumulates. PV_t of the previous tile has completed: its commit
        // preceded S_t(g)'s.
        auto rescale_o = [&](float f) {
#pragma unroll 1
          for (int cc = 0; cc < D / 16; ++cc) {
            uint32_t orow[16];
            tmem_ld16(to + cc * 16, orow);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 16; ++c) orow[c] = __float_as_uint(__uint_as_float(orow[c]) * f);
            tmem_st16(to + cc * 16, orow);
          }
        };
        uint64_t rs2 = f2_pack(0.f, 0.f);
        if constexpr (!KV8) {
          uint32_t sr[kN / 32][32];
#pragma unroll
          for (int h = 0; h < kN / 32; ++h) tmem_ld32(ts + h * 32, sr[h]);
          tmem_ld_wait();
          // Raw-score row max (scale > 0 keeps the order).
          if (!full_vis) {
#pragma unroll
            for (int h = 0; h < kN / 32; ++h)
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                const int key = k0 + h * 32 + c;
                if (key > lim) sr[h][c] = __float_as_uint(-CUDART_INF_F);
              }
          }
          float mx = -CUDART_INF_F;
#pragma unroll
          for (int h = 0; h < kN / 32; ++h)
#pragma unroll
            for (int c = 0; c < 32; c += 2) mx = fmax3(mx, __uint_as_float(sr[h][c]), __uint_as_float(sr[h][c + 1]));
          update_max(mx);
          if (!zero_v_tail()) { bad = true; break; }
          const bool rescale = j > 0 && __any_sync(0xffffffffu, alpha != 1.f);
          const float neg = m == -CUDART_INF_F ? 0.f : -m * sl2;
          // p = 2^(s * scale * log2(e) - m * scale * log2(e)), two keys per
          // paired FMA; the row sum accumulates in pairs. P goes to tensor
          // memory 64 keys (32 columns) at a time.
          const uint64_t sl2x2 = f2_pack(sl2, sl2), negx2 = f2_pack(neg, neg);
#pragma unroll
          for (int hh = 0; hh < kN / 64; ++hh) {
            uint32_t pk[32];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
              for (int c = 0; c < 32; c += 2) {
                const int h = hh * 2 + h2;
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[h][c]), __uint_as_float(sr[h][c + 1])), sl2x2, negx2),
                          x0, x1);
                const float a = fast_exp2(x0), b = fast_exp2(x1);
                rs2 = f2_add(rs2, f2_pack(a, b));
                pk[h2 * 16 + c / 2] = MmaOp<T>::pack(a, b);
              }
            // (here, once half of the scores are dead, to keep registers free)
            if (hh == 0 && rescale) rescale_o(alpha);
            tmem_st32(ts + hh * 32, pk);
          }
        } else {
          // 8-bit cache: two passes over the S row in tensor memory, 32 keys
          // at a time, so only 32 scores are held in registers. A score is
          // s * f(group), f = s_K(block) * rf >= 0 per 16-key group (log2
          // units). Pass 1: the row max, taken on the raw scores of each
          // group and scaled once (rounding is monotonic, so this equals the
          // largest scaled score exactly). Pass 2: p = 2^(s * f - m) in one
          // fused multiply-add, the row sum, and P = p * s_V(block) * 2^kap
          // over the S columns already read (P of keys 32h.. goes to columns
          // 16h..). Keys past the row's limit get p = 0 (their scores may be
          // anything, NaN included).
          auto load = [&](uint32_t (&v)[32], int h, float& f0, float& f1) {
            tmem_ld32(ts + h * 32, v);
            f0 = __shfl_sync(0xffffffffu, csc.x, 2 * h) * rf;
            f1 = __shfl_sync(0xffffffffu, csc.x, 2 * h + 1) * rf;
            tmem_ld_wait();
          };
          // max_c(s_c) * f over a group; -inf if every key is masked (also when f == 0).
          auto group_max = [&](const uint32_t (&v)[32], int c0, int key0, float f) -> float {
            float r = -CUDART_INF_F;
            if (full_vis) {
#pragma unroll
              for (int c = 0; c < 16; c += 2) r = fmax3(r, __uint_as_float(v[c0 + c]), __uint_as_float(v[c0 + c + 1]));
            } else {
#pragma unroll
              for (int c = 0; c < 16; ++c) r = key0 + c > lim ? r : fmaxf(r, __uint_as_float(v[c0 + c]));
            }
            return r == -CUDART_INF_F ? r : r * f;
          };
          float mx = -CUDART_INF_F;
#pragma unroll 1
          for (int h = 0; h < kN / 32; ++h) {
            uint32_t v[32];
            float f0, f1;
            load(v, h, f0, f1);
            mx = fmax3(mx, group_max(v, 0, k0 + h * 32, f0), group_max(v, 16, k0 + h * 32 + 16, f1));
          }
          update_max(mx);
          if (!zero_v_tail()) { bad = true; break; }
          // O takes alpha and the drop of kap; l takes alpha alone.
          const float oalpha = alpha * kap_r;
          const bool rescale = j > 0 && __any_sync(0xffffffffu, oalpha != 1.f);
          const float neg = m == -CUDART_INF_F ? 0.f : -m;
          const uint64_t negx2 = f2_pack(neg, neg);
#pragma unroll 1
          for (int h = 0; h < kN / 32; ++h) {
            uint32_t v[32];
            float f0, f1;
            load(v, h, f0, f1);
            const float fv0 = __shfl_sync(0xffffffffu, csc.y, 2 * h) * pw;
            const float fv1 = __shfl_sync(0xffffffffu, csc.y, 2 * h + 1) * pw;
            const uint64_t f0x2 = f2_pack(f0, f0), f1x2 = f2_pack(f1, f1);
            const uint64_t fv0x2 = f2_pack(fv0, fv0), fv1x2 = f2_pack(fv1, fv1);
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), c < 16 ? f0x2 : f1x2, negx2),
                        x0, x1);
              float a = fast_exp2(x0), b = fast_exp2(x1);
              if (!full_vis) {
                const int key = k0 + h * 32 + c;
                a = key > lim ? 0.f : a;
                b = key + 1 > lim ? 0.f : b;
              }
              const uint64_t ab = f2_pack(a, b);
              rs2 = f2_add(rs2, ab);
              float pa, pb;
              f2_unpack(f2_mul(ab, c < 16 ? fv0x2 : fv1x2), pa, pb);
              pk[c / 2] = MmaOp<MT>::pack(pa, pb);
            }
            if (h == 1 && rescale) rescale_o(oalpha);
            tmem_st16(ts + h * 16, pk);
          }
        }
        float rs0, rs1;
        f2_unpack(rs2, rs0, rs1);
        l = l * alpha + (rs0 + rs1);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_pfull);
      }
      if (!live) {
      } else if (!bad && mbar_wait(b_odone, (t == 0 ? it : items1) & 1, p.status)) {
        tc_fence_after();
        if constexpr (!PREFIX) {
          const float inv = 1.f / (l * pw);  // pw = 2^kap with an e4m3 cache, else 1
          T* orow = static_cast<T*>(p.out) + ((int64_t)(q0 + pos) * p.num_q_heads + kvh * G + head) * D;
          const bool valid = row_used && pos < ql;
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t ov[32];
            tmem_ld32(to + cc * 32, ov);
            tmem_ld_wait();
            if (valid) {
#pragma unroll
              for (int c = 0; c < 32; c += 4)
                store4(orow + cc * 32 + c,
                       make_float4(__uint_as_float(ov[c]) * inv, __uint_as_float(ov[c + 1]) * inv,
                                   __uint_as_float(ov[c + 2]) * inv, __uint_as_float(ov[c + 3]) * inv));
            }
          }
        } else {
          // Partial of the prefix in log2 units: reference max m*scale*log2(e),
          // l = sum 2^(s - m) and o~ = sum 2^(s - m) v, into slot 0 of the
          // member's partials.
          const bool valid = lim >= 0;
          const int64_t base = ((int64_t)(s0 + pos) * p.num_q_heads + kvh * G + head) * p.max_parts;
          const float ipw = 1.f / pw;  // exact: a power of two
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t ov[32];
            tmem_ld32(to + cc * 32, ov);
            tmem_ld_wait();
            if (valid) {
#pragma unroll
              for (int c = 0; c < 32; c += 4)
                __stcg(reinterpret_cast<float4*>(p.part_o + base * D + cc * 32 + c),
                       make_float4(__uint_as_float(ov[c]) * ipw, __uint_as_float(ov[c + 1]) * ipw,
                                   __uint_as_float(ov[c + 2]) * ipw, __uint_as_float(ov[c + 3]) * ipw));
            }
          }
          if (valid) __stcg(reinterpret_cast<float2*>(p.part_ml + base * 2), make_float2(m * sl2, l));
        }
      } else {
        bad = true;
      }
      if (bad) abort_flag[0] = 1;
      tc_fence_before();
    }
    tile_base += ntiles;
    if (nq == 2) {
      tile_base1 += ntiles;
      ++items1;
    }
    __syncthreads();
    if (abort_flag[0]) break;
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <typename T, int BS, bool PREFIX, bool KV8, bool E5, int D>
static int launch_prefill_kernel(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 const PrefillParams& p, int ctas, cudaStream_t stream) {
  auto kern = prefill_tc_kernel<T, BS, PREFIX, KV8, E5, D>;
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(kern), pf::kSmem) != PA_OK) return PA_ERR_CUDA;
  return launch_dependent(kern, dim3(ctas), dim3(pf::threads<KV8>()), pf::kSmem, stream, qmap, kmap, vmap, p) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

template <bool PREFIX, bool KV8, bool E5 = false, int D = 128>
static int dispatch_prefill_bs(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               const PrefillParams& p, int ctas, pa_dtype dt, cudaStream_t stream) {
  const bool bf = dt == PA_BF16;
  if (p.block_size == 16)
    return bf ? launch_prefill_kernel<__nv_bfloat16, 16, PREFIX, KV8, E5, D>(qmap, kmap, vmap, p, ctas, stream)
              : launch_prefill_kernel<__half, 16, PREFIX, KV8, E5, D>(qmap, kmap, vmap, p, ctas, stream);
  return bf ? launch_prefill_kernel<__nv_bfloat16, 32, PREFIX, KV8, E5, D>(qmap, kmap, vmap, p, ctas, stream)
            : launch_prefill_kernel<__half, 32, PREFIX, KV8, E5, D>(qmap, kmap, vmap, p, ctas, stream);
}

template <bool PREFIX>
static int dispatch_prefill_kernel(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                   const PrefillParams& p, int ctas, pa_dtype dt, cudaStream_t stream) {
  if (!p.kv_scales)
    return p.head_dim == 64 ? dispatch_prefill_bs<PREFIX, false, false, 64>(qmap, kmap, vmap, p, ctas, dt, stream)
                            : dispatch_prefill_bs<PREFIX, false>(qmap, kmap, vmap, p, ctas, dt, stream);
  return p.kv_fmt == PA_KV_E5M2 ? dispatch_prefill_bs<PREFIX, true, true>(qmap, kmap, vmap, p, ctas, dt, stream)
                                : dispatch_prefill_bs<PREFIX, true>(qmap, kmap, vmap, p, ctas, dt, stream);
}

// Tensor maps of the pools: 16-token sub-tiles of 128 16-bit columns (two
// 64-column boxes), or of 128 e4m3 codes (one 128-byte box).
static int make_pool_maps(const PrefillParams& p, const void* k_cache, const void* v_cache, pa_dtype dt,
                          CUtensorMap* kmap, CUtensorMap* vmap) {
  const int64_t rows = (int64_t)p.num_blocks * p.num_kv_heads * p.block_size;
  int rc = p.kv_scales ? make_u8_tensor_map(kmap, k_cache, rows, p.head_dim, 16)
                       : make_kv_tensor_map(kmap, k_cache, rows, p.head_dim, dt, 16);
  if (rc != PA_OK) return rc;
  return p.kv_scales ? make_u8_tensor_map(vmap, v_cache, rows, p.head_dim, 16)
                     : make_kv_tensor_map(vmap, v_cache, rows, p.head_dim, dt, 16);
}

int launch_prefill(const PrefillParams& p0, const void* k_cache, const void* v_cache, pa_dtype dt,
                   cudaStream_t stream, const DecodeParams* beside) {
  PrefillParams p = p0;
  if (!(p.head_dim == 128 || (p.head_dim == 64 && !p.kv_scales))) return PA_ERR_UNSUPPORTED;
  if (p.group < 1 || p.group > pf::kM) return PA_ERR_UNSUPPORTED;
  p.tile_pos = pf::kM / p.group;
  CUtensorMap qmap, kmap, vmap;
  {
    // q seen as [total_q][num_q_heads][head_dim]; box = 64 columns x G heads x 128/G positions.
    int rc = make_3d_tensor_map(&qmap, p.q, p.total_q, p.num_q_heads, p.head_dim, dt, pf::kM / p.group, p.group, 64);
    if (rc != PA_OK) return rc;
    rc = make_pool_maps(p, k_cache, v_cache, dt, &kmap, &vmap);
    if (rc != PA_OK) return rc;
  }
  const int64_t upper = (int64_t)(p.total_q > 0 ? p.total_q : 1) * p.num_kv_heads;
  p.num_sms = num_sms_current_device();
  const int64_t resident = (int64_t)pf::kCtasPerSm * p.num_sms;
  const int ctas = (int)(upper < resident ? upper : resident);
  p.ctas = ctas;
  if (beside) {
    DecodeParams dp = *beside;
    decode_set_rows(dp, dt);
    if (dt == PA_BF16)
      mixed_plan_kernel<__nv_bfloat16><<<1, 1024, 0, stream>>>(p, dp);
    else
      mixed_plan_kernel<__half><<<1, 1024, 0, stream>>>(p, dp);
  } else {
    prefill_plan_kernel<<<1, 1024, 0, stream>>>(p);
  }
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  return dispatch_prefill_kernel<false>(qmap, kmap, vmap, p, ctas, dt, stream);
}

int launch_prefix_pass(const PrefillParams& p0, const void* k_cache, const void* v_cache, pa_dtype dt,
                       cudaStream_t stream) {
  PrefillParams p = p0;
  if (!(p.head_dim == 128 || (p.head_dim == 64 && !p.kv_scales))) return PA_ERR_UNSUPPORTED;
  if (p.group < 1 || p.group > pf::kM) return PA_ERR_UNSUPPORTED;
  p.tile_pos = pf::kM / p.group;
  CUtensorMap qmap, kmap, vmap;
  // Decode queries [num_seqs][num_q_heads][head_dim]: members of a group are
  // consecutive sequences, so a tile is one box of 128/G sequences x G heads.
  int rc = make_3d_tensor_map(&qmap, p.q, p.num_seqs, p.num_q_heads, p.head_dim, dt, pf::kM / p.group, p.group, 64);
  if (rc != PA_OK) return rc;
  rc = make_pool_maps(p, k_cache, v_cache, dt, &kmap, &vmap);
  if (rc != PA_OK) return rc;
  // The suffix decode runs beside this pass and cannot share an SM with it
  // (shared memory), so the pass takes only a fraction of the SMs: it is
  // bound by the latency of its shared-prefix reads, not by SM count, and
  // the decode keeps the rest streaming from the start.
#ifndef PA_PREFIX_SM_DIV
#define PA_PREFIX_SM_DIV 4
#endif
  const int64_t upper = (int64_t)p.num_seqs * p.num_kv_heads;
  int64_t resident = (int64_t)pf::kCtasPerSm * num_sms_current_device() / PA_PREFIX_SM_DIV;
  if (resident < 1) resident = 1;
  const int ctas = (int)(upper < resident ? upper : resident);
  return dispatch_prefill_kernel<true>(qmap, kmap, vmap, p, ctas, dt, stream);
}

}  // namespace pa
