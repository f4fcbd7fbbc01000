// Paged decode attention for sm_103a.
//
// Work decomposition. A sequence of L keys is cut into split-KV partitions of
// `partition` tokens; a work item is one (sequence, partition, KV head
// [, query-row group]). A one-CTA plan kernel lists the items that exist
// (sequence-major, so the sequences of a prefix-sharing group are processed
// close together in time and read their shared blocks from L2) and resets
// the work counter. The main kernel is persistent: each CTA pulls items from
// the counter until none is left.
//
// Inside a CTA (160 threads): warp 4 is the producer. For every item it
// copies the group's query rows into an item slot, then walks the sequence's
// block table over the partition and stages each logical block's K and V
// tiles for the item's KV head (block_size x head_dim contiguous elements of
// the pool each) into a ring of shared-memory stages with 2-D TMA copies
// (128-byte swizzle), one mbarrier per stage. It runs ahead across item
// boundaries, so the ring never drains between items ("03 - PagedAttention &
// the vLLM V1 Architecture", section "The attention kernel side": look the
// block up in the table, fetch its K/V tiles, attend over the gathered
// tiles).
//
// Warps 0-3 consume blocks round-robin. All query heads of the GQA group
// sharing the KV head are the N columns of warp-level MMAs (m16n8k16, fp32
// accumulate) with the block's 16 tokens as the M rows: S^T = K Q^T, an
// online softmax per head column, then O^T += V^T P^T (P^T moves from the
// accumulator layout to the B-operand layout with movmatrix). Every KV block
// is therefore read once per KV head. Decode is HBM-bound (about 8 flop per
// KV byte at group 8): the warp-level MMA has ample headroom, and tcgen05
// tiles (M >= 64) would only pad the 8 live heads.
//
// The four warps' (m, l, o) are merged through shared memory. A sequence
// with one partition is written directly; otherwise the item writes fp32
// partials and a merge kernel combines the partitions of every (sequence,
// query head) with log-sum-exp weights.
//
// fp32 I/O takes a CUDA-core path (exact fp32 FMAs, no TF32) with one CTA
// per (partition, head group, sequence) and the same merge kernel.
#include <math_constants.h>

#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_plan.cuh"

// Bytes of the K/V stage ring of one decode CTA.
#ifndef PA_DECODE_RING_BYTES
#define PA_DECODE_RING_BYTES 65536
#endif
namespace pa {

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}




__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier over `threads` threads that also returns the OR of every
// participant's predicate (the same value in all of them).
__device__ __forceinline__ bool named_barrier_or(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

template <typename T>
__global__ void __launch_bounds__(1024) decode_plan_kernel(const DecodeParams p) {
  pdl_trigger();  // the main kernel may start its set-up now; it waits for this plan
  decode_plan_body<T>(p);
}


// ---------------------------------------------------------------------------
// Persistent tensor-core decode kernel (fp16 / bf16).
// ---------------------------------------------------------------------------
// A stage holds 16 tokens (bf16/fp16 cache) or 32 tokens (e4m3 cache) of a
// sequence's K and V for one KV head: one or two 16-token sub-tiles, each a
// slice of one (block, KV head) tile (a 32-token block fills two sub-tiles;
// the two sub-tiles of an e4m3 stage may come from two blocks). Either way a
// stage is 8 KB at head_dim 128. Stage s is only ever consumed by consumer
// warp s % 4, so each stage's mbarrier is waited on in phase order by one
// warp (a parity wait can never alias a phase not yet begun).
template <int D, int BS, int NT, bool KV8 = false>
struct DecCfg {
  static constexpr int kEsz = KV8 ? 1 : 2;            // bytes per cached element
  static constexpr int kBoxCols = 128 / kEsz;         // elements in one 128-byte TMA box row
  static constexpr int kHalves = D * kEsz / 128;      // 128-byte swizzle boxes across head_dim
  static constexpr int kSubTiles = KV8 ? 2 : 1;       // 16-token sub-tiles per stage
  static constexpr int kStageTok = 16 * kSubTiles;    // tokens per stage
  static constexpr int kSub = 16 * D * kEsz;          // bytes of one sub-tile of K (or V)
  static constexpr int kTile = kSubTiles * kSub;      // K (or V) bytes of a stage
  static constexpr int kStage = 2 * kTile;            // K + V
  static constexpr int kStages = PA_DECODE_RING_BYTES / kStage;
  static constexpr int kHeads = NT * 8;               // query heads per item (MMA N)
  static constexpr int kConsumers = 4;
  static constexpr int kThreads = (kConsumers + 1) * 32;
  static constexpr int kSlots = 2;                    // item slots (metadata + query rows)
  static constexpr int kQBytes = kHeads * D * 2;
  static constexpr int kDp = D + 4;                   // fp32 scratch row stride (+4: bank spread)
  static constexpr size_t kRing = 0;
  static constexpr size_t kQ = kRing + (size_t)kStages * kStage;
  static constexpr size_t kScratch = kQ + (size_t)kSlots * kQBytes;
  static constexpr size_t kMl = kScratch + (size_t)kConsumers * kHeads * kDp * 4;
  static constexpr size_t kMeta = kMl + (size_t)kConsumers * kHeads * 2 * 4;
  static constexpr size_t kValid = kMeta + (size_t)kSlots * 16 * 4;
  static constexpr size_t kBars = (kValid + (size_t)kStages * 4 + 7) & ~size_t(7);
  static constexpr size_t kFlags = kBars + (size_t)(2 * kStages + 2 * kSlots) * 8;
  // e4m3 cache: (K, V) scales of the blocks of each stage's two sub-tiles.
  static constexpr size_t kScl = (kFlags + 16 + 15) & ~size_t(15);
  static constexpr size_t kSmem = kScl + (KV8 ? (size_t)kStages * 16 : 0) + 1024;  // + alignment slack
  static_assert(kStages % kConsumers == 0, "stage s belongs to consumer warp s % 4");
  static_assert(BS % 16 == 0, "block size must be a multiple of 16");
};

// How an item's result leaves the CTA.
enum ItemOut : int {
  kOutPartial = 0,     // fp32 partial into its slot (merged later)
  kOutDirect = 1,      // the sequence's only partition: normalised output
  kOutWithPrefix = 2,  // the only suffix partition: merged here with the prefix pass's partial (slot 0)
  kOutSkip = 3,        // a row with an illegal length (its output was zeroed by the plan): nothing to write
};

struct ItemMeta {
  int seq, qrow, h0, nrows, t_begin, t_end, nsub, jstart, part, n_parts, hg, out_mode, pad[4];
};

template <typename T, int D, int BS, int NT, bool KV8, bool E5 = false>
__global__ void __launch_bounds__(DecCfg<D, BS, NT, KV8>::kThreads, NT == 1 ? 2 : 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                     const DecodeParams p) {
  using C = DecCfg<D, BS, NT, KV8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  ItemMeta* meta = reinterpret_cast<ItemMeta*>(smem + C::kMeta);
  int* stage_valid = reinterpret_cast<int*>(smem + C::kValid);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBars);
  uint64_t* empty = full + C::kStages;
  uint64_t* ifull = empty + C::kStages;
  uint64_t* iempty = ifull + C::kSlots;
  float* scratch = reinterpret_cast<float*>(smem + C::kScratch);
  float* ml = reinterpret_cast<float*>(smem + C::kMl);
  float4* stage_scale = reinterpret_cast<float4*>(smem + C::kScl);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hr = p.num_kv_heads * p.row_groups;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(smem_u32(&ifull[s]), 1);
      mbar_init(smem_u32(&iempty[s]), C::kConsumers);
    }
    fence_barrier_init();
  }
  // Query slots start zeroed: rows past a ragged group stay finite.
  for (int i = threadIdx.x; i < C::kSlots * C::kQBytes / 16; i += blockDim.x)
    reinterpret_cast<int4*>(smem + C::kQ)[i] = make_int4(0, 0, 0, 0);
  __syncthreads();
  // Plain decode waits here for its plan kernel. Shared-prefix decode reads
  // a work list built by the preparation kernel two launches back (complete
  // before this launch: the prefix pass in between waited for it before
  // letting this kernel start), so it streams its suffix at once, overlapping
  // the prefix pass, and waits for that pass only before reading a prefix
  // partial and before it exits (so the merge kernel sees both).
  // The decode rows of a mixed batch (beside) likewise stream at once,
  // beside the chunk kernel, and wait for it before exiting; they let the
  // merge kernel launch only as they exit, so its CTAs take no SM that a
  // decode CTA could use once a chunk CTA leaves.
  // Standalone plain decode runs each CTA's first work item (known without
  // the plan, see DecodeParams::static_first) while the plan runs; the
  // producer waits for the plan before it takes further items.
  const bool overlap = (p.planned && (p.prefix || p.beside)) || p.static_first;
  if (!overlap) pdl_wait();
  if (!p.beside) pdl_trigger();
  const uint32_t ring0 = smem_u32(smem + C::kRing);

  if (warp == C::kConsumers) {
    // =========================== producer ===========================
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    // First item: CTA c < first_static runs item c (row c / hr, its first
    // partition) before the plan has finished; every other CTA, and every
    // later item, comes from the plan's list and the work counter.
    const bool stat = p.static_first && (int)blockIdx.x < p.first_static;
    bool planned_now = !p.static_first;  // the plan's results are visible to this warp
    if (p.static_first && !stat) {
      pdl_wait();
      planned_now = true;
    }
    int total = planned_now ? p.work[1] : 0x7fffffff;
    int next = 0;
    if (stat) {
      next = blockIdx.x;
    } else {
      if (lane == 0) next = atomicAdd(&p.work[0], 1);
      next = __shfl_sync(0xffffffffu, next, 0);
    }
    // The (sequence, partition) pair and length of the next item are loaded
    // one item ahead, so the item switch costs no dependent global loads.
    int next_pr = 0, next_qrow = 0, next_len = 0, next_pfx = 0;
    if (next < total) {
      next_pr = stat ? pack_pair(next / hr, 0) : p.pairs[next / hr];
      decode_row(p, pair_hi(next_pr), next_qrow, next_len);
      next_pfx = p.prefix ? p.prefix[pair_hi(next_pr)] : 0;
    }
    int jg = 0;  // stages issued so far (global stage sequence)
    bool bad = false;
    unsigned fail_mask = 0;  // lanes of the group whose slot wait ran out
    int fail_n = 0;          // size of that group
    constexpr int kSubPerBlock = BS / 16;
    for (int it = 0;; ++it) {
      const int item = next;
      const int slot = it % C::kSlots;
      if (lane == 0 && it >= C::kSlots &&
          !mbar_wait(smem_u32(&iempty[slot]), ((it / C::kSlots) & 1) ^ 1, p.status))
        bad = true;
      bad = __shfl_sync(0xffffffffu, bad, 0);
      if (bad) break;
      if (item >= total) {
        if (lane == 0) {
          meta[slot].seq = -1;
          mbar_arrive(smem_u32(&ifull[slot]));
        }
        break;
      }
      const int pr = next_pr, qrow = next_qrow, len = next_len, pfx = next_pfx;
      // fetch the following item (a CTA that started ahead of the plan does
      // so once its first item is issued)
      if (planned_now && lane == 0) next = atomicAdd(&p.work[0], 1);
      const int hg = item - (item / hr) * hr;
      const int seq = pair_hi(pr), part = pair_lo(pr);
      const int kvh = hg / p.row_groups, rgi = hg - kvh * p.row_groups;
      const int t_begin = pfx + part * p.partition;  // the suffix starts after the shared prefix
      // A row of illegal length (listed only so that first partitions keep
      // their places) gets no stages and no output.
      const bool skip = p.static_first && !len_ok(p, len);
      const int t_end = skip ? t_begin : min(t_begin + p.partition, len);
      const int nsub16 = (t_end - t_begin + 15) / 16;                 // 16-token sub-tiles
      const int nsub = (nsub16 + C::kSubTiles - 1) / C::kSubTiles;    // stages
      // Items are padded to a multiple of 4 stages with empty stages, so
      // every item starts on stage 0 mod 4 and stage u always lands on
      // consumer warp u % 4: the summation order, hence the result, does not
      // depend on which CTA ran the item or what it ran before.
      const int nsub_pad = (nsub + 3) & ~3;
      const int h0 = kvh * p.group + rgi * p.rows_per_cta;
      const int nrows = min(p.rows_per_cta, p.group - rgi * p.rows_per_cta);
      if (lane == 0) {
        ItemMeta& m = meta[slot];
        m.seq = seq;
        m.qrow = qrow;
        m.h0 = h0;
        m.nrows = nrows;
        m.t_begin = t_begin;
        m.t_end = t_end;
        m.nsub = nsub_pad;
        m.jstart = jg;
        m.part = p.slot0 + part;
        const int ns = (len - pfx + p.partition - 1) / p.partition;  // suffix partitions
        m.n_parts = ns + (pfx > 0 ? 1 : 0);
        m.out_mode = skip ? kOutSkip : ns > 1 ? kOutPartial : (pfx > 0 ? kOutWithPrefix : kOutDirect);
        m.hg = seq * hr + hg;
        const uint32_t fb = smem_u32(&ifull[slot]);
        mbar_arrive_expect_tx(fb, nrows * D * 2);
        bulk_copy_g2s(smem_u32(smem + C::kQ + slot * C::kQBytes),
                      static_cast<const T*>(p.q) + ((int64_t)qrow * p.num_q_heads + h0) * D, nrows * D * 2, fb);
      }
      const int32_t* bt = p.block_tables + (int64_t)seq * p.max_blocks_per_seq + t_begin / BS;
      // Lane k holds the physical blocks of the sub-tiles of stage ub + k of
      // a batch of 32 stages (-1: padding) and, for an e4m3 cache, those
      // blocks' (K, V) scales. Loads run ahead of use: at the start of batch
      // ub the scales of batch ub + 32 and the ids of batch ub + 64 are
      // requested, so no batch waits on a table or scale load.
      auto load_ids = [&](int ub, int (&id)[C::kSubTiles]) {
#pragma unroll
        for (int h = 0; h < C::kSubTiles; ++h) {
          id[h] = -1;
          const int sub = (ub + lane) * C::kSubTiles + h;
          if (sub < nsub16) {
            id[h] = bt[sub / kSubPerBlock];
            if (id[h] < 0 || id[h] >= p.num_blocks) {
              record_error(p.status, PA_ERR_BLOCK_OOB);
              id[h] = -1;
            }
          }
        }
      };
      auto load_scales = [&](const int (&id)[C::kSubTiles], float2 (&sc)[C::kSubTiles]) {
#pragma unroll
        for (int h = 0; h < C::kSubTiles; ++h) {
          sc[h] = make_float2(0.f, 0.f);
          if constexpr (KV8) {
            if (id[h] >= 0)
              sc[h] = __ldg(reinterpret_cast<const float2*>(p.kv_scales) + (int64_t)id[h] * p.num_kv_heads + kvh);
          }
        }
      };
      int id[C::kSubTiles], id_next[C::kSubTiles];
      float2 bsc[C::kSubTiles];
      load_ids(0, id);
      load_scales(id, bsc);
      load_ids(32, id_next);
      for (int ub = 0; ub < nsub_pad && !bad; ub += 32) {
        int id_after[C::kSubTiles];
        float2 bsc_next[C::kSubTiles];
        load_scales(id_next, bsc_next);
        load_ids(ub + 64, id_after);
        const int cnt = min(32, nsub_pad - ub);
        // Issue the batch in groups of up to kStages stages, one lane per
        // stage: each lane waits for its own ring slot (all distinct within
        // a group, so no parity wait can alias an older phase), publishes
        // the stage's validity (and scales) and issues its copies, so a
        // single pass of the warp issues a whole group.
        for (int g = 0; g < cnt; g += C::kStages) {
          const int n = min(C::kStages, cnt - g);
          const int src = g + (lane < n ? lane : 0);
          int idk[C::kSubTiles];
          float2 sck[C::kSubTiles];
#pragma unroll
          for (int h = 0; h < C::kSubTiles; ++h) {
            idk[h] = __shfl_sync(0xffffffffu, id[h], src);
            sck[h] = make_float2(0.f, 0.f);
            if constexpr (KV8) {
              sck[h].x = __shfl_sync(0xffffffffu, bsc[h].x, src);
              sck[h].y = __shfl_sync(0xffffffffu, bsc[h].y, src);
            }
          }
          bool failed = false;
          if (lane < n) {
            const int j = jg + lane;
            const int s = j % C::kStages;
            if (j >= C::kStages && !mbar_wait(smem_u32(&empty[s]), ((j / C::kStages) & 1) ^ 1, p.status)) {
              failed = true;
            } else {
              int vmask = 0;
#pragma unroll
              for (int h = 0; h < C::kSubTiles; ++h) vmask |= (idk[h] >= 0 ? 1 : 0) << h;
              stage_valid[s] = vmask;
              if constexpr (KV8) stage_scale[s] = make_float4(sck[0].x, sck[0].y, sck[1].x, sck[1].y);  // published by the arrive below
              const uint32_t fb = smem_u32(&full[s]);
              if (vmask) {
                mbar_arrive_expect_tx(fb, __popc(vmask) * 2 * C::kSub);
                const uint32_t kd = ring0 + s * C::kStage;
#pragma unroll
                for (int h = 0; h < C::kSubTiles; ++h) {
                  if (idk[h] < 0) continue;
                  const int sub = (ub + g + lane) * C::kSubTiles + h;
                  const int32_t row = (idk[h] * p.num_kv_heads + kvh) * BS + (sub % kSubPerBlock) * 16;
#pragma unroll
                  for (int hf = 0; hf < C::kHalves; ++hf) {
                    tma_load_2d(kd + h * C::kSub + hf * 2048, &kmap, hf * C::kBoxCols, row, fb);
                    tma_load_2d(kd + C::kTile + h * C::kSub + hf * 2048, &vmap, hf * C::kBoxCols, row, fb);
                  }
                }
              } else {
                mbar_arrive(fb);
              }
            }
          }
          fail_mask = __ballot_sync(0xffffffffu, failed);
          if (fail_mask) {
            fail_n = n;
            bad = true;
            break;
          }
          jg += n;
        }
        if (ub == 0 && planned_now) {
          // The counter has answered by now: load the next item's metadata
          // while the rest of this item is issued.
          next = __shfl_sync(0xffffffffu, next, 0);
          if (next < total) {
            next_pr = p.pairs[next / hr];
            decode_row(p, pair_hi(next_pr), next_qrow, next_len);
            next_pfx = p.prefix ? p.prefix[pair_hi(next_pr)] : 0;
          }
        }
#pragma unroll
        for (int h = 0; h < C::kSubTiles; ++h) {
          id[h] = id_next[h];
          bsc[h] = bsc_next[h];
          id_next[h] = id_after[h];
        }
      }
      if (bad) break;
      if (!planned_now) {
        // The first item is issued: wait for the plan, then take the next
        // item from its list.
        pdl_wait();
        planned_now = true;
        total = p.work[1];
        if (lane == 0) next = atomicAdd(&p.work[0], 1);
        next = __shfl_sync(0xffffffffu, next, 0);
        if (next < total) {
          next_pr = p.pairs[next / hr];
          decode_row(p, pair_hi(next_pr), next_qrow, next_len);
          next_pfx = p.prefix ? p.prefix[pair_hi(next_pr)] : 0;
        }
      }
    }
    if (bad && lane < C::kStages) {
      // Let copies still in flight land before the CTA exits: lane s waits
      // for the last stage issued on ring slot s. Stages before jg were all
      // issued; of a group that failed (stages jg .. jg + fail_n - 1) only
      // those whose lane did not fail.
      const int sl = lane;
      const int off = ((sl - jg) % C::kStages + C::kStages) % C::kStages;  // slot sl's place in that group
      int last = jg + off;
      if (off >= fail_n || ((fail_mask >> off) & 1u)) last -= C::kStages;
      if (last >= 0) mbar_wait(smem_u32(&full[sl]), (last / C::kStages) & 1, nullptr);
    }
    pdl_wait();
    return;
  }

  // =========================== consumers ===========================
  const int ctid = threadIdx.x;  // 0..127
  const int mi = lane >> 3, rr = lane & 7;
  const int ti = lane & 3;   // column pair (heads 2ti, 2ti+1) of the accumulators
  const int tr = lane >> 2;  // row (token / dim) of the accumulators
  const float sl2 = p.scale_log2;
  for (int it = 0;; ++it) {
    const int slot = it % C::kSlots;
    // A failed wait in any consumer warp ends all four together (the OR is
    // the same in every thread, so no warp is left at a later barrier).
    const bool waited = mbar_wait(smem_u32(&ifull[slot]), (it / C::kSlots) & 1, p.status);
    if (named_barrier_or(1, C::kConsumers * 32, !waited)) break;
    const ItemMeta mt = meta[slot];
    if (mt.seq < 0) break;
    // Q^T fragments (B operand: k = dims, n = heads) from the item slot.
    uint32_t qf[D / 16][NT][2];
    // e4m3 cache: 2^e for the head of each accumulator column, undoing the
    // power-of-two scaling that brought that head's query row into fp16.
    float qsh[NT][2];
    if constexpr (!KV8) {
      const uint32_t qs = smem_u32(smem + C::kQ + slot * C::kQBytes);
#pragma unroll
      for (int kk = 0; kk < D / 16; kk += 2)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int head = nt * 8 + rr;
          const int chunk = (kk + (mi >> 1)) * 2 + (mi & 1);
          ldsm_x4(qs + head * (D * 2) + chunk * 16, qf[kk][nt][0], qf[kk][nt][1], qf[kk + 1][nt][0],
                  qf[kk + 1][nt][1]);
        }
    } else {
      // The e4m3 K fragments hold head_dim elements 16c + 4t .. 16c + 4t + 3
      // of a token in MMA k slots (2t, 2t+1, 2t+8, 2t+9) (see below), so the
      // query takes the same order: lane (g, t) reads 4 consecutive elements
      // of head g per 16-wide chunk. The MMA runs in fp16; a bf16 query row
      // is scaled by 2^-e (e from its largest magnitude) so that it fits
      // fp16's range with bf16's precision, and the scores are scaled back.
      const uint8_t* qs = smem + C::kQ + slot * C::kQBytes;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const T* row = reinterpret_cast<const T*>(qs) + (nt * 8 + tr) * D;
        float v[D / 16][4];
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          const uint2 raw = *reinterpret_cast<const uint2*>(row + c * 16 + 4 * ti);
          const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v[c][i] = to_f32(e[i]);
            amax = fmaxf(amax, fabsf(v[c][i]));
          }
        }
        int sh = 0;
        if constexpr (std::is_same<T, __nv_bfloat16>::value) {
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
          int ex = 0;
          frexpf(amax, &ex);
          sh = amax > 0.f ? ex - 15 : 0;  // amax * 2^-sh in [2^14, 2^15)
        }
        const float mul = ldexpf(1.f, -sh);
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          qf[c][nt][0] = MmaOp<__half>::pack(v[c][0] * mul, v[c][1] * mul);
          qf[c][nt][1] = MmaOp<__half>::pack(v[c][2] * mul, v[c][3] * mul);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) qsh[nt][c] = ldexpf(1.f, __shfl_sync(0xffffffffu, sh, (2 * ti + c) * 4));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&iempty[slot]));

    float o[D / 16][NT][4];
#pragma unroll
    for (int a = 0; a < D / 16; ++a)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) o[a][nt][0] = o[a][nt][1] = o[a][nt][2] = o[a][nt][3] = 0.f;
    float m[NT][2], l[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) m[nt][0] = m[nt][1] = -CUDART_INF_F, l[nt][0] = l[nt][1] = 0.f;
    // e4m3 cache: O accumulates p * s_V(block) * 2^kap * code, with kap the
    // largest exponent that keeps s_V * 2^kap <= 2^15 for every block seen
    // so far (so p * s_V * 2^kap fits fp16); kap only decreases, and O is
    // rescaled by the exact power of two when it does. kap_unset until the
    // first block with a non-zero V scale.
    constexpr int kap_unset = 1 << 20;
    int kap = kap_unset;
    float pw = 0.f;  // 2^kap

    const int jend = mt.jstart + mt.nsub;
    bool bad = false;
    if constexpr (!KV8) {
      // This warp's sub-tiles: j = warp (mod 4), i.e. the stages it owns
      // (jstart is a multiple of 4).
      for (int j = mt.jstart + warp; j < jend; j += C::kConsumers) {
        const int s = j % C::kStages;
        if (!mbar_wait(smem_u32(&full[s]), (j / C::kStages) & 1, p.status)) {
          bad = true;
          break;
        }
        const bool valid = stage_valid[s] != 0;
        // Copy the sub-tile's K and V fragments to registers and hand the
        // stage back at once: the producer refills it while this warp
        // computes, so the ring's bytes stay in flight.
        uint32_t ka[D / 16][4], va[D / 16][4];
        if (valid) {
          const uint32_t kb = ring0 + s * C::kStage;
          const uint32_t vb = kb + C::kTile;
          const int tk_a = (mi & 1) * 8 + rr;   // K rows as the A operand (non-transposed)
          const int tk_v = (mi >> 1) * 8 + rr;  // V rows, transposed into the A operand
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int cg = kk * 2 + (mi >> 1);
            ldsm_x4(kb + (cg >> 3) * 2048 + tk_a * 128 + (((cg & 7) ^ (tk_a & 7)) << 4), ka[kk][0], ka[kk][1],
                    ka[kk][2], ka[kk][3]);
          }
#pragma unroll
          for (int a = 0; a < D / 16; ++a) {
            const int cg = a * 2 + (mi & 1);
            ldsm_x4_t(vb + (cg >> 3) * 2048 + tk_v * 128 + (((cg & 7) ^ (tk_v & 7)) << 4), va[a][0], va[a][1],
                      va[a][2], va[a][3]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        if (!valid) continue;
        const int tok0 = mt.t_begin + (j - mt.jstart) * 16;
        // S^T = K Q^T: rows = 16 tokens, columns = heads. Two accumulator
        // chains over the head_dim halves shorten the dependent MMA chain.
        float sc[NT][4], sc2[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = sc2[nt][0] = sc2[nt][1] = sc2[nt][2] = sc2[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; kk += 2)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            MmaOp<T>::run(sc[nt], ka[kk], qf[kk][nt][0], qf[kk][nt][1]);
            MmaOp<T>::run(sc2[nt], ka[kk + 1], qf[kk + 1][nt][0], qf[kk + 1][nt][1]);
          }
        // Scale to log2 units, mask keys past the partition end.
        const int t_lo = tok0 + tr, t_hi = tok0 + tr + 8;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          sc[nt][0] = t_lo < mt.t_end ? (sc[nt][0] + sc2[nt][0]) * sl2 : -CUDART_INF_F;
          sc[nt][1] = t_lo < mt.t_end ? (sc[nt][1] + sc2[nt][1]) * sl2 : -CUDART_INF_F;
          sc[nt][2] = t_hi < mt.t_end ? (sc[nt][2] + sc2[nt][2]) * sl2 : -CUDART_INF_F;
          sc[nt][3] = t_hi < mt.t_end ? (sc[nt][3] + sc2[nt][3]) * sl2 : -CUDART_INF_F;
        }
        // Online softmax per head column (max over the 16 tokens = over
        // the 8 lanes that share lane % 4).
        bool rescale = false;
        float alpha[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float mx = fmaxf(sc[nt][c], sc[nt][c + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m[nt][c], mx);
            const bool dead = mn == -CUDART_INF_F;
            alpha[nt][c] = dead ? 1.f : exp2f(m[nt][c] - mn);
            rescale |= mn != m[nt][c];
            const float p0 = dead ? 0.f : exp2f(sc[nt][c] - mn);
            const float p1 = dead ? 0.f : exp2f(sc[nt][c + 2] - mn);
            sc[nt][c] = p0;
            sc[nt][c + 2] = p1;
            l[nt][c] = l[nt][c] * alpha[nt][c] + (p0 + p1);
            m[nt][c] = mn;
          }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int a = 0; a < D / 16; ++a)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              o[a][nt][0] *= alpha[nt][0];
              o[a][nt][1] *= alpha[nt][1];
              o[a][nt][2] *= alpha[nt][0];
              o[a][nt][3] *= alpha[nt][1];
            }
        }
        // P^T as the B operand (k = tokens, n = heads).
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          pb[nt][0] = movmatrix_trans(MmaOp<T>::pack(sc[nt][0], sc[nt][1]));
          pb[nt][1] = movmatrix_trans(MmaOp<T>::pack(sc[nt][2], sc[nt][3]));
        }
        // Keys past the end carry p = 0, but their V slots may hold any
        // bits (NaN included): zero those V elements so 0 * V stays 0.
        if (tok0 + 16 > mt.t_end) {
          const int tk = tok0 + 2 * ti;
          const uint32_t keep_lo = (tk < mt.t_end ? 0x0000ffffu : 0u) | (tk + 1 < mt.t_end ? 0xffff0000u : 0u);
          const uint32_t keep_hi = (tk + 8 < mt.t_end ? 0x0000ffffu : 0u) | (tk + 9 < mt.t_end ? 0xffff0000u : 0u);
#pragma unroll
          for (int a = 0; a < D / 16; ++a) {
            va[a][0] &= keep_lo;
            va[a][1] &= keep_lo;
            va[a][2] &= keep_hi;
            va[a][3] &= keep_hi;
          }
        }
        // O^T += V^T P^T: rows = head_dim (16 per m-tile), k = tokens.
#pragma unroll
        for (int a = 0; a < D / 16; ++a)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) MmaOp<T>::run(o[a][nt], va[a], pb[nt][0], pb[nt][1]);
      }
    } else {
      // e4m3 cache: a stage holds two 16-token sub-tiles (halves), so the
      // softmax reductions and the bookkeeping are paid once per 32 tokens
      // and the two halves' MMA chains overlap.
      for (int j = mt.jstart + warp; j < jend; j += C::kConsumers) {
        const int s = j % C::kStages;
        if (!mbar_wait(smem_u32(&full[s]), (j / C::kStages) & 1, p.status)) {
          bad = true;
          break;
        }
        const int vmask = stage_valid[s];
        const bool valid0 = (vmask & 1) != 0, valid1 = (vmask & 2) != 0;
        // Raw codes of both halves: 8x16-byte matrices, lane group mi reads
        // tokens (mi & 1) * 8 + rr of 16-byte chunk 2q + (mi >> 1).
        uint32_t kr[2][D / 32][4], vr[2][D / 32][4];
        float2 bs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        {
          const int tk = (mi & 1) * 8 + rr;
          const float4 sc4 = stage_scale[s];
          bs[0] = make_float2(sc4.x, sc4.y);
          bs[1] = make_float2(sc4.z, sc4.w);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (!(h ? valid1 : valid0)) continue;
            const uint32_t kb = ring0 + s * C::kStage + h * C::kSub, vb = kb + C::kTile;
#pragma unroll
            for (int q2 = 0; q2 < D / 32; ++q2) {
              const int cg = 2 * q2 + (mi >> 1);
              const uint32_t off = (cg >> 3) * 2048 + tk * 128 + (((cg & 7) ^ (tk & 7)) << 4);
              ldsm_x4(kb + off, kr[h][q2][0], kr[h][q2][1], kr[h][q2][2], kr[h][q2][3]);
              ldsm_x4_t(vb + off, vr[h][q2][0], vr[h][q2][1], vr[h][q2][2], vr[h][q2][3]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        if (!valid0 && !valid1) continue;
        const int tok0 = mt.t_begin + (j - mt.jstart) * 32;
        // S^T per half: K widened to fp16 pairs (A rows g / g+8; k slots
        // (2t, 2t+1) <- elements (4t, 4t+1), (2t+8, 2t+9) <- (4t+2, 4t+3)
        // of the 16-element chunk), times the query in the same order.
        float sc[2][NT][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float acc[NT][4], acc2[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = acc2[nt][0] = acc2[nt][1] = acc2[nt][2] =
                acc2[nt][3] = 0.f;
          if (h ? valid1 : valid0) {
#pragma unroll
            for (int q2 = 0; q2 < D / 32; ++q2) {
              uint32_t a0[4], a1[4];
              fp8x4_to_f16x4<E5>(kr[h][q2][0], a0[0], a0[2]);
              fp8x4_to_f16x4<E5>(kr[h][q2][1], a0[1], a0[3]);
              fp8x4_to_f16x4<E5>(kr[h][q2][2], a1[0], a1[2]);
              fp8x4_to_f16x4<E5>(kr[h][q2][3], a1[1], a1[3]);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                MmaOp<__half>::run(acc[nt], a0, qf[2 * q2][nt][0], qf[2 * q2][nt][1]);
                MmaOp<__half>::run(acc2[nt], a1, qf[2 * q2 + 1][nt][0], qf[2 * q2 + 1][nt][1]);
              }
            }
          }
          // Scale by the block's K scale, the query rows' exponents and
          // log2(e) * softmax scale; mask keys past the partition end.
          const int t_lo = tok0 + 16 * h + tr, t_hi = t_lo + 8;
          const bool vh = h ? valid1 : valid0;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const float f0 = sl2 * bs[h].x * qsh[nt][0], f1 = sl2 * bs[h].x * qsh[nt][1];
            sc[h][nt][0] = vh && t_lo < mt.t_end ? (acc[nt][0] + acc2[nt][0]) * f0 : -CUDART_INF_F;
            sc[h][nt][1] = vh && t_lo < mt.t_end ? (acc[nt][1] + acc2[nt][1]) * f1 : -CUDART_INF_F;
            sc[h][nt][2] = vh && t_hi < mt.t_end ? (acc[nt][2] + acc2[nt][2]) * f0 : -CUDART_INF_F;
            sc[h][nt][3] = vh && t_hi < mt.t_end ? (acc[nt][3] + acc2[nt][3]) * f1 : -CUDART_INF_F;
          }
        }
        // Online softmax per head column over the 32 tokens.
        bool rescale = false;
        float alpha[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float mx = fmaxf(fmaxf(sc[0][nt][c], sc[0][nt][c + 2]), fmaxf(sc[1][nt][c], sc[1][nt][c + 2]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m[nt][c], mx);
            const bool dead = mn == -CUDART_INF_F;
            alpha[nt][c] = dead ? 1.f : fast_exp2(m[nt][c] - mn);
            rescale |= mn != m[nt][c];
            float ps = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float p0 = dead ? 0.f : fast_exp2(sc[h][nt][c] - mn);
              const float p1 = dead ? 0.f : fast_exp2(sc[h][nt][c + 2] - mn);
              sc[h][nt][c] = p0;
              sc[h][nt][c + 2] = p1;
              ps += p0 + p1;
            }
            l[nt][c] = l[nt][c] * alpha[nt][c] + ps;
            m[nt][c] = mn;
          }
        // The weight of each half's V codes is p * s_V * 2^kap; lower kap
        // first if a half's V scale needs it.
        float fv[2];
        {
          const float smax = fmaxf(valid0 ? bs[0].y : 0.f, valid1 ? bs[1].y : 0.f);
          if (smax > 0.f) {
            // smax in [2^(ex-1), 2^ex) with ex from the exponent field (a
            // subnormal counts as ex = -126, which keeps smax * 2^kap below 2^15).
            const int ex = (int)((__float_as_uint(smax) >> 23) & 0xffu) - 126;
            const int kmax = min(15 - ex, 127);
            if (kmax < kap) {
              const int d = kap == kap_unset ? -1000 : kmax - kap;
              const float r = d < -126 ? 0.f : __uint_as_float((uint32_t)(d + 127) << 23);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) alpha[nt][0] *= r, alpha[nt][1] *= r;
              rescale = true;
              kap = kmax;
              pw = __uint_as_float((uint32_t)(kmax + 127) << 23);
            }
          }
          fv[0] = valid0 ? bs[0].y * pw : 0.f;
          fv[1] = valid1 ? bs[1].y * pw : 0.f;
        }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int a = 0; a < D / 16; ++a)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              o[a][nt][0] *= alpha[nt][0];
              o[a][nt][1] *= alpha[nt][1];
              o[a][nt][2] *= alpha[nt][0];
              o[a][nt][3] *= alpha[nt][1];
            }
        }
        // O^T += V^T P^T per half. V (transposed load): lane (g, t) holds
        // elements (2g, 2g+1) of tokens 2t and 2t+1; a byte permute pairs
        // the tokens per element, so A row g <- element 2g and row g+8 <-
        // element 2g+1 of the chunk, k slots = the tokens.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!(h ? valid1 : valid0)) continue;
          uint32_t pb[NT][2];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            pb[nt][0] = movmatrix_trans(MmaOp<__half>::pack(sc[h][nt][0] * fv[h], sc[h][nt][1] * fv[h]));
            pb[nt][1] = movmatrix_trans(MmaOp<__half>::pack(sc[h][nt][2] * fv[h], sc[h][nt][3] * fv[h]));
          }
          const int th = tok0 + 16 * h;
          uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
          if (th + 16 > mt.t_end) {
            // Keys past the end carry p = 0, but their V codes may hold any
            // bits (NaN included): zero those V elements so 0 * V stays 0.
            const int tk = th + 2 * ti;
            keep_lo = (tk < mt.t_end ? 0x0000ffffu : 0u) | (tk + 1 < mt.t_end ? 0xffff0000u : 0u);
            keep_hi = (tk + 8 < mt.t_end ? 0x0000ffffu : 0u) | (tk + 9 < mt.t_end ? 0xffff0000u : 0u);
          }
#pragma unroll
          for (int q2 = 0; q2 < D / 32; ++q2) {
            uint32_t a0[4], a1[4];
            fp8x4_to_f16x4<E5>(__byte_perm(vr[h][q2][0], 0, 0x3120), a0[0], a0[1]);
            fp8x4_to_f16x4<E5>(__byte_perm(vr[h][q2][1], 0, 0x3120), a0[2], a0[3]);
            fp8x4_to_f16x4<E5>(__byte_perm(vr[h][q2][2], 0, 0x3120), a1[0], a1[1]);
            fp8x4_to_f16x4<E5>(__byte_perm(vr[h][q2][3], 0, 0x3120), a1[2], a1[3]);
            a0[0] &= keep_lo, a0[1] &= keep_lo, a0[2] &= keep_hi, a0[3] &= keep_hi;
            a1[0] &= keep_lo, a1[1] &= keep_lo, a1[2] &= keep_hi, a1[3] &= keep_hi;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              MmaOp<__half>::run(o[2 * q2][nt], a0, pb[nt][0], pb[nt][1]);
              MmaOp<__half>::run(o[2 * q2 + 1][nt], a1, pb[nt][0], pb[nt][1]);
            }
          }
        }
      }
    }
    if (named_barrier_or(1, C::kConsumers * 32, bad)) break;

    // ---- merge the four warps: per head h, (m_w, l_w, o_w) ----
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float lv = l[nt][c];
        lv += __shfl_xor_sync(0xffffffffu, lv, 4);
        lv += __shfl_xor_sync(0xffffffffu, lv, 8);
        lv += __shfl_xor_sync(0xffffffffu, lv, 16);
        l[nt][c] = lv;
        if (tr == 0) {
          const int h = nt * 8 + 2 * ti + c;
          ml[(warp * C::kHeads + h) * 2 + 0] = m[nt][c];
          ml[(warp * C::kHeads + h) * 2 + 1] = lv;
        }
      }
    named_barrier_sync(1, C::kConsumers * 32);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int h = nt * 8 + 2 * ti + c;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < C::kConsumers; ++w) M = fmaxf(M, ml[(w * C::kHeads + h) * 2]);
        float f = m[nt][c] == -CUDART_INF_F ? 0.f : exp2f(m[nt][c] - M);
        float* row = scratch + (warp * C::kHeads + h) * C::kDp;
        if constexpr (KV8) {
          // O rows: m-row tr <-> element 16a + 2tr, m-row tr + 8 <-> 16a + 2tr + 1.
          f = pw > 0.f ? f / pw : 0.f;  // undo 2^kap (exact: a power of two)
#pragma unroll
          for (int a = 0; a < D / 16; ++a)
            *reinterpret_cast<float2*>(row + a * 16 + 2 * tr) = make_float2(o[a][nt][c] * f, o[a][nt][c + 2] * f);
        } else {
#pragma unroll
          for (int a = 0; a < D / 16; ++a) {
            row[a * 16 + tr] = o[a][nt][c] * f;
            row[a * 16 + tr + 8] = o[a][nt][c + 2] * f;
          }
        }
      }
    named_barrier_sync(1, C::kConsumers * 32);
    for (int idx = ctid; idx < mt.nrows * (D / 4); idx += C::kConsumers * 32) {
      const int h = idx / (D / 4);
      const int d4 = (idx - h * (D / 4)) * 4;
      float M = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < C::kConsumers; ++w) M = fmaxf(M, ml[(w * C::kHeads + h) * 2]);
      float L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < C::kConsumers; ++w) {
        const float mw = ml[(w * C::kHeads + h) * 2];
        L += mw == -CUDART_INF_F ? 0.f : ml[(w * C::kHeads + h) * 2 + 1] * exp2f(mw - M);
        const float4 v = *reinterpret_cast<const float4*>(scratch + (w * C::kHeads + h) * C::kDp + d4);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      if (mt.out_mode == kOutSkip) {
        // nothing to write
      } else if (mt.out_mode == kOutWithPrefix) {
        // Merge with the prefix pass's partial (written by the previous
        // launch on this stream): M' = max(M, m0), weights 2^(M - M'), 2^(m0 - M').
        pdl_wait();
        const int64_t b0 = ((int64_t)mt.seq * p.num_q_heads + mt.h0 + h) * p.max_parts;
        const float2 ml0 = __ldcg(reinterpret_cast<const float2*>(p.part_ml + b0 * 2));
        const float4 o0 = __ldcg(reinterpret_cast<const float4*>(p.part_o + b0 * D + d4));
        const float Mx = fmaxf(M, ml0.x);
        const float w1 = exp2f(M - Mx), w0 = exp2f(ml0.x - Mx);
        const float inv = 1.f / (L * w1 + ml0.y * w0);
        store4(static_cast<T*>(p.out) + ((int64_t)mt.qrow * p.num_q_heads + mt.h0 + h) * D + d4,
               make_float4((acc.x * w1 + o0.x * w0) * inv, (acc.y * w1 + o0.y * w0) * inv,
                           (acc.z * w1 + o0.z * w0) * inv, (acc.w * w1 + o0.w * w0) * inv));
      } else if (mt.out_mode == kOutDirect) {
        const float inv = 1.f / L;
        store4(static_cast<T*>(p.out) + ((int64_t)mt.qrow * p.num_q_heads + mt.h0 + h) * D + d4,
               make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
      } else {
        const int64_t base = ((int64_t)mt.seq * p.num_q_heads + mt.h0 + h) * p.max_parts + mt.part;
        __stcg(reinterpret_cast<float4*>(p.part_o + base * D + d4), acc);
        if (d4 == 0) __stcg(reinterpret_cast<float2*>(p.part_ml + base * 2), make_float2(M, L));
      }
    }
    named_barrier_sync(1, C::kConsumers * 32);
  }
  pdl_wait();
}

// ---------------------------------------------------------------------------
// fp32 I/O: CUDA-core path. One CTA per (partition, head group, sequence);
// four warps take the partition's tokens round-robin, each lane holds
// head_dim/32 dimensions and dot products are reduced across the warp.
// ---------------------------------------------------------------------------
template <int VEC>
__global__ void __launch_bounds__(128) decode_simt_kernel(const DecodeParams p) {
  pdl_wait();
  pdl_trigger();
  constexpr int D = VEC * 32;
  constexpr int ROWS = 8;
  constexpr int NW = 4;
  __shared__ int32_t ids[kMaxPartition / 16];
  __shared__ float mls[NW][ROWS][2];
  __shared__ float ob[NW][ROWS][D];

  const int part = blockIdx.x;
  const int kvh = blockIdx.y / p.row_groups;
  const int rg = blockIdx.y - kvh * p.row_groups;
  const int seq = blockIdx.z;
  const int BS = p.block_size;
  int qrow, len;
  if (!decode_row(p, seq, qrow, len)) return;
  if (!len_ok(p, len)) return;  // reported and zeroed by the plan kernel
  const int h0 = kvh * p.group + rg * p.rows_per_cta;
  const int nrows = min(p.rows_per_cta, p.group - rg * p.rows_per_cta);
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
      mls[warp][g][0] = m[g];
      mls[warp][g][1] = l[g];
    }
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < ROWS; ++g) {
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mls[w][g][0]);
    const float f = m[g] == -CUDART_INF_F ? 0.f : exp2f(m[g] - M);
#pragma unroll
    for (int v = 0; v < VEC; ++v) ob[warp][g][lane + 32 * v] = o[g][v] * f;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nrows * D; idx += blockDim.x) {
    const int g = idx / D, d = idx - g * D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mls[w][g][0]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = mls[w][g][0];
      L += mw == -CUDART_INF_F ? 0.f : mls[w][g][1] * exp2f(mw - M);
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
// M = max_p m_p (scores are kept in log2 units). One warp per (sequence,
// query head), eight heads per work unit, over the sequences the plan listed
// (those with more than one partition), on a fixed grid. Each lane reads
// every partition's (m, l) and its own four head_dim columns of every
// partial, all loads in flight together (up to eight partitions), then
// accumulates in partition order.
template <typename T>
__global__ void __launch_bounds__(256) splitkv_merge_kernel(const DecodeParams p) {
  pdl_wait();  // every partial of the decode kernel, and the plan's list
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hgroups = (p.num_q_heads + 7) / 8;
  // The first unit's list entry is read together with the count (the
  // grid never exceeds num_seqs x hgroups, so the index is in range).
  int4 e = p.merge_list[blockIdx.x / hgroups];
  const int units = p.work[2] * hgroups;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    if (u != (int)blockIdx.x) e = p.merge_list[u / hgroups];
    const int h = (u - (u / hgroups) * hgroups) * 8 + warp;
    if (h >= p.num_q_heads) continue;
    const int seq = e.x, qrow = e.y, first = e.z, n = e.w;
    const int64_t base = ((int64_t)seq * p.num_q_heads + h) * p.max_parts + first;
    const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + base;
    const int D = p.head_dim;
    T* out = static_cast<T*>(p.out) + ((int64_t)qrow * p.num_q_heads + h) * D;
    for (int c0 = 0; c0 < D; c0 += 128) {
      const int d4 = c0 + lane * 4;
      const bool col = d4 < D;
      const float* src = p.part_o + base * D + d4;
      float M = -CUDART_INF_F, L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      auto add = [&](float2 mv, float4 ov) {
        const float w = mv.x == -CUDART_INF_F ? 0.f : exp2f(mv.x - M);
        L += w * mv.y;
        acc.x = fmaf(w, ov.x, acc.x);
        acc.y = fmaf(w, ov.y, acc.y);
        acc.z = fmaf(w, ov.z, acc.z);
        acc.w = fmaf(w, ov.w, acc.w);
      };
      if (n <= 8) {
        float2 mv[8];
        float4 ov[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          mv[i] = make_float2(-CUDART_INF_F, 0.f);
          ov[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (i < n) {
            mv[i] = __ldcg(ml + i);
            if (col) ov[i] = __ldcg(reinterpret_cast<const float4*>(src + (int64_t)i * D));
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) M = fmaxf(M, mv[i].x);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i < n) add(mv[i], ov[i]);
      } else {
        for (int i = 0; i < n; ++i) M = fmaxf(M, __ldcg(ml + i).x);
        for (int i = 0; i < n; ++i)
          add(__ldcg(ml + i), col ? __ldcg(reinterpret_cast<const float4*>(src + (int64_t)i * D))
                                  : make_float4(0.f, 0.f, 0.f, 0.f));
      }
      const float invL = 1.f / L;
      if (col) store4(out + d4, make_float4(acc.x * invL, acc.y * invL, acc.z * invL, acc.w * invL));
    }
  }
}

static int launch_merge(const DecodeParams& p, pa_dtype dt, cudaStream_t stream) {
  if (p.max_parts <= 1) return PA_OK;
  // A fixed grid (one wave of 256-thread CTAs) over however many sequences
  // the plan listed.
  const int64_t units = (int64_t)p.num_seqs * ((p.num_q_heads + 7) / 8);
  const int64_t cap = 4LL * num_sms_current_device();
  const dim3 grid((unsigned)(units < cap ? units : cap));
  cudaError_t e;
  if (dt == PA_F32)
    e = launch_dependent(splitkv_merge_kernel<float>, grid, dim3(256), 0, stream, p);
  else if (dt == PA_BF16)
    e = launch_dependent(splitkv_merge_kernel<__nv_bfloat16>, grid, dim3(256), 0, stream, p);
  else
    e = launch_dependent(splitkv_merge_kernel<__half>, grid, dim3(256), 0, stream, p);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <typename T, int D, int BS, int NT, bool KV8, bool E5 = false>
static int launch_tc(const DecodeParams& p, cudaStream_t stream) {
  using C = DecCfg<D, BS, NT, KV8>;
  constexpr pa_dtype dt = std::is_same<T, __half>::value ? PA_F16 : PA_BF16;
  CUtensorMap kmap, vmap;
  const int64_t rows = (int64_t)p.num_blocks * p.num_kv_heads * BS;
  int rc;
  if constexpr (KV8) {
    rc = make_u8_tensor_map(&kmap, p.k_cache, rows, D, 16);
    if (rc != PA_OK) return rc;
    rc = make_u8_tensor_map(&vmap, p.v_cache, rows, D, 16);
  } else {
    rc = make_kv_tensor_map(&kmap, p.k_cache, rows, D, dt, 16);
    if (rc != PA_OK) return rc;
    rc = make_kv_tensor_map(&vmap, p.v_cache, rows, D, dt, 16);
  }
  if (rc != PA_OK) return rc;
  auto kern = decode_tc_kernel<T, D, BS, NT, KV8, E5>;
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(kern), (int)C::kSmem) != PA_OK) return PA_ERR_CUDA;
  const int64_t upper = (int64_t)p.num_seqs * p.max_parts * p.num_kv_heads * p.row_groups;
  const int64_t resident = (NT == 1 ? 2LL : 1LL) * num_sms_current_device();
  const int ctas = (int)(upper < resident ? upper : resident);
  DecodeParams pk = p;
  if (!p.planned) {
    // Standalone plain decode: the first items run while the plan runs.
    if (!p.cu_q_lens && !p.prefix) {
      const int64_t firsts = (int64_t)p.num_seqs * p.num_kv_heads * p.row_groups;
      pk.static_first = 1;
      pk.first_static = (int32_t)(firsts < ctas ? firsts : ctas);
    }
    decode_plan_kernel<T><<<1, 1024, 0, stream>>>(pk);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  }
  if (launch_dependent(kern, dim3(ctas), dim3(C::kThreads), C::kSmem, stream, kmap, vmap, pk) != cudaSuccess)
    return PA_ERR_CUDA;
  return launch_merge(pk, dt, stream);
}

// fp32 I/O chunk rows (q_len > 1) of a mixed batch: a CUDA-core path with
// exact fp32 FMAs (the tensor cores' fp32 input kind rounds to TF32). One
// CTA per (query row, KV-head row group); its four warps take the row's keys
// 0 .. ctx + r round-robin, each lane holding head_dim / 32 dimensions, and
// merge through shared memory. Every row reads its keys itself (no reuse
// across the rows of a chunk): a path for exactness, not speed.
template <int VEC>
__global__ void __launch_bounds__(128) prefill_simt_kernel(const DecodeParams p) {
  pdl_wait();
  pdl_trigger();
  constexpr int D = VEC * 32;
  constexpr int ROWS = 8;
  constexpr int NW = 4;
  __shared__ float mls[NW][ROWS][2];
  __shared__ float ob[NW][ROWS][D];

  const int t = blockIdx.x;  // query row
  const int kvh = blockIdx.y / p.row_groups;
  const int rg = blockIdx.y - kvh * p.row_groups;
  // The row's sequence: the last s with cu_q_lens[s] <= t.
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cu_q_lens[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  const int seq = lo;
  const int q0 = p.cu_q_lens[seq], ql = p.cu_q_lens[seq + 1] - q0;
  if (ql <= 1 || t < q0 || t >= q0 + ql) return;  // decode rows go through the decode kernels
  const int ctx = p.lens[seq];
  const int BS = p.block_size;
  if (ctx < 0 || ctx + ql > p.len_cap || ctx + ql > p.max_blocks_per_seq * BS) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && t == q0) record_error(p.status, PA_ERR_SEQLEN);
    return;
  }
  const int nkeys = ctx + (t - q0) + 1;  // causal: keys 0 .. ctx + r
  const int h0 = kvh * p.group + rg * p.rows_per_cta;
  const int nrows = min(p.rows_per_cta, p.group - rg * p.rows_per_cta);
  const int32_t* bt = p.block_tables + (int64_t)seq * p.max_blocks_per_seq;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* qb = static_cast<const float*>(p.q) + ((int64_t)t * p.num_q_heads + h0) * D;
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
  for (int key = warp; key < nkeys; key += NW) {
    const int id = bt[key / BS];
    if (id < 0 || id >= p.num_blocks) {
      if (lane == 0) record_error(p.status, PA_ERR_BLOCK_OOB);
      continue;
    }
    const int64_t row = ((int64_t)id * p.num_kv_heads + kvh) * BS + (key % BS);
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
      const float sc = d * p.scale_log2;
      const float mn = fmaxf(m[g], sc);
      const float a = exp2f(m[g] - mn);
      const float e = exp2f(sc - mn);
      l[g] = l[g] * a + e;
#pragma unroll
      for (int v = 0; v < VEC; ++v) o[g][v] = fmaf(e, vv[v], o[g][v] * a);
      m[g] = mn;
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int g = 0; g < ROWS; ++g) {
      mls[warp][g][0] = m[g];
      mls[warp][g][1] = l[g];
    }
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < ROWS; ++g) {
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mls[w][g][0]);
    const float f = m[g] == -CUDART_INF_F ? 0.f : exp2f(m[g] - M);
#pragma unroll
    for (int v = 0; v < VEC; ++v) ob[warp][g][lane + 32 * v] = o[g][v] * f;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nrows * D; idx += blockDim.x) {
    const int g = idx / D, d = idx - g * D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mls[w][g][0]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = mls[w][g][0];
      L += mw == -CUDART_INF_F ? 0.f : mls[w][g][1] * exp2f(mw - M);
      acc += ob[w][g][d];
    }
    static_cast<float*>(p.out)[((int64_t)t * p.num_q_heads + h0 + g) * D + d] = acc / L;
  }
}

template <int VEC>
static int launch_prefill_simt_vec(const DecodeParams& p, int32_t total_q, cudaStream_t stream) {
  const dim3 grid((unsigned)total_q, (unsigned)(p.num_kv_heads * p.row_groups));
  return launch_dependent(prefill_simt_kernel<VEC>, grid, dim3(128), 0, stream, p) == cudaSuccess ? PA_OK
                                                                                               : PA_ERR_CUDA;
}

int launch_prefill_simt(const DecodeParams& p0, int32_t total_q, cudaStream_t stream) {
  DecodeParams p = p0;
  decode_set_rows(p, PA_F32);
  if ((int64_t)p.num_kv_heads * p.row_groups > 65535) return PA_ERR_UNSUPPORTED;
  switch (p.head_dim) {
    case 32: return launch_prefill_simt_vec<1>(p, total_q, stream);
    case 64: return launch_prefill_simt_vec<2>(p, total_q, stream);
    case 96: return launch_prefill_simt_vec<3>(p, total_q, stream);
    case 128: return launch_prefill_simt_vec<4>(p, total_q, stream);
    case 160: return launch_prefill_simt_vec<5>(p, total_q, stream);
    case 192: return launch_prefill_simt_vec<6>(p, total_q, stream);
    case 224: return launch_prefill_simt_vec<7>(p, total_q, stream);
    case 256: return launch_prefill_simt_vec<8>(p, total_q, stream);
  }
  return PA_ERR_UNSUPPORTED;
}

template <int VEC>
static int launch_simt(const DecodeParams& p, cudaStream_t stream) {
  decode_plan_kernel<float><<<1, 1024, 0, stream>>>(p);
  dim3 grid(p.max_parts, p.num_kv_heads * p.row_groups, p.num_seqs);
  if (launch_dependent(decode_simt_kernel<VEC>, grid, dim3(128), 0, stream, p) != cudaSuccess) return PA_ERR_CUDA;
  return launch_merge(p, PA_F32, stream);
}

template <typename T>
static int launch_tc_dispatch(const DecodeParams& p, cudaStream_t stream) {
  const int nt = p.rows_per_cta <= 8 ? 1 : 2;
  if (p.kv_scales) {  // 8-bit cache: head_dim 128 only
    if (p.head_dim != 128) return PA_ERR_UNSUPPORTED;
    const int k8 = ((p.kv_fmt == PA_KV_E5M2 ? 1 : 0) * 2 + (p.block_size == 16 ? 0 : 1)) * 2 + (nt - 1);
    switch (k8) {
      case 0: return launch_tc<T, 128, 16, 1, true>(p, stream);
      case 1: return launch_tc<T, 128, 16, 2, true>(p, stream);
      case 2: return launch_tc<T, 128, 32, 1, true>(p, stream);
      case 3: return launch_tc<T, 128, 32, 2, true>(p, stream);
      case 4: return launch_tc<T, 128, 16, 1, true, true>(p, stream);
      case 5: return launch_tc<T, 128, 16, 2, true, true>(p, stream);
      case 6: return launch_tc<T, 128, 32, 1, true, true>(p, stream);
      case 7: return launch_tc<T, 128, 32, 2, true, true>(p, stream);
    }
    return PA_ERR_UNSUPPORTED;
  }
  const int key = ((p.head_dim == 64 ? 0 : 1) * 2 + (p.block_size == 16 ? 0 : 1)) * 2 + (nt - 1);
  switch (key) {
    case 0: return launch_tc<T, 64, 16, 1, false>(p, stream);
    case 1: return launch_tc<T, 64, 16, 2, false>(p, stream);
    case 2: return launch_tc<T, 64, 32, 1, false>(p, stream);
    case 3: return launch_tc<T, 64, 32, 2, false>(p, stream);
    case 4: return launch_tc<T, 128, 16, 1, false>(p, stream);
    case 5: return launch_tc<T, 128, 16, 2, false>(p, stream);
    case 6: return launch_tc<T, 128, 32, 1, false>(p, stream);
    case 7: return launch_tc<T, 128, 32, 2, false>(p, stream);
  }
  return PA_ERR_UNSUPPORTED;
}

void decode_set_rows(DecodeParams& p, pa_dtype dt) {
  const int rows_max = dt == PA_F32 ? 8 : 16;
  p.rows_per_cta = p.group < rows_max ? p.group : rows_max;
  p.row_groups = (p.group + p.rows_per_cta - 1) / p.rows_per_cta;
}

int launch_decode(const DecodeParams& p0, pa_dtype dt, cudaStream_t stream) {
  DecodeParams p = p0;
  decode_set_rows(p, dt);
  if ((int64_t)p.num_kv_heads * p.row_groups > 65535) return PA_ERR_UNSUPPORTED;
  if (dt == PA_F32) {
    if (p.kv_scales) return PA_ERR_DTYPE;
    switch (p.head_dim) {
      case 32: return launch_simt<1>(p, stream);
      case 64: return launch_simt<2>(p, stream);
      case 96: return launch_simt<3>(p, stream);
      case 128: return launch_simt<4>(p, stream);
      case 160: return launch_simt<5>(p, stream);
      case 192: return launch_simt<6>(p, stream);
      case 224: return launch_simt<7>(p, stream);
      case 256: return launch_simt<8>(p, stream);
    }
    return PA_ERR_UNSUPPORTED;
  }
  if (p.head_dim != 64 && p.head_dim != 128) return PA_ERR_UNSUPPORTED;
  return dt == PA_BF16 ? launch_tc_dispatch<__nv_bfloat16>(p, stream) : launch_tc_dispatch<__half>(p, stream);
}

int launch_decode_plan(const DecodeParams& p0, pa_dtype dt, cudaStream_t stream) {
  DecodeParams p = p0;
  decode_set_rows(p, dt);
  if (dt == PA_BF16)
    decode_plan_kernel<__nv_bfloat16><<<1, 1024, 0, stream>>>(p);
  else if (dt == PA_F16)
    decode_plan_kernel<__half><<<1, 1024, 0, stream>>>(p);
  else
    return PA_ERR_DTYPE;
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
