/*
 * libpagedattn — paged KV-cache attention for one NVIDIA GB300 (sm_103a).
 *
 * The KV cache of every sequence lives in fixed-size physical blocks of
 * `block_size` tokens; a per-sequence block table maps logical block
 * floor(pos / block_size) to a physical block id, and the token sits at
 * offset pos mod block_size inside it ("High-Throughput Local LLM
 * Infrastructure: Architecting a Distributed Go API Gateway for vLLM &
 * PagedAttention Clusters", section 1.2 "PagedAttention Mechanics & Virtual
 * Page Tables"; "Inside vLLM: Anatomy of a High-Throughput LLM Inference
 * System (2025)", section "Physical Block Mapping and Kernel Invocation").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All pointers named *_cache, q, k, v, out, block_tables, seq_lens,
 *    ctx_lens, cu_q_lens, slot_mapping, seq_ids, positions and workspace are
 *    DEVICE pointers on the current CUDA device, owned by the caller. The
 *    library allocates nothing and keeps no pointer after a call returns.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream). Host-side argument errors return a negative
 *    status BEFORE anything is launched, and then no output is touched.
 *  - Errors found on the device (an out-of-range block id or slot, a
 *    sequence longer than its table or than max_seq_len, a bounded wait that
 *    ran out) never trap: the kernel skips the bad access, records the first
 *    error code in a per-device status word and carries on. pa_get_status()
 *    reads and clears that word. Rows hit by such an error hold unspecified
 *    values.
 *  - Cache layout: k_cache and v_cache are separate pools, each
 *    [num_blocks][num_kv_heads][block_size][head_dim], contiguous, so one
 *    (block, KV head) tile of block_size x head_dim elements is contiguous.
 *  - q, k, v, out and the caches of one call share one dtype (pa_dtype).
 *    Arithmetic is fp32 (scores, softmax, accumulation) whatever the I/O
 *    dtype.
 *  - Grouped-query attention: num_q_heads must be a multiple of
 *    num_kv_heads; query head h reads KV head h / (num_q_heads/num_kv_heads).
 *  - Device pointers to tensors must be 16-byte aligned.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_dtype {
  PA_F32 = 0,
  PA_F16 = 1,
  PA_BF16 = 2
} pa_dtype;

/* Status codes. 0 is success; every error is negative. */
#define PA_OK 0
#define PA_ERR_ARG (-1)         /* null pointer, negative size, bad stride */
#define PA_ERR_DTYPE (-2)       /* dtype not supported by this entry point  */
#define PA_ERR_HEADS (-3)       /* num_q_heads not a multiple of num_kv_heads */
#define PA_ERR_BLOCKSIZE (-4)   /* block_size must be 16 or 32              */
#define PA_ERR_WORKSPACE (-5)   /* workspace null or smaller than required  */
#define PA_ERR_ALIAS (-6)       /* copy_blocks: dst repeated or also a src  */
#define PA_ERR_BLOCK_OOB (-7)   /* device: block id / slot outside the pool */
#define PA_ERR_SEQLEN (-8)      /* device: length < 1, > table, > max given */
#define PA_ERR_CUDA (-9)        /* a CUDA runtime call failed               */
#define PA_ERR_UNSUPPORTED (-10)/* head_dim (or shape) not supported        */
#define PA_ERR_TIMEOUT (-11)    /* device: a bounded wait ran out           */
#define PA_ERR_ALIGN (-12)      /* a tensor pointer is not 16-byte aligned  */
#define PA_ERR_SCRATCH (-13)    /* pa_decode_noalloc: call needs more scratch than its fixed array */

/* Human-readable name of a status code (static storage). */
const char* pa_strerror(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int pa_version(void);

/*
 * pa_get_status — synchronise `stream`, return the first device-side error
 * recorded since the last call (PA_OK if none), and clear it. The status
 * word is per device and shared by all streams. Its device address is looked
 * up once per device and cached for the life of the process, so the library
 * must not be used across a cudaDeviceReset.
 */
int pa_get_status(void* stream);

/*
 * pa_slot_mapping — slot of every new token.
 *   slot_mapping[t] = block_tables[seq_ids[t]][positions[t] / block_size]
 *                     * block_size + positions[t] % block_size
 * (logical block index and block offset of section 1.2 of the "High-
 * Throughput Local LLM Infrastructure" page).
 *   block_tables : int32 [num_seqs][max_blocks_per_seq]
 *   seq_ids      : int32 [num_tokens], 0 <= seq_ids[t] < num_seqs
 *   positions    : int32 [num_tokens], 0 <= positions[t] < max_blocks_per_seq*block_size
 *   slot_mapping : int64 [num_tokens] (output)
 * A token whose seq id, position or physical block (>= num_blocks) is out of
 * range gets slot -1 and PA_ERR_BLOCK_OOB is recorded. num_tokens == 0 is a
 * no-op.
 */
int pa_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq, int32_t num_seqs,
                    const int32_t* seq_ids, const int32_t* positions, int64_t num_tokens,
                    int32_t block_size, int32_t num_blocks, int64_t* slot_mapping, void* stream);

/*
 * pa_reshape_and_cache — scatter new tokens' K and V into their cache slots
 * (section 2.1 "PagedAttention Memory Allocation Life-Cycle", step 4: the
 * kernels write new K/V into the assigned physical blocks).
 *   k, v         : [num_tokens][num_kv_heads][head_dim], contiguous
 *   slot_mapping : int64 [num_tokens]; slot s writes block s / block_size,
 *                  offset s % block_size; s < 0 skips the token (padding);
 *                  s >= num_blocks*block_size records PA_ERR_BLOCK_OOB and
 *                  skips the token
 *   k_cache, v_cache : the pools (layout above), updated in place
 * Bit-exact copy. head_dim * sizeof(dtype) must be a multiple of 16.
 * Two tokens with the same slot race (one of them wins).
 */
int pa_reshape_and_cache(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                         void* k_cache, void* v_cache, int32_t num_blocks, int32_t block_size,
                         int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype, void* stream);

/*
 * pa_copy_blocks — copy-on-write copies: for every pair, the whole K block
 * and V block (all KV heads) dst <- src ("High-Throughput Local LLM
 * Infrastructure...", section 1.2, "Reference Counting & Copy-on-Write";
 * "03 - PagedAttention & the vLLM V1 Architecture", section "The block
 * table walkthrough": the whole block is copied when a write inside it would
 * diverge).
 *   src_dst_pairs : HOST int64 [num_pairs][2] (src, dst). The pairs are
 *                   validated on the host before any launch: every id in
 *                   [0, num_blocks) else PA_ERR_BLOCK_OOB; no dst repeated
 *                   and no dst equal to any src, else PA_ERR_ALIAS. They are
 *                   passed to the kernel by value (no device copy), so the
 *                   host array may be reused as soon as the call returns.
 *   block_bytes   : bytes of one block of one pool
 *                   (num_kv_heads*block_size*head_dim*sizeof(dtype)),
 *                   a multiple of 16.
 * Bit-exact. num_pairs == 0 is a no-op.
 */
int pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* src_dst_pairs, int32_t num_pairs,
                   int32_t num_blocks, int64_t block_bytes, void* stream);

/*
 * pa_swap_blocks — swap preemption ("Inside vLLM: Anatomy of a
 * High-Throughput LLM Inference System (2025)", section "Preemption
 * Mechanics: Swapping vs. Recomputation"; "03 - PagedAttention & the vLLM V1
 * Architecture", section "Preemption & eviction": a preempted sequence's
 * blocks are written out to a host pool and later brought back, possibly
 * into other physical blocks). For every pair, the whole block
 * dst_pool[dst] <- src_pool[src] of the K pool and, if given, the V pool.
 *   src_k, src_v : source pools ([src_num_blocks] blocks of block_bytes)
 *   dst_k, dst_v : destination pools ([dst_num_blocks] blocks)
 *                  Each pool is device memory, managed memory or pinned
 *                  (page-locked: cudaHostAlloc / cudaHostRegister) host
 *                  memory; the kernel reads and writes host memory directly
 *                  (over NVLink-C2C on Grace-Blackwell). Pageable host memory
 *                  returns PA_ERR_ARG. src_v and dst_v are both NULL (one
 *                  pool, e.g. the scales of an e4m3 cache) or both given.
 *   src_dst_pairs : HOST int64 [num_pairs][2] (src, dst), validated before
 *                  any launch: src in [0, src_num_blocks), dst in
 *                  [0, dst_num_blocks) else PA_ERR_BLOCK_OOB; no dst repeated
 *                  and, when src and dst are the same pool, no dst equal to a
 *                  src, else PA_ERR_ALIAS. Passed to the kernel by value.
 *   block_bytes  : bytes of one block of one pool, a multiple of 4
 *                  (PA_ERR_UNSUPPORTED otherwise); 16-byte vectors are used
 *                  when it is a multiple of 16 and the pools are aligned.
 * Bit-exact. num_pairs == 0 is a no-op.
 */
int pa_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v, const int64_t* src_dst_pairs,
                   int32_t num_pairs, int32_t src_num_blocks, int32_t dst_num_blocks, int64_t block_bytes,
                   void* stream);

/*
 * Split-KV partitioning of decode. A sequence of L keys is cut into
 * ceil(L / partition_size) partitions; each is reduced to (m, l, o~)
 * partials (running max, sum of exp(s - m), unnormalised output) in the
 * workspace, and a second pass merges them:
 *   out = sum_p exp(m_p - M) o~_p / sum_p exp(m_p - M) l_p,  M = max_p m_p.
 * A sequence with one partition is written directly. partition_size must be
 * a positive multiple of block_size, or 0 for the library's choice, which
 * depends on (num_seqs, num_kv_heads, num_q_heads, block_size, max_seq_len)
 * and the current device's SM count.
 *
 * pa_decode_partition_size returns the partition size a call with these
 * arguments uses (resolving 0), or a negative status.
 * pa_decode_workspace_size returns the workspace bytes pa_decode needs for
 * these arguments: a work list (about num_seqs*max_parts*4 bytes) plus,
 * when a sequence can need
 * more than one partition, fp32 partials of
 * num_seqs*num_q_heads*max_parts*(head_dim+2)*4 bytes, with
 * max_parts = ceil(max_seq_len / partition_size). It is never 0 for a
 * non-empty batch.
 */
int32_t pa_decode_partition_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t block_size, int32_t max_seq_len, int32_t partition_size);
size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t block_size, int32_t max_seq_len,
                                int32_t partition_size);

/*
 * pa_decode — paged decode attention, one new query token per sequence
 * ("03 - PagedAttention & the vLLM V1 Architecture", section "The attention
 * kernel side": walk the block table, fetch each block's K and V tiles,
 * compute softmax(Q K^T / sqrt(d)) V over the gathered tiles; the attention
 * equation of "Inside vLLM...", section "Physical Block Mapping and Kernel
 * Invocation").
 *   q            : [num_seqs][num_q_heads][head_dim]
 *   block_tables : int32 [num_seqs][max_blocks_per_seq]
 *   seq_lens     : int32 [num_seqs]; sequence i attends to keys
 *                  0 .. seq_lens[i]-1 (its newest token included: cache it
 *                  with pa_reshape_and_cache first)
 *   max_seq_len  : an upper bound of seq_lens (host value; sizes the grid);
 *                  a longer sequence records PA_ERR_SEQLEN
 *   scale        : multiplies q.k (usually 1/sqrt(head_dim))
 *   out          : [num_seqs][num_q_heads][head_dim]
 *   workspace    : device scratch of pa_decode_workspace_size() bytes,
 *                  16-byte aligned; contents need no initialisation (every
 *                  call rewrites what it uses). Two calls whose executions
 *                  overlap on the device (different streams) must not share
 *                  a workspace.
 * Supported: block_size 16 or 32; fp16/bf16 with head_dim 64 or 128 (tensor-
 * core path); fp32 with head_dim a multiple of 32 up to 256 (CUDA-core
 * path). Each KV block is read once per KV head: all query heads of a GQA
 * group are processed together.
 */
int pa_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
              int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
              int32_t num_blocks, float scale, void* out, int32_t partition_size, void* workspace,
              size_t workspace_bytes, pa_dtype dtype, void* stream);

/*
 * pa_decode_shared_prefix — pa_decode for batches in which groups of
 * consecutive sequences share leading KV blocks through their block tables
 * (prefix caching or parallel sampling: several tables name the same
 * refcounted physical blocks, "High-Throughput Local LLM Infrastructure...",
 * section 1.2 "Reference Counting & Copy-on-Write"; "Inside vLLM...",
 * section "Zero-Copy Branching and Parallel Sampling"). The result is the
 * same attention as pa_decode; what changes is the work: each group's shared
 * blocks are read once per KV head for all its members, in one tcgen05
 * tensor-core pass whose rows are (member, query head), and each member's
 * private suffix goes through the split-KV decode kernel; the two are merged
 * with log-sum-exp weights.
 *   group_starts : int32 [num_groups+1] device; group g is the sequences
 *                  group_starts[g] .. group_starts[g+1]-1 (consecutive;
 *                  group_starts[0] = 0, group_starts[num_groups] = num_seqs)
 *   prefix_lens  : int32 [num_seqs] device; a hint: sequence i shares its
 *                  first prefix_lens[i] tokens with its group. A hint is used
 *                  only if it is a positive multiple of block_size, shorter
 *                  than seq_lens[i], and the first prefix_lens[i]/block_size
 *                  table entries of sequence i equal those of the group member
 *                  with the longest hint; otherwise it is ignored for that
 *                  sequence (same result, no saving). Malformed group_starts
 *                  record PA_ERR_ARG and disable every hint.
 *   workspace    : pa_decode_shared_prefix_workspace_size() bytes.
 * Other arguments as pa_decode. fp16/bf16, head_dim 64 or 128, GQA group G of at
 * most 128 (2 * floor(128 / G) members per tensor-core work item, in two
 * tiles; larger groups take several items), scale > 0.
 */
size_t pa_decode_shared_prefix_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                              int32_t head_dim, int32_t block_size, int32_t max_seq_len,
                                              int32_t partition_size, int32_t num_groups);
int pa_decode_shared_prefix(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                            int32_t max_seq_len, const int32_t* group_starts, const int32_t* prefix_lens,
                            int32_t num_groups, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_blocks, float scale, void* out, int32_t partition_size,
                            void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream);

/*
 * pa_decode_step — one decode step in a single call: the same work and
 * results as pa_copy_blocks, pa_slot_mapping, pa_reshape_and_cache and
 * pa_decode, in that order. The decode plan (it reads only block_tables
 * and seq_lens, which the other three do not write) is launched first and
 * the copies, slots and cache write run beside it; the decode kernel starts
 * once the cache write has completed. Arguments as pa_decode_step_shared_prefix
 * without the sharing groups; the workspace is pa_decode_workspace_size()
 * bytes. fp16/bf16 only (PA_ERR_DTYPE otherwise). Every host check runs
 * before the first launch.
 */
int pa_decode_step(const int64_t* cow_pairs, int32_t num_cow_pairs, const int32_t* new_seq_ids,
                   const int32_t* new_positions, const void* k_new, const void* v_new, int64_t num_new_tokens,
                   int64_t* slot_mapping, const void* q, void* k_cache, void* v_cache, const int32_t* block_tables,
                   int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                   int32_t num_blocks, float scale, void* out, int32_t partition_size, void* workspace,
                   size_t workspace_bytes, pa_dtype dtype, void* stream);

/*
 * pa_decode_step_shared_prefix — one decode step of a prefix-sharing batch
 * in a single call: the same work and results as, in this order,
 *   pa_copy_blocks(k_cache, v_cache, cow_pairs, num_cow_pairs, ...),
 *   pa_slot_mapping(block_tables, ..., new_seq_ids, new_positions,
 *                   num_new_tokens, ..., slot_mapping),
 *   pa_reshape_and_cache(k_new, v_new, slot_mapping, num_new_tokens, ...),
 *   pa_decode_shared_prefix(q, k_cache, v_cache, block_tables, ...)
 * (a serving step: copy-on-write of shared blocks about to be written,
 * "High-Throughput Local LLM Infrastructure...", section 1.2; slots and the
 * cache write of the step's new tokens, section 1.2 and "Inside vLLM...",
 * "PagedAttention"; then the attention of the new query tokens).
 * Because every kernel of the step is this library's, the call launches the
 * shared-prefix check first and runs the copies, slots and cache write beside
 * it (it reads only block_tables, seq_lens, group_starts and prefix_lens,
 * which they do not write); the attention kernels start once the cache write
 * has completed.
 *   cow_pairs      : int64 [num_cow_pairs][2] HOST (src, dst) block ids, as
 *                    pa_copy_blocks (may be NULL when num_cow_pairs == 0)
 *   new_seq_ids, new_positions : int32 [num_new_tokens] device, as
 *                    pa_slot_mapping
 *   k_new, v_new   : [num_new_tokens][num_kv_heads][head_dim] device, dtype
 *   slot_mapping   : int64 [num_new_tokens] device, written
 * Other arguments as pa_decode_shared_prefix. Every host check of the four
 * calls runs before the first launch: a rejected call launches nothing.
 * fp16/bf16 only (PA_ERR_DTYPE otherwise). Errors as the four calls.
 */
int pa_decode_step_shared_prefix(const int64_t* cow_pairs, int32_t num_cow_pairs, const int32_t* new_seq_ids,
                                 const int32_t* new_positions, const void* k_new, const void* v_new,
                                 int64_t num_new_tokens, int64_t* slot_mapping, const void* q, void* k_cache,
                                 void* v_cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                                 const int32_t* group_starts, const int32_t* prefix_lens, int32_t num_groups,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int32_t num_blocks, float scale, void* out, int32_t partition_size, void* workspace,
                                 size_t workspace_bytes, pa_dtype dtype, void* stream);

/*
 * pa_decode_noalloc — pa_decode for callers that cannot allocate device
 * memory when they call (for example a plugin running inside another
 * runtime's fixed memory pool, a serving loop that forbids cudaMalloc after
 * start-up because it synchronises the device, or code that must not create
 * allocations while a stream is being captured). The pages describe no such
 * call; it exists for these callers only.
 * Same arguments, checks and results as pa_decode, without workspace
 * arguments: the split-KV scratch is a fixed device array of
 * pa_decode_noalloc_scratch_limit() bytes (64 MiB) inside the library, held
 * on a device until the process exits once the library's code is loaded
 * there. The call itself calls no cudaMalloc, cudaFree or allocating
 * library routine. A call whose pa_decode_workspace_size() exceeds the limit
 * returns PA_ERR_SCRATCH before launching anything.
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it. Under CUDA's default lazy module loading
 * that lookup is what loads the library's module on the device, so the first
 * call makes a one-time 64 MiB device reservation and may synchronise: make
 * it during set-up, before any stream capture and before the point after
 * which the caller may not allocate. All calls share the one array and it
 * keeps the last call's contents (nothing in it needs to start at zero): two
 * calls whose executions overlap on the device, on different streams, race
 * on it. The cached address is that of the device's primary context: do not
 * use the library across a cudaDeviceReset.
 */
size_t pa_decode_noalloc_scratch_limit(void);
int pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                      int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                      int32_t num_blocks, float scale, void* out, int32_t partition_size, pa_dtype dtype,
                      void* stream);

/*
 * pa_chunked_prefill — attention of a mixed batch (prefill chunks and
 * decode rows) over the paged context (chunked prefill: "Tech Radar: vLLM v1
 * Production Engine Architecture...", section 3 "Dynamic Chunked Prefill").
 *   q          : [total_q][num_q_heads][head_dim]; sequence i owns rows
 *                cu_q_lens[i] .. cu_q_lens[i+1]-1
 *   cu_q_lens  : int32 [num_seqs+1], cu_q_lens[0] = 0, non-decreasing,
 *                cu_q_lens[num_seqs] = total_q
 *   ctx_lens   : int32 [num_seqs]; tokens before sequence i's chunk. Row r
 *                of the chunk sits at position ctx_lens[i] + r and attends to
 *                keys 0 .. ctx_lens[i] + r (causal inside the chunk). The
 *                chunk's own K/V must already be cached (pa_reshape_and_cache
 *                of its tokens first).
 *   max_q_len, max_kv_len : host upper bounds of the q_len and of
 *                ctx_len + q_len over the batch; a sequence above them
 *                records PA_ERR_SEQLEN and is skipped
 *   out        : [total_q][num_q_heads][head_dim]
 *   workspace  : pa_chunked_prefill_workspace_size() bytes, 16-byte aligned,
 *                no initialisation needed; not shared by overlapping calls
 * Rows with q_len == 1 go through the decode path (any supported dtype and
 * head_dim). Longer chunks in fp16/bf16 go through a tcgen05 tensor-core
 * kernel that needs head_dim 64 or 128, a GQA group G of at most 128 (a
 * tensor-core tile holds floor(128 / G) query positions x G heads)
 * (PA_ERR_UNSUPPORTED otherwise) and scale > 0 (PA_ERR_ARG); fp32 chunks go
 * through a CUDA-core kernel with exact fp32 arithmetic (head_dim as for
 * fp32 decode, any scale), one query row at a time: exact, not fast.
 * Precondition of the tensor-core kernel, not checked by this version: one
 * chunk holds at most 65536 work items of two tiles, i.e. max_q_len <=
 * 65536 * 2 * floor(128 / G) (131072 rows at G = 128, 2097152 at G = 8);
 * rows of a longer chunk past that bound are not computed.
 */
size_t pa_chunked_prefill_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t block_size, int32_t total_q,
                                         int32_t max_kv_len);
int pa_chunked_prefill(const void* q, int32_t total_q, const int32_t* cu_q_lens, const void* k_cache,
                       const void* v_cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* ctx_lens, int32_t num_seqs, int32_t max_q_len, int32_t max_kv_len,
                       int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                       int32_t num_blocks, float scale, void* out, void* workspace, size_t workspace_bytes,
                       pa_dtype dtype, void* stream);

/*
 * FP8 (e4m3) KV cache with per-block scales ("Tech Radar: vLLM v1 Production
 * Engine Architecture...", section 2, "Hopper TMA Warp Specialization & FP8
 * Kernel Integration", item 3 "FP8 Block-Quantized Caching": keys and values
 * are quantized dynamically to 8-bit floating point at block boundaries,
 * halving the bytes per token; "High-Throughput Local LLM Infrastructure...",
 * section 6, Q5: e4m3).
 *   k_cache, v_cache : uint8 pools [num_blocks][num_kv_heads][block_size][head_dim]
 *                      of e4m3 codes (OCP FP8 E4M3: bias 7, no infinity,
 *                      largest finite 448)
 *   kv_scales        : float32 [num_blocks][num_kv_heads][2], 16-byte aligned:
 *                      the K (index 0) and V (index 1) scale of every (block,
 *                      KV head) tile. Stored value = e4m3 value * scale.
 * Scale rule of a cache write, per (block, KV head, pool), with a = the
 * largest |x| the call writes into the block and o_min the lowest offset it
 * writes there: s_old = 0 if o_min == 0 (the write starts the block afresh),
 * else the stored scale; s_new = max(s_old, fl32(a / 448)); if s_new > s_old
 * > 0 the codes at offsets < o_min are re-encoded as e4m3(fl32(value *
 * fl32(s_old / s_new))); each new row is encoded as e4m3(fl32(x / s_new))
 * (code 0 when s_new == 0). e4m3() rounds to nearest, ties to even, and
 * saturates at +-448. Codes at offsets above the written ones are untouched.
 */

/*
 * pa_reshape_and_cache_fp8 — cache write into the e4m3 pools.
 *   k, v         : [num_tokens][num_kv_heads][head_dim] of dtype (fp32, fp16
 *                  or bf16), 16-byte aligned
 *   slot_mapping : int64 [num_tokens], as for pa_reshape_and_cache. All the
 *                  tokens a call writes into one block must be consecutive
 *                  entries of slot_mapping (entries with slot < 0 may sit
 *                  between them): the order in which a batch lists each
 *                  sequence's new tokens. Tokens of one block split into two
 *                  separate runs race on that block's codes and scale (the
 *                  result is unspecified; nothing outside the block is
 *                  touched).
 * head_dim must be 64 or 128 (PA_ERR_UNSUPPORTED). Bit-exact (see the rule
 * above). Two tokens with the same slot: the later one in the list wins.
 */
int pa_reshape_and_cache_fp8(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                             void* k_cache, void* v_cache, float* kv_scales, int32_t num_blocks, int32_t block_size,
                             int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype, void* stream);

/*
 * pa_copy_blocks_fp8 — copy-on-write for the e4m3 pools: for every pair the
 * whole K and V block and the block's 2 * num_kv_heads scales, dst <- src.
 * Pairs are validated as for pa_copy_blocks (HOST array, PA_ERR_BLOCK_OOB,
 * PA_ERR_ALIAS). Bit-exact.
 */
int pa_copy_blocks_fp8(void* k_cache, void* v_cache, float* kv_scales, const int64_t* src_dst_pairs,
                       int32_t num_pairs, int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                       int32_t head_dim, void* stream);

/*
 * pa_decode_fp8 — pa_decode over the e4m3 pools: every stored value is the
 * e4m3 code times its (block, KV head) scale, and the attention is that of
 * pa_decode on those values. q and out are fp16 or bf16 (dtype;
 * PA_ERR_DTYPE otherwise); head_dim must be 128 (PA_ERR_UNSUPPORTED). The
 * workspace is pa_decode_workspace_size() bytes, as for pa_decode. Codes are
 * widened to fp16 exactly; scores, softmax and accumulation are fp32.
 */
int pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache, const float* kv_scales,
                  const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                  int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t block_size, int32_t num_blocks, float scale, void* out, int32_t partition_size,
                  void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream);

/*
 * pa_decode_shared_prefix_fp8 — pa_decode_shared_prefix over the e4m3 pools:
 * the attention of pa_decode_fp8 (every stored value is the e4m3 code times
 * its (block, KV head) scale), computed as pa_decode_shared_prefix computes
 * it: each group's shared blocks once per KV head for all its members in the
 * tcgen05 tensor-core pass, the private suffixes in the split-KV decode, the
 * two merged with log-sum-exp weights. FP8 block-quantised caching is the
 * page's pairing for serving many concurrent 70B-class sequences ("Tech
 * Radar: vLLM v1 Production Engine Architecture...", section 2, item 3;
 * "High-Throughput Local LLM Infrastructure...", section 6, Q5); prefix
 * sharing is section 1.2 of the latter, "Reference Counting &
 * Copy-on-Write".
 *   k_cache, v_cache, kv_scales : the e4m3 pools and scales, as for
 *                  pa_decode_fp8 (kv_scales 16-byte aligned, else PA_ERR_ALIGN;
 *                  NULL with num_seqs > 0: PA_ERR_ARG)
 * Other arguments, hints, checks and errors as pa_decode_shared_prefix; the
 * workspace is pa_decode_shared_prefix_workspace_size() bytes. q/out fp16
 * or bf16, head_dim 128, GQA group up to 128, scale > 0.
 * The codes are widened to fp16 exactly (a bf16 query row is moved into fp16
 * by a power of two); scores, softmax and accumulation are fp32.
 */
int pa_decode_shared_prefix_fp8(const void* q, const void* k_cache, const void* v_cache, const float* kv_scales,
                                const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                int32_t num_seqs, int32_t max_seq_len, const int32_t* group_starts,
                                const int32_t* prefix_lens, int32_t num_groups, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                float scale, void* out, int32_t partition_size, void* workspace,
                                size_t workspace_bytes, pa_dtype dtype, void* stream);

/*
 * pa_chunked_prefill_fp8 — pa_chunked_prefill over the e4m3 pools (chunked
 * prefill mixed with decode rows, "Tech Radar...", section 3 "Dynamic
 * Chunked Prefill", over the FP8 block-quantised cache of section 2, item
 * 3): the attention of pa_chunked_prefill on the dequantised values. Decode
 * rows go through the e4m3 decode kernel, chunks through the tcgen05 kernel
 * with the codes widened to fp16 in shared memory. Arguments as
 * pa_chunked_prefill plus kv_scales (as pa_decode_fp8); the workspace is
 * pa_chunked_prefill_workspace_size() bytes. q/out fp16 or bf16 (else
 * PA_ERR_DTYPE), head_dim 128 (else PA_ERR_UNSUPPORTED); chunks need a
 * GQA group up to 128 and scale > 0.
 */
int pa_chunked_prefill_fp8(const void* q, int32_t total_q, const int32_t* cu_q_lens, const void* k_cache,
                           const void* v_cache, const float* kv_scales, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* ctx_lens, int32_t num_seqs, int32_t max_q_len,
                           int32_t max_kv_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int32_t num_blocks, float scale, void* out, void* workspace,
                           size_t workspace_bytes, pa_dtype dtype, void* stream);

/*
 * e5m2 KV cache: the other 8-bit format the page names for block-quantised
 * caching ("Tech Radar: vLLM v1 Production Engine Architecture...", section
 * 2, "Hopper TMA Warp Specialization & FP8 Kernel Integration", item 3:
 * e4m3 or e5m2). Same pools, scales, scale rule and errors as the e4m3 calls
 * above, with the OCP FP8 E5M2 codec in place of e4m3:
 *   k_cache, v_cache : uint8 pools [num_blocks][num_kv_heads][block_size][head_dim]
 *                      of e5m2 codes (sign, 5 exponent bits with bias 15, 2
 *                      mantissa bits; exponent field 31 holds infinities and
 *                      NaNs; largest finite 57344)
 *   kv_scales        : float32 [num_blocks][num_kv_heads][2], as above
 * The cache write's scale is s_new = max(s_old, fl32(a / 57344)) and every
 * code is e5m2(fl32(x / s)) (round to nearest even, saturating at +-57344,
 * so the cache only ever writes finite codes); re-encoding on scale growth
 * as for e4m3. The attention calls widen every code to fp16 exactly (an
 * e5m2 code is the upper byte of the fp16 of the same value). Codes past a
 * sequence's end may hold any bits, infinities and NaNs included.
 * pa_copy_blocks_fp8 copies e5m2 pools and their scales unchanged (it moves
 * bytes and scales, whatever the format).
 */

/* pa_reshape_and_cache_e5m2 — pa_reshape_and_cache_fp8 writing e5m2 codes. */
int pa_reshape_and_cache_e5m2(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                              void* k_cache, void* v_cache, float* kv_scales, int32_t num_blocks, int32_t block_size,
                              int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype, void* stream);

/* pa_decode_e5m2 — pa_decode_fp8 over e5m2 pools (same arguments). */
int pa_decode_e5m2(const void* q, const void* k_cache, const void* v_cache, const float* kv_scales,
                   const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                   int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                   int32_t block_size, int32_t num_blocks, float scale, void* out, int32_t partition_size,
                   void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream);

/* pa_decode_shared_prefix_e5m2 — pa_decode_shared_prefix_fp8 over e5m2 pools
 * (same arguments, hints, checks and workspace). */
int pa_decode_shared_prefix_e5m2(const void* q, const void* k_cache, const void* v_cache, const float* kv_scales,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                 int32_t num_seqs, int32_t max_seq_len, const int32_t* group_starts,
                                 const int32_t* prefix_lens, int32_t num_groups, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                 float scale, void* out, int32_t partition_size, void* workspace,
                                 size_t workspace_bytes, pa_dtype dtype, void* stream);

/* pa_chunked_prefill_e5m2 — pa_chunked_prefill_fp8 over e5m2 pools (same
 * arguments and workspace). */
int pa_chunked_prefill_e5m2(const void* q, int32_t total_q, const int32_t* cu_q_lens, const void* k_cache,
                            const void* v_cache, const float* kv_scales, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* ctx_lens, int32_t num_seqs, int32_t max_q_len,
                            int32_t max_kv_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_blocks, float scale, void* out, void* workspace,
                            size_t workspace_bytes, pa_dtype dtype, void* stream);

/*
 * pa_selftest_bounded_wait — exercises the failure path every kernel relies
 * on: one warp waits on an mbarrier that nothing completes; the wait gives up
 * after limit_ns nanoseconds of device time (1 us .. 1 s, else PA_ERR_ARG),
 * records PA_ERR_TIMEOUT in the status word read by pa_get_status, and the
 * kernel returns, leaving the context usable. Nothing faults or traps.
 */
int pa_selftest_bounded_wait(int64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
