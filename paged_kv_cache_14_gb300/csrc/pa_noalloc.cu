// pa_decode_noalloc: paged decode for callers that cannot allocate device
// memory at call time, such as a plugin called inside another runtime's
// fixed memory pool, a serving loop that forbids cudaMalloc after start-up
// (it synchronises the device and fragments the pool), or code that must not
// create allocations while a stream is being captured. Instead of a
// caller-provided workspace, the split-KV scratch lives in one fixed,
// file-scope device array that every device holding this library keeps
// until the process exits.
#include <mutex>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// Upper bound of the scratch a pa_decode_noalloc call may use (64 MiB).
constexpr size_t kNoAllocScratchBytes = 64ull << 20;

// The scratch itself. Host code must not use this name as an address: it is
// a host-side stand-in. Its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDev] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached. nullptr on failure. The
// lookup is also what loads this file's module on a device under lazy module
// loading, so it is the moment the 64 MiB array is reserved there. The cached
// address belongs to the device's primary context: after a cudaDeviceReset it
// is stale, and the library must not be used across one.
void* noalloc_scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
    g_noalloc_addr[dev] = ptr;
  }
  return g_noalloc_addr[dev];
}

}  // namespace
}  // namespace pa

extern "C" size_t pa_decode_noalloc_scratch_limit(void) { return pa::kNoAllocScratchBytes; }

extern "C" int pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                 int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale, void* out,
                                 int32_t partition_size, pa_dtype dtype, void* stream) {
  // An empty or malformed call needs no scratch (size 0) and gets pa_decode's
  // own argument checks and result.
  const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                               max_seq_len, partition_size);
  if (need > pa::kNoAllocScratchBytes) return PA_ERR_SCRATCH;
  void* scratch = pa::noalloc_scratch_address();
  if (!scratch) return PA_ERR_CUDA;
  return pa_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                   num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, out, partition_size, scratch,
                   pa::kNoAllocScratchBytes, dtype, stream);
}
