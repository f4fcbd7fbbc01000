// Chunked-prefill attention on tcgen05 tensor cores (sm_103a).
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

int launch_prefill(const PrefillParams& p, const void* k_cache, const void* v_cache, pa_dtype dt,
                   cudaStream_t stream) {
  (void)p; (void)k_cache; (void)v_cache; (void)dt; (void)stream;
  return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
