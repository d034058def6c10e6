// Tiled causal prefill on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
#include "common.cuh"

namespace pkv {

bool prefill_supported(int head_dim, bool bf16) {
  (void)head_dim;
  (void)bf16;
  return false;
}

cudaError_t launch_prefill(const AttnArgs& a, const void* k_cache, const void* v_cache,
                           int head_dim, cudaStream_t stream) {
  (void)a; (void)k_cache; (void)v_cache; (void)head_dim; (void)stream;
  return cudaErrorNotSupported;
}

}  // namespace pkv
