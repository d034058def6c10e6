// Slot-mapped KV-cache write.
//
// "Model execution", section "Flattening a step": slot_mapping names, per new
// token, the physical slot block_id * block_size + offset where its K and V
// go.  "Inside the engine ...", section "Attention over a block table, not a
// contiguous tensor": the KV-write kernel scatters into non-contiguous blocks.
//
// One thread moves one 16-byte chunk of a token's K row and the same chunk of
// its V row (a row is num_kv_heads * head_dim elements, contiguous in both the
// input and the cache), so a warp covers 512 contiguous bytes of each: the
// copy is fully coalesced and HBM-bound (algorithmic bytes per token:
// 2 tensors x (read + write) x row bytes).
#include "common.cuh"

namespace pkv {

__global__ void __launch_bounds__(256) kv_write_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int64_t* __restrict__ slots, int64_t num_tokens, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, int64_t num_slots, uint32_t chunks_per_row,
    int32_t* flag) {
  // Let the next kernel (attention) launch and run its set-up at once: its own
  // dependency wait still returns only after this grid completes.
  pdl_launch_dependents();
  pdl_wait_primary();        // inputs and cache are safe to touch only after the predecessor
  const int64_t total = num_tokens * chunks_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t t = i / chunks_per_row;
    const int64_t c = i - t * chunks_per_row;
    // the row loads do not depend on the slot: all three in flight together
    const int64_t slot = __ldg(slots + t);
    const uint4 kv = __ldcs(k_new + i);     // read once: streaming
    const uint4 vv = __ldcs(v_new + i);
    if (slot < 0) continue;                 // padding token: nothing to write
    if (slot >= num_slots) {                // outside the cache: skip, report
      if (c == 0) raise_flag(flag, PKV_FLAG_BAD_SLOT);
      continue;
    }
    k_cache[slot * chunks_per_row + c] = kv;
    v_cache[slot * chunks_per_row + c] = vv;
  }
}

cudaError_t launch_kv_write(const void* k_new, const void* v_new, const int64_t* slots,
                            int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_slots,
                            uint32_t row_bytes, int32_t* flag, int num_sms,
                            cudaStream_t stream) {
  const uint32_t chunks = row_bytes / 16;
  const int64_t total = num_tokens * chunks;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kv_write_kernel, static_cast<const uint4*>(k_new),
                            static_cast<const uint4*>(v_new), slots, num_tokens,
                            static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_slots,
                            chunks, flag);
}

}  // namespace pkv
