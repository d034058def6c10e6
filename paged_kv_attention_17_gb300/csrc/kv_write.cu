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

// E4M3 variant: each thread converts 8 consecutive elements of a token's K
// row and of its V row (fp32 or bf16) to codes of value / scale - the
// division correctly rounded in fp32, then the nearest code (ties to even,
// saturating at 448) - and stores them as one 8-byte word per tensor.
// Algorithmic bytes per token: 2 x row elements x (input size + 1).
template <typename S>
__device__ __forceinline__ void load8(const S* p, float (&f)[8]) {
  if constexpr (sizeof(S) == 4) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  } else {
    const uint4 w = __ldcs(reinterpret_cast<const uint4*>(p));
    f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
  }
}

__device__ __forceinline__ uint2 encode8(const float (&f)[8], float scale) {
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    c[i] = float2_to_e4m3x2(__fdiv_rn(f[2 * i], scale), __fdiv_rn(f[2 * i + 1], scale));
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

template <typename S>
__global__ void __launch_bounds__(256) kv_write_e4m3_kernel(
    const S* __restrict__ k_new, const S* __restrict__ v_new, const int64_t* __restrict__ slots,
    int64_t num_tokens, uint2* __restrict__ k_cache, uint2* __restrict__ v_cache,
    int64_t num_slots, uint32_t groups_per_row, float k_scale, float v_scale, int32_t* flag) {
  pdl_launch_dependents();
  pdl_wait_primary();
  const int64_t total = num_tokens * groups_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t t = i / groups_per_row;
    const int64_t c = i - t * groups_per_row;
    const int64_t slot = __ldg(slots + t);
    float kf[8], vf[8];
    load8<S>(k_new + i * 8, kf);
    load8<S>(v_new + i * 8, vf);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (c == 0) raise_flag(flag, PKV_FLAG_BAD_SLOT);
      continue;
    }
    k_cache[slot * groups_per_row + c] = encode8(kf, k_scale);
    v_cache[slot * groups_per_row + c] = encode8(vf, v_scale);
  }
}

// Staging copy of a step's packed inputs (pkv_stage_inputs): 16-byte words
// from src (device memory, or pinned host memory mapped into the device's
// address space) to dst in device memory.  "Inside the engine ...", section
// on CUDA graphs: inputs are copied asynchronously into fixed buffers before
// the step's kernels run.  Done with the device's own loads rather than a
// copy-engine transfer, so it sits in the kernels' dependent-launch chain:
// the next kernel is released at once (its set-up and hinted loads overlap
// the transfer) and its dependency wait returns when the copy is complete.
// A CUDA graph holding copy nodes instead runs them on the copy engine
// between the kernels, each a few microseconds with the chain broken.
// Every thread issues all its loads before its first store, so one round
// trip over the host link covers the whole transfer.
constexpr int kStageWords = 4;          // 16-byte words per thread per pass

__global__ void __launch_bounds__(256) stage_copy_kernel(const uint4* __restrict__ src,
                                                         uint4* __restrict__ dst, int64_t words) {
  pdl_launch_dependents();
  pdl_wait_primary();                   // earlier work on the stream may still use src or dst
  const int64_t pass = static_cast<int64_t>(gridDim.x) * blockDim.x * kStageWords;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x * kStageWords + threadIdx.x;
       base < words; base += pass) {
    uint4 w[kStageWords];
#pragma unroll
    for (int u = 0; u < kStageWords; ++u) {
      const int64_t i = base + static_cast<int64_t>(u) * blockDim.x;
      if (i < words) w[u] = __ldcs(src + i);
    }
#pragma unroll
    for (int u = 0; u < kStageWords; ++u) {
      const int64_t i = base + static_cast<int64_t>(u) * blockDim.x;
      if (i < words) dst[i] = w[u];
    }
  }
}

cudaError_t launch_stage_copy(void* dst, const void* src, int64_t bytes, int num_sms,
                              cudaStream_t stream) {
  const int64_t words = bytes / 16;
  const int threads = 256;
  int64_t blocks = (words + threads * kStageWords - 1) / (threads * kStageWords);
  const int64_t cap = static_cast<int64_t>(num_sms) * 4;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stage_copy_kernel, static_cast<const uint4*>(src),
                            static_cast<uint4*>(dst), words);
}

static cudaLaunchConfig_t write_config(int64_t total, int num_sms, cudaStream_t stream,
                                       cudaLaunchAttribute* attr) {
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

cudaError_t launch_kv_write(const void* k_new, const void* v_new, const int64_t* slots,
                            int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_slots,
                            uint32_t row_bytes, int32_t* flag, int num_sms,
                            cudaStream_t stream) {
  const uint32_t chunks = row_bytes / 16;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = write_config(num_tokens * chunks, num_sms, stream, attr);
  return cudaLaunchKernelEx(&cfg, kv_write_kernel, static_cast<const uint4*>(k_new),
                            static_cast<const uint4*>(v_new), slots, num_tokens,
                            static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_slots,
                            chunks, flag);
}

// row_elems: num_kv_heads * head_dim, a multiple of 8.
cudaError_t launch_kv_write_e4m3(const void* k_new, const void* v_new, bool src_bf16,
                                 const int64_t* slots, int64_t num_tokens, void* k_cache,
                                 void* v_cache, int64_t num_slots, uint32_t row_elems,
                                 float k_scale, float v_scale, int32_t* flag, int num_sms,
                                 cudaStream_t stream) {
  const uint32_t groups = row_elems / 8;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = write_config(num_tokens * groups, num_sms, stream, attr);
  if (src_bf16)
    return cudaLaunchKernelEx(&cfg, kv_write_e4m3_kernel<__nv_bfloat16>,
                              static_cast<const __nv_bfloat16*>(k_new),
                              static_cast<const __nv_bfloat16*>(v_new), slots, num_tokens,
                              static_cast<uint2*>(k_cache), static_cast<uint2*>(v_cache),
                              num_slots, groups, k_scale, v_scale, flag);
  return cudaLaunchKernelEx(&cfg, kv_write_e4m3_kernel<float>, static_cast<const float*>(k_new),
                            static_cast<const float*>(v_new), slots, num_tokens,
                            static_cast<uint2*>(k_cache), static_cast<uint2*>(v_cache), num_slots,
                            groups, k_scale, v_scale, flag);
}

}  // namespace pkv
