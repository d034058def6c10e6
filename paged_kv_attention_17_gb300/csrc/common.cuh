// Device-side helpers shared by the kernels: shared-memory barriers, TMA
// loads, bounded waits and the launch-argument structs.  Inline PTX only; no
// library code.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

// One 8-bit E4M3 code of an FP8 KV cache (the value is decoded in registers).
struct e4m3_t {
  uint8_t bits;
};

// Cache element type of a launch.
enum class ElemType { kF32, kBf16, kE4m3 };

constexpr int kBlock = 16;                       // tokens per KV-cache block
constexpr int kDecodeMaxQ = PKV_DECODE_MAX_QLEN; // decode-class bound on q_len
constexpr int kMaxSplits = 64;
constexpr int kLptMaxSeqs = 256;                // longest-first dispatch: up to this many requests
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // ~2 s per wait

// ---------------------------------------------------------------------------
// Launch arguments
// ---------------------------------------------------------------------------
struct AttnArgs {
  const void* q;
  void* out;
  float* lse_out;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* block_table;
  int max_blocks_per_seq;
  int num_seqs;
  int64_t num_tokens;
  int max_query_len;
  int max_seq_len;        // host bound on seq_lens (speculative table prefetch)
  int hq, hkv, group;
  float scale_log2;       // softmax_scale * log2(e) (* k_scale for E4M3 caches): log2-domain scores
  float v_scale;          // output multiplier: v_scale for E4M3 caches, else 1
  int causal;
  int window;             // > 0: row at position p sees keys j > p - window only
  int num_splits;         // >= 1
  int long_rows;          // decode kernel also runs requests with q_len > kDecodeMaxQ
  float* ws_o;            // [S][num_seqs][kDecodeMaxQ][hq][D]
  float* ws_lse;          // [S][num_seqs][kDecodeMaxQ][hq] (log2 domain)
  int32_t* flag;
  int64_t num_blocks;
  const void* k_cache;    // cache bases, for L2 prefetch hints
  const void* v_cache;
  // Shared-prefix (cascade) passes.  1: every row of the batch as one request
  // over the prefix_len shared keys (non-causal), split partials to the
  // workspace; 2: each request over its own keys, its result written as
  // partial cascade_slot; 3: merge of num_splits partials per row.  Partials
  // are indexed [slot][token][q head] in these passes.  0: a plain call.
  int cascade;
  int prefix_len;
  int cascade_slot;
  // Fused write (decode-class steps): each CTA stores the K/V rows (its KV
  // head) of the new tokens whose positions it reads, before loading them.
  int fuse_write;
  // Prefill launched behind the same call's decode kernel: its dependency
  // wait moves from the start to each CTA's exit (see prefill.cu).
  int defer_wait;
  // Prefill: an odd GQA group pairs two query tiles of one head per CTA
  // instead of two query heads of one tile (see prefill.cu).
  int pair_tiles;
  // Unsplit decode launch of 2..256 requests: blockIdx.z is read as a rank of
  // the requests by decreasing seq_len (longest first; see decode.cu).
  int lpt;
  const void* k_new;      // [num_tokens, hkv, D], the cache's element type
  const void* v_new;
  const int64_t* slots;   // slot_mapping
  float wk_scale, wv_scale;  // E4M3 caches: the write stores codes of value / scale
};

// ---------------------------------------------------------------------------
// Small device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void raise_flag(int32_t* flag, int bits) {
  if (flag != nullptr) atomicOr(flag, bits);
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// bf16 pair (packed in a 32-bit word, element 0 in the low half) -> two floats
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two E4M3 codes (element 0 in the low byte of the 16-bit value) -> two
// floats, through the hardware E4M3x2 -> f16x2 conversion (exact: every E4M3
// value is an f16 value).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
  uint32_t h2;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
      : "=r"(h2)
      : "r"(two_codes));
  float lo, hi;
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\t"
      "cvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
  return make_float2(lo, hi);
}

// Two floats -> two E4M3 codes (a in the low byte): round to nearest even,
// magnitudes beyond 448 saturate to 448, NaN stays NaN.
__device__ __forceinline__ uint32_t float2_to_e4m3x2(float a, float b) {
  uint32_t r;
  asm("{\n\t.reg .b16 c;\n\tcvt.rn.satfinite.e4m3x2.f32 c, %1, %2;\n\tcvt.u32.u16 %0, c;\n\t}"
      : "=r"(r)
      : "f"(b), "f"(a));
  return r;
}

// ---------------------------------------------------------------------------
// mbarrier (shared memory, CTA scope)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One wait attempt: the thread is suspended (not spinning) until the phase
// completes or a time hint of about 1 ms elapses.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

// Non-blocking check: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_ready(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after about
// two seconds and returns false, so a broken pipeline can never hang the GPU.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_test(bar, parity)) return true;
    if (globaltimer() - t0 > kWaitLimitNs) return false;
  }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), no multicast
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Read-only load issued where it stands in the program (volatile asm): used
// for loads that must be in flight early rather than next to their first use.
__device__ __forceinline__ int32_t ld_early(const int32_t* p) {
  int32_t v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// 32- and 64-bit read-only loads issued where they stand (volatile asm).
__device__ __forceinline__ uint32_t ld_early_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld_early_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_early_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// Bring the 128-byte line holding p into L2 (a hint: no data is returned).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Bring `bytes` contiguous bytes at p into L2 with one bulk operation (a hint
// carried out by the asynchronous copy unit; p 16-byte aligned, bytes a
// multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue / wait until the previous kernel's writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace pkv
