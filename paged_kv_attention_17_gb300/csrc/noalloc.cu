// Attention entry point for callers that cannot allocate device memory.
//
// pkv_attention_varlen needs a caller-provided workspace for the split-KV
// partials.  Some callers have no way to provide one: a host program written
// in plain C whose device memory belongs to another runtime's caching
// allocator (raw cudaMalloc/cudaFree calls would fragment that pool, and
// cudaFree can synchronise the whole device), or code on a latency-critical
// path that must never block in the allocator.  This entry point serves them
// from a fixed scratch array compiled into the library instead.
//
// The array is a file-scope __device__ variable of kStaticWorkspaceBytes
// (8 MiB): every GPU that loads the library holds it until the process exits.
// Its name is only a host-side stand-in in host code, so the first call on
// each device looks up the array's device address with cudaGetSymbolAddress
// (with that device current) and every call passes that address to the
// kernels.  Make that first call on a device before any stream capture.
// All calls on a device share the one array: calls whose kernels overlap on
// the GPU (e.g. on two streams) race on it and must be serialised by the
// caller.  Nothing in it has to start at zero: every partial the combine
// kernel reads is written earlier in the same call by the decode kernel.
// The per-device address cache is atomic, so host threads may make their
// first calls on a device concurrently (each stores the same address).
#include <atomic>

#include "common.cuh"

namespace {

constexpr size_t kStaticWorkspaceBytes = static_cast<size_t>(8) << 20;

__device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

// device address of the array, per device (relaxed atomics: every thread that
// resolves it stores the same value)
std::atomic<void*> g_workspace_ptr[64];

}  // namespace

extern "C" pkv_status pkv_attention_varlen_noalloc(
    const void* q, const void* k_cache, const void* v_cache, void* out, float* lse_out,
    const int32_t* query_start_loc, const int32_t* seq_lens, const int32_t* block_table,
    int max_blocks_per_seq, int num_seqs, int64_t num_tokens, int max_query_len, int max_seq_len,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, float softmax_scale,
    int causal, int num_splits, int32_t* error_flag, int64_t num_blocks, pkv_dtype dtype,
    void* stream) {
  if (num_splits < 0 || num_splits > pkv::kMaxSplits) return PKV_ERR_INVALID_ARG;
  if (num_seqs <= 0 || num_tokens <= 0)
    return pkv_attention_varlen(q, k_cache, v_cache, out, lse_out, query_start_loc, seq_lens,
                                block_table, max_blocks_per_seq, num_seqs, num_tokens,
                                max_query_len, max_seq_len, num_q_heads, num_kv_heads, head_dim,
                                block_size, softmax_scale, causal, num_splits, nullptr, 0,
                                error_flag, num_blocks, dtype, stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  int splits = num_splits;
  if (splits == 0) {
    // automatic: the heuristic's count, lowered until the partials fit the
    // array (the split count never changes the result; one split needs none)
    splits = pkv_num_splits(num_seqs, max_query_len, max_seq_len, num_q_heads, num_kv_heads,
                            head_dim, dev);
    if (splits < 1) return PKV_ERR_INVALID_ARG;
    while (splits > 1 &&
           pkv_workspace_bytes(num_seqs, num_q_heads, head_dim, splits) > kStaticWorkspaceBytes)
      --splits;
  }
  // an explicit split count whose partials do not fit is rejected
  if (pkv_workspace_bytes(num_seqs, num_q_heads, head_dim, splits) > kStaticWorkspaceBytes)
    return PKV_ERR_WORKSPACE;
  void* ws = g_workspace_ptr[dev].load(std::memory_order_relaxed);
  if (ws == nullptr) {
    if (cudaGetSymbolAddress(&ws, g_static_workspace) != cudaSuccess || ws == nullptr) {
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
    g_workspace_ptr[dev].store(ws, std::memory_order_relaxed);
  }
  return pkv_attention_varlen(q, k_cache, v_cache, out, lse_out, query_start_loc, seq_lens,
                              block_table, max_blocks_per_seq, num_seqs, num_tokens, max_query_len,
                              max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size,
                              softmax_scale, causal, splits, ws,
                              kStaticWorkspaceBytes, error_flag, num_blocks, dtype, stream);
}
