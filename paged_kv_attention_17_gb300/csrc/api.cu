// C ABI of the paged KV attention library: host-side validation, the split
// heuristic, workspace sizing, TMA descriptor encoding and kernel launches.
// Every entry point only enqueues work on the caller's stream: no allocation,
// no synchronisation, no host read of device data.
#include <cmath>
#include <cstring>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace pkv {
cudaError_t launch_stage_copy(void* dst, const void* src, int64_t bytes, int num_sms,
                              cudaStream_t stream);
cudaError_t launch_kv_write(const void* k_new, const void* v_new, const int64_t* slots,
                            int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_slots,
                            uint32_t row_bytes, int32_t* flag, int num_sms, cudaStream_t stream);
cudaError_t launch_kv_write_e4m3(const void* k_new, const void* v_new, bool src_bf16,
                                 const int64_t* slots, int64_t num_tokens, void* k_cache,
                                 void* v_cache, int64_t num_slots, uint32_t row_elems,
                                 float k_scale, float v_scale, int32_t* flag, int num_sms,
                                 cudaStream_t stream);
cudaError_t launch_decode(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          ElemType et, int head_dim, bool pdl, cudaStream_t stream);
cudaError_t launch_combine(const AttnArgs& a, ElemType et, int head_dim, cudaStream_t stream);
int decode_rows_per_tile(int group, int max_query_len, bool long_rows);
bool decode_swizzled(ElemType et, int head_dim);
int decode_ctas_per_sm(ElemType et, int head_dim);
bool prefill_supported(int head_dim, ElemType et, int group);
bool prefill_packed_supported(int head_dim, ElemType et, int group);
cudaError_t launch_prefill(const AttnArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int head_dim, ElemType et,
                           cudaStream_t stream);
}  // namespace pkv

using namespace pkv;

namespace {

constexpr int kMinBlocksPerSplit = 8;    // 128 keys
constexpr int kTcMinWindow = 128;        // shortest window the tensor-core prefill takes
constexpr int kCascadeRows = 16;         // rows per tile of the cascade prefix pass

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int device_sms(int device) {
  static int cache[64] = {0};
  if (device < 0 || device >= 64) return 0;
  if (cache[device] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[device] = v;
  }
  return cache[device];
}

int current_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return device_sms(dev);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

// 3-D map over one cache tensor viewed as [num_slots, num_kv_heads, head_dim]
// (innermost first for TMA); a box covers 16 slots (one block) of one kv
// head: the whole row unswizzled (decode kernel), or a 128-byte slice of it
// with the 128B swizzle (prefill tensor-core operands).
bool encode_cache_map(CUtensorMap* map, const void* base, int64_t num_slots, int hkv, int d,
                      ElemType et, bool swizzle128) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t es = et == ElemType::kF32 ? 4 : (et == ElemType::kBf16 ? 2 : 1);
  const CUtensorMapDataType dt = et == ElemType::kF32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : et == ElemType::kBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hkv),
                        static_cast<cuuint64_t>(num_slots)};
  cuuint64_t strides[2] = {d * es, static_cast<cuuint64_t>(hkv) * d * es};
  const cuuint32_t inner = swizzle128 ? static_cast<cuuint32_t>(128 / es) : static_cast<cuuint32_t>(d);
  cuuint32_t box[3] = {inner, 1, static_cast<cuuint32_t>(kBlock)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dt, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D map for the tensor-core decode over a cache viewed as (column within a
// 128-byte slice, slot, slice, KV head): a box is every 128-byte column slice
// of 16 slots' rows of one head, landing slice-major ([slice][16 rows][128
// B], 128B swizzle), so one copy brings a block's K (or V) of one head.  The
// dimensions' strides need not increase: the slot stride is a whole cache
// row, the slice stride 128 bytes, the head stride one head's row.
bool encode_slices_map(CUtensorMap* map, const void* base, int64_t num_slots, int hkv, int d,
                       ElemType et) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t es = et == ElemType::kBf16 ? 2 : 1;
  const CUtensorMapDataType dt = et == ElemType::kBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const cuuint64_t row = static_cast<cuuint64_t>(d) * es;   // one head's row, bytes
  if (row % 128 != 0) return false;
  cuuint64_t dims[4] = {128 / es, static_cast<cuuint64_t>(num_slots), row / 128,
                        static_cast<cuuint64_t>(hkv)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(hkv) * row, 128, row};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(kBlock),
                       static_cast<cuuint32_t>(row / 128), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The decode kernel's maps: rows of several 128-byte slices (bf16, D 128)
// take the 4-D slice map; other tensor-core rows the 128B-swizzled 3-D map
// (one slice per row); the CUDA-core build unswizzled whole rows.
bool encode_decode_maps(CUtensorMap* kmap, CUtensorMap* vmap, const void* k_cache,
                        const void* v_cache, int64_t num_slots, int hkv, int d, ElemType et) {
  const bool sw = decode_swizzled(et, d);
  const int64_t row = static_cast<int64_t>(d) * (et == ElemType::kF32 ? 4 : (et == ElemType::kBf16 ? 2 : 1));
  if (sw && row > 128)
    return encode_slices_map(kmap, k_cache, num_slots, hkv, d, et) &&
           encode_slices_map(vmap, v_cache, num_slots, hkv, d, et);
  return encode_cache_map(kmap, k_cache, num_slots, hkv, d, et, sw) &&
         encode_cache_map(vmap, v_cache, num_slots, hkv, d, et, sw);
}

// 3-D map over q viewed as [num_tokens, num_q_heads, head_dim]: a box is 128
// tokens of one head (or, with heads_per_box = a GQA group, 128 / group tokens
// of the group's heads), 64 columns wide (128 bytes, 128B swizzle).
bool encode_q_map(CUtensorMap* map, const void* q, int64_t num_tokens, int hq, int d,
                  int heads_per_box = 1) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hq),
                        static_cast<cuuint64_t>(num_tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(hq) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(heads_per_box),
                       static_cast<cuuint32_t>(128 / heads_per_box)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool valid_dtype(pkv_dtype dt) { return dt == PKV_F32 || dt == PKV_BF16; }

bool valid_scale(float s) { return std::isfinite(s) && s > 0.f; }

// The split rule for a cache type: as many splits as fit in 7/8 of the
// device's decode CTA slots in one wave (none when the grid is already nearly
// full), every split keeping at least kMinBlocksPerSplit blocks.
int split_rule(int num_seqs, int max_query_len, int max_seq_len, int num_q_heads,
               int num_kv_heads, int head_dim, int device, ElemType et) {
  if (num_seqs < 1 || max_seq_len < 0 || max_query_len < 0 || num_q_heads < 1 ||
      num_kv_heads < 1 || num_q_heads % num_kv_heads != 0)
    return 0;
  const int sms = device_sms(device);
  if (sms <= 0) return 0;
  const int group = num_q_heads / num_kv_heads;
  const int qd = max_query_len < kDecodeMaxQ ? (max_query_len < 1 ? 1 : max_query_len) : kDecodeMaxQ;
  const int R = decode_rows_per_tile(group, qd, false);
  const int64_t units = static_cast<int64_t>(num_seqs) * num_kv_heads * ((group * qd + R - 1) / R);
  // decode CTA slots of the device (two per SM for the tensor-core build);
  // 7/8 of them leave room for the combine and the next launch's prologue
  // (decode at context 8192, 8 KV heads, bf16, 152 SMs: 16 splits take
  // 14 us a call, 32 splits 10.8 us; a second wave at 40 splits 18 us)
  const int64_t capacity = static_cast<int64_t>(sms) * decode_ctas_per_sm(et, head_dim);
  const int64_t target = capacity * 7 / 8;
  int64_t s = target / units;
  if (s <= 1) return 1;
  const int64_t nblk = (static_cast<int64_t>(max_seq_len) + kBlock - 1) / kBlock;
  int64_t by_len = nblk / kMinBlocksPerSplit;
  if (by_len < 1) by_len = 1;
  if (s > by_len) s = by_len;
  if (s > kMaxSplits) s = kMaxSplits;
  return static_cast<int>(s < 1 ? 1 : s);
}

static pkv_status attention(const void* q, const void* k_cache, const void* v_cache, void* out,
                            float* lse_out, const int32_t* query_start_loc,
                            const int32_t* seq_lens, const int32_t* block_table,
                            int max_blocks_per_seq, int num_seqs, int64_t num_tokens,
                            int max_query_len, int max_seq_len, int num_q_heads, int num_kv_heads,
                            int head_dim, int block_size, float softmax_scale, float k_scale,
                            float v_scale, int causal, int window, int num_splits,
                            void* workspace, size_t workspace_bytes, int32_t* error_flag,
                            int64_t num_blocks, ElemType et, void* stream,
                            const void* fuse_k_new = nullptr, const void* fuse_v_new = nullptr,
                            const int64_t* fuse_slots = nullptr) {
  // (fuse_*: the step's new K/V, stored by the decode kernel - bf16 rows
  // quantised with k_scale / v_scale for an E4M3 cache)
  // ---- host-checkable arguments ----
  if (window < 0 || num_seqs < 0 || num_tokens < 0 || num_q_heads < 1 ||
      num_kv_heads < 1 || num_q_heads % num_kv_heads != 0 || num_splits < 0 ||
      num_splits > kMaxSplits || num_blocks < 1 || max_seq_len < 0 || max_query_len < 0 ||
      !std::isfinite(softmax_scale))
    return PKV_ERR_INVALID_ARG;
  if (block_size != kBlock || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0 || num_tokens == 0) return PKV_OK;
  if (max_query_len < 1 || max_blocks_per_seq < 1) return PKV_ERR_INVALID_ARG;
  // a table row of max_blocks_per_seq blocks holds at most 16x that many keys:
  // a larger bound on seq_lens cannot describe a valid batch
  if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * kBlock)
    return PKV_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !out || !query_start_loc || !seq_lens || !block_table)
    return PKV_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(query_start_loc, 4) || !aligned(seq_lens, 4) || !aligned(block_table, 4) ||
      (lse_out && !aligned(lse_out, 4)) || (error_flag && !aligned(error_flag, 4)))
    return PKV_ERR_INVALID_ARG;
  if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
  const int64_t num_slots = num_blocks * kBlock;
  if (num_slots > 0x7FFFFFFFll) return PKV_ERR_UNSUPPORTED;   // TMA row coordinates are int32

  // a window of at least max_seq_len positions excludes no key (a row at
  // position p < max_seq_len sees keys j > p - window, and p - window < 0):
  // it is the plain call, launched as such
  if (window >= max_seq_len) window = 0;
  int splits = num_splits;
  if (splits == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
    // a window bounds the keys a decode row reads: size the split by that span
    const int span = window > 0 && window < max_seq_len - kDecodeMaxQ
                         ? window + kDecodeMaxQ : max_seq_len;
    splits = split_rule(num_seqs, max_query_len, span, num_q_heads, num_kv_heads, head_dim, dev,
                        et);
  }
  if (splits < 1) return PKV_ERR_CUDA;
  const size_t need = pkv_workspace_bytes(num_seqs, num_q_heads, head_dim, splits);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)))
    return PKV_ERR_WORKSPACE;

  const bool bf16 = et == ElemType::kBf16;
  AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = q;
  a.out = out;
  a.lse_out = lse_out;
  a.qsl = query_start_loc;
  a.seq_lens = seq_lens;
  a.block_table = block_table;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.num_tokens = num_tokens;
  a.max_query_len = max_query_len;
  a.max_seq_len = max_seq_len;
  a.hq = num_q_heads;
  a.hkv = num_kv_heads;
  a.group = num_q_heads / num_kv_heads;
  a.scale_log2 = softmax_scale * k_scale * kLog2e;
  a.v_scale = v_scale;
  a.causal = causal ? 1 : 0;
  a.window = window;
  a.num_splits = splits;
  // the tensor-core softmax takes the row max before scaling: positive scales
  // only.  Windows shorter than its 128-key tile run on the CUDA-core tiles:
  // a tensor-core tile would be mostly masked, and rows averaging so few keys
  // have outputs large enough for its bf16 P rounding to show.
  const bool tc_prefill = prefill_supported(head_dim, et, num_q_heads / num_kv_heads) &&
                          softmax_scale > 0.f && (window == 0 || window >= kTcMinWindow);
  // E4M3 caches: decode rows take the register-q tiles, longer requests the
  // CUDA-core tiles of the same kernel
  a.long_rows = tc_prefill ? 0 : (et == ElemType::kE4m3 ? (max_query_len > kDecodeMaxQ) : 1);
  if (need > 0) {
    const size_t rows = static_cast<size_t>(splits) * num_seqs * kDecodeMaxQ * num_q_heads;
    a.ws_o = static_cast<float*>(workspace);
    a.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        align256(rows * head_dim * sizeof(float)));
  }
  a.flag = error_flag;
  a.num_blocks = num_blocks;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  if (fuse_slots != nullptr) {
    // the step's new K/V are stored by the decode kernel (every request is
    // decode-class, checked by the caller)
    a.fuse_write = 1;
    a.k_new = fuse_k_new;
    a.v_new = fuse_v_new;
    a.slots = fuse_slots;
    a.wk_scale = k_scale;
    a.wv_scale = v_scale;
  }

  // the decode kernel's maps (the tensor-core prefill encodes its own below)
  CUtensorMap kmap, vmap;
  if (!encode_decode_maps(&kmap, &vmap, k_cache, v_cache, num_slots, num_kv_heads, head_dim, et))
    return PKV_ERR_CUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // an unsplit launch of a few requests starts the longest first, unless a
  // prefill launch follows: that one starts once every decode CTA has
  // started, which the long CTAs first would delay
  const bool prefill_follows = tc_prefill && max_query_len > kDecodeMaxQ;
  a.lpt = splits == 1 && num_seqs >= 2 && num_seqs <= kLptMaxSeqs && !prefill_follows ? 1 : 0;
  cudaError_t e = launch_decode(a, kmap, vmap, et, head_dim, /*pdl=*/true, st);
  if (e == cudaSuccess && splits > 1) e = launch_combine(a, et, head_dim, st);
  if (e == cudaSuccess && tc_prefill && max_query_len > kDecodeMaxQ) {
    CUtensorMap qmap, kmap_sw, vmap_sw;
    if (num_tokens > 0x7FFFFFFFll || !encode_q_map(&qmap, q, num_tokens, num_q_heads, head_dim) ||
        !encode_cache_map(&kmap_sw, k_cache, num_slots, num_kv_heads, head_dim, et, true) ||
        !encode_cache_map(&vmap_sw, v_cache, num_slots, num_kv_heads, head_dim, et, true))
      return PKV_ERR_CUDA;
    // the decode kernel (and the combine) ahead of it release it only after
    // their own dependency waits: its inputs are complete at launch
    AttnArgs p = a;
    p.defer_wait = 1;
    p.pair_tiles = a.group % 2 != 0 ? 1 : 0;
    e = launch_prefill(p, qmap, kmap_sw, vmap_sw, head_dim, et, st);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

}  // namespace

// The prefix split count: splits of at least four whole 128-key tiles over
// the tensor-core prefix pass's 256-row tiles (tc), or of >= 8 blocks over
// the CUDA-core pass's 16-row tiles, filling 7/8 of the SMs.
static int cascade_split_rule(int64_t num_tokens, int shared_blocks, int num_q_heads,
                              int num_kv_heads, int head_dim, bool tc, int device) {
  if (num_tokens < 1 || shared_blocks < 0 || num_q_heads < 1 || num_kv_heads < 1 ||
      num_q_heads % num_kv_heads != 0)
    return -1;
  if (shared_blocks == 0) return 0;
  const int sms = device_sms(device);
  if (sms <= 0) return -1;
  const int group = num_q_heads / num_kv_heads;
  // tensor-core prefix pass: 256 (token, head) rows per CTA, splits of at
  // least four whole 128-key tiles (fewer tiles per CTA leave its pipeline
  // short of its steady state); CUDA-core pass: 16-row tiles, splits of >= 8
  // blocks
  (void)head_dim;
  const int rows = tc ? 256 : kCascadeRows;
  const int64_t tiles = static_cast<int64_t>(num_kv_heads) * ((group * num_tokens + rows - 1) / rows);
  const int64_t target =
      static_cast<int64_t>(sms) * 7 / 8;
  int64_t s = target / tiles;
  int64_t by_len = tc ? (shared_blocks + 31) / 32 : shared_blocks / kMinBlocksPerSplit;
  if (s > by_len) s = by_len;
  if (s > kMaxSplits - 1) s = kMaxSplits - 1;        // + the own-key partial <= kMaxSplits
  return static_cast<int>(s < 1 ? 1 : s);
}

extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    case PKV_ERR_DEVICE_CHECK: return "PKV_ERR_DEVICE_CHECK";
    case PKV_ERR_DEVICE_TIMEOUT: return "PKV_ERR_DEVICE_TIMEOUT";
  }
  return "PKV_UNKNOWN_STATUS";
}

pkv_status pkv_write(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                     int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_blocks,
                     int block_size, int num_kv_heads, int head_dim, pkv_dtype dtype,
                     int32_t* error_flag, void* stream) {
  if (num_tokens < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 1 || !valid_dtype(dtype))
    return PKV_ERR_INVALID_ARG;
  if (block_size != kBlock) return PKV_ERR_UNSUPPORTED;
  const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * (dtype == PKV_BF16 ? 2 : 4);
  if (row_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8) || (error_flag && !aligned(error_flag, 4)))
    return PKV_ERR_INVALID_ARG;
  const int sms = current_sms();
  if (sms <= 0) return PKV_ERR_CUDA;
  cudaError_t e = launch_kv_write(k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache,
                                  num_blocks * kBlock, static_cast<uint32_t>(row_bytes), error_flag,
                                  sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_stage_inputs(void* dst, const void* src, int64_t nbytes, void* stream) {
  if (nbytes < 0 || nbytes % 16 != 0) return PKV_ERR_INVALID_ARG;
  if (nbytes == 0) return PKV_OK;
  if (!dst || !src || !aligned(dst, 16) || !aligned(src, 16)) return PKV_ERR_INVALID_ARG;
  const int sms = current_sms();
  if (sms <= 0) return PKV_ERR_CUDA;
  cudaError_t e = launch_stage_copy(dst, src, nbytes, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_write_e4m3(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                          int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_blocks,
                          int block_size, int num_kv_heads, int head_dim, pkv_dtype src_dtype,
                          float k_scale, float v_scale, int32_t* error_flag, void* stream) {
  if (num_tokens < 0 || num_blocks < 1 || num_kv_heads < 1 || head_dim < 1 ||
      !valid_dtype(src_dtype) || !valid_scale(k_scale) || !valid_scale(v_scale))
    return PKV_ERR_INVALID_ARG;
  if (block_size != kBlock) return PKV_ERR_UNSUPPORTED;
  const int64_t row_elems = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (row_elems % 16 != 0 || row_elems > 0x7FFFFFFFll) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8) || (error_flag && !aligned(error_flag, 4)))
    return PKV_ERR_INVALID_ARG;
  const int sms = current_sms();
  if (sms <= 0) return PKV_ERR_CUDA;
  cudaError_t e = launch_kv_write_e4m3(k_new, v_new, src_dtype == PKV_BF16, slot_mapping,
                                       num_tokens, k_cache, v_cache, num_blocks * kBlock,
                                       static_cast<uint32_t>(row_elems), k_scale, v_scale,
                                       error_flag, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int pkv_num_splits(int num_seqs, int max_query_len, int max_seq_len, int num_q_heads,
                   int num_kv_heads, int head_dim, int device) {
  // the rule for bf16 and E4M3 caches (an fp32 cache's automatic count may be
  // lower, so a workspace sized from this count always suffices)
  return split_rule(num_seqs, max_query_len, max_seq_len, num_q_heads, num_kv_heads, head_dim,
                    device, ElemType::kBf16);
}

size_t pkv_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int num_splits) {
  if (num_splits <= 1 || num_seqs < 1 || num_q_heads < 1 || head_dim < 1) return 0;
  const size_t rows = static_cast<size_t>(num_splits) * num_seqs * kDecodeMaxQ * num_q_heads;
  return align256(rows * head_dim * sizeof(float)) + align256(rows * sizeof(float));
}

pkv_status pkv_attention_varlen(const void* q, const void* k_cache, const void* v_cache, void* out,
                                float* lse_out, const int32_t* query_start_loc,
                                const int32_t* seq_lens, const int32_t* block_table,
                                int max_blocks_per_seq, int num_seqs, int64_t num_tokens,
                                int max_query_len, int max_seq_len, int num_q_heads,
                                int num_kv_heads, int head_dim, int block_size,
                                float softmax_scale, int causal, int num_splits, void* workspace,
                                size_t workspace_bytes, int32_t* error_flag, int64_t num_blocks,
                                pkv_dtype dtype, void* stream) {
  if (!valid_dtype(dtype)) return PKV_ERR_INVALID_ARG;
  return attention(q, k_cache, v_cache, out, lse_out, query_start_loc, seq_lens, block_table,
                   max_blocks_per_seq, num_seqs, num_tokens, max_query_len, max_seq_len,
                   num_q_heads, num_kv_heads, head_dim, block_size, softmax_scale, 1.f, 1.f,
                   causal, 0, num_splits, workspace, workspace_bytes, error_flag, num_blocks,
                   dtype == PKV_BF16 ? ElemType::kBf16 : ElemType::kF32, stream);
}

pkv_status pkv_write_attention_varlen(
    const void* k_new, const void* v_new, const int64_t* slot_mapping, const void* q,
    void* k_cache, void* v_cache, void* out, float* lse_out, const int32_t* query_start_loc,
    const int32_t* seq_lens, const int32_t* block_table, int max_blocks_per_seq, int num_seqs,
    int64_t num_tokens, int max_query_len, int max_seq_len, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, float softmax_scale, int causal, int num_splits,
    void* workspace, size_t workspace_bytes, int32_t* error_flag, int64_t num_blocks,
    pkv_dtype dtype, void* stream) {
  if (!valid_dtype(dtype)) return PKV_ERR_INVALID_ARG;
  if (num_tokens > 0 && num_seqs > 0) {
    if (!k_new || !v_new || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 8))
      return PKV_ERR_INVALID_ARG;
  }
  const ElemType et = dtype == PKV_BF16 ? ElemType::kBf16 : ElemType::kF32;
  if (max_query_len <= kDecodeMaxQ) {
    // every request decode-class: the write rides in the decode kernel
    return attention(q, k_cache, v_cache, out, lse_out, query_start_loc, seq_lens, block_table,
                     max_blocks_per_seq, num_seqs, num_tokens, max_query_len, max_seq_len,
                     num_q_heads, num_kv_heads, head_dim, block_size, softmax_scale, 1.f, 1.f,
                     causal, 0, num_splits, workspace, workspace_bytes, error_flag, num_blocks,
                     et, stream, k_new, v_new, slot_mapping);
  }
  pkv_status st = pkv_write(k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache, num_blocks,
                            block_size, num_kv_heads, head_dim, dtype, error_flag, stream);
  if (st != PKV_OK) return st;
  return attention(q, k_cache, v_cache, out, lse_out, query_start_loc, seq_lens, block_table,
                   max_blocks_per_seq, num_seqs, num_tokens, max_query_len, max_seq_len,
                   num_q_heads, num_kv_heads, head_dim, block_size, softmax_scale, 1.f, 1.f,
                   causal, 0, num_splits, workspace, workspace_bytes, error_flag, num_blocks, et,
                   stream);
}

pkv_status pkv_write_attention_varlen_e4m3(
    const void* k_new, const void* v_new, const int64_t* slot_mapping, const void* q,
    void* k_cache, void* v_cache, void* out, float* lse_out, const int32_t* query_start_loc,
    const int32_t* seq_lens, const int32_t* block_table, int max_blocks_per_seq, int num_seqs,
    int64_t num_tokens, int max_query_len, int max_seq_len, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, float softmax_scale, float k_scale, float v_scale, int causal,
    int num_splits, void* workspace, size_t workspace_bytes, int32_t* error_flag,
    int64_t num_blocks, void* stream) {
  if (!valid_scale(k_scale) || !valid_scale(v_scale)) return PKV_ERR_INVALID_ARG;
  if (num_tokens > 0 && num_seqs > 0) {
    if (!k_new || !v_new || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 8))
      return PKV_ERR_INVALID_ARG;
  }
  if (max_query_len <= kDecodeMaxQ) {
    return attention(q, k_cache, v_cache, out, lse_out, query_start_loc, seq_lens, block_table,
                     max_blocks_per_seq, num_seqs, num_tokens, max_query_len, max_seq_len,
                     num_q_heads, num_kv_heads, head_dim, block_size, softmax_scale, k_scale,
                     v_scale, causal, 0, num_splits, workspace, workspace_bytes, error_flag,
                     num_blocks, ElemType::kE4m3, stream, k_new, v_new, slot_mapping);
  }
  pkv_status st = pkv_write_e4m3(k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache,
                                 num_blocks, block_size, num_kv_heads, head_dim, PKV_BF16,
                                 k_scale, v_scale, error_flag, stream);
  if (st != PKV_OK) return st;
  return attention(q, k_cache, v_cache, out, lse_out, query_start_loc, seq_lens, block_table,
                   max_blocks_per_seq, num_seqs, num_tokens, max_query_len, max_seq_len,
                   num_q_heads, num_kv_heads, head_dim, block_size, softmax_scale, k_scale,
                   v_scale, causal, 0, num_splits, workspace, workspace_bytes, error_flag,
                   num_blocks, ElemType::kE4m3, stream);
}

pkv_status pkv_attention_varlen_window(const void* q, const void* k_cache, const void* v_cache,
                                       void* out, float* lse_out,
                                       const int32_t* query_start_loc, const int32_t* seq_lens,
                                       const int32_t* block_table, int max_blocks_per_seq,
                                       int num_seqs, int64_t num_tokens, int max_query_len,
                                       int max_seq_len, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, float softmax_scale,
                                       int causal, int window, int num_splits, void* workspace,
                                       size_t workspace_bytes, int32_t* error_flag,
                                       int64_t num_blocks, pkv_dtype dtype, void* stream) {
  if (!valid_dtype(dtype) || window < 0) return PKV_ERR_INVALID_ARG;
  return attention(q, k_cache, v_cache, out, lse_out, query_start_loc, seq_lens, block_table,
                   max_blocks_per_seq, num_seqs, num_tokens, max_query_len, max_seq_len,
                   num_q_heads, num_kv_heads, head_dim, block_size, softmax_scale, 1.f, 1.f,
                   causal, window, num_splits, workspace, workspace_bytes, error_flag,
                   num_blocks, dtype == PKV_BF16 ? ElemType::kBf16 : ElemType::kF32, stream);
}

pkv_status pkv_attention_varlen_e4m3(const void* q, const void* k_cache, const void* v_cache,
                                     void* out, float* lse_out, const int32_t* query_start_loc,
                                     const int32_t* seq_lens, const int32_t* block_table,
                                     int max_blocks_per_seq, int num_seqs, int64_t num_tokens,
                                     int max_query_len, int max_seq_len, int num_q_heads,
                                     int num_kv_heads, int head_dim, int block_size,
                                     float softmax_scale, float k_scale, float v_scale, int causal,
                                     int num_splits, void* workspace, size_t workspace_bytes,
                                     int32_t* error_flag, int64_t num_blocks, void* stream) {
  if (!valid_scale(k_scale) || !valid_scale(v_scale)) return PKV_ERR_INVALID_ARG;
  return attention(q, k_cache, v_cache, out, lse_out, query_start_loc, seq_lens, block_table,
                   max_blocks_per_seq, num_seqs, num_tokens, max_query_len, max_seq_len,
                   num_q_heads, num_kv_heads, head_dim, block_size, softmax_scale, k_scale,
                   v_scale, causal, 0, num_splits, workspace, workspace_bytes, error_flag,
                   num_blocks, ElemType::kE4m3, stream);
}

int pkv_cascade_splits(int64_t num_tokens, int shared_blocks, int num_q_heads, int num_kv_heads,
                       int head_dim, pkv_dtype dtype, int device) {
  if (!valid_dtype(dtype) || num_q_heads < 1 || num_kv_heads < 1 ||
      num_q_heads % num_kv_heads != 0)
    return -1;
  return cascade_split_rule(num_tokens, shared_blocks, num_q_heads, num_kv_heads, head_dim,
                            prefill_packed_supported(head_dim,
                                                     dtype == PKV_BF16 ? ElemType::kBf16
                                                                       : ElemType::kF32,
                                                     num_q_heads / num_kv_heads),
                            device);
}

size_t pkv_cascade_workspace_bytes(int64_t num_tokens, int num_q_heads, int head_dim,
                                   int prefix_splits) {
  if (num_tokens < 1 || num_q_heads < 1 || head_dim < 1 || prefix_splits < 0) return 0;
  const size_t rows = static_cast<size_t>(prefix_splits + 1) * num_tokens * num_q_heads;
  return align256(rows * head_dim * sizeof(float)) + align256(rows * sizeof(float));
}

// The cascade call over a cache of element type et (E4M3: k_scale folded
// into the score scale, v_scale into the output).
static pkv_status cascade_call(const void* q, const void* k_cache, const void* v_cache,
                               void* out, float* lse_out, const int32_t* query_start_loc,
                               const int32_t* suffix_lens, const int32_t* suffix_block_table,
                               int max_blocks_per_seq, const int32_t* shared_block_table,
                               int shared_blocks, int num_seqs, int64_t num_tokens,
                               int max_query_len, int max_suffix_len, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size,
                               float softmax_scale, int prefix_splits, void* workspace,
                               size_t workspace_bytes, int32_t* error_flag, int64_t num_blocks,
                               ElemType et, float k_scale, float v_scale, void* stream) {
  if (num_seqs < 0 || num_tokens < 0 || num_q_heads < 1 ||
      num_kv_heads < 1 || num_q_heads % num_kv_heads != 0 || shared_blocks < 0 ||
      prefix_splits < 0 || prefix_splits > kMaxSplits - 1 || num_blocks < 1 ||
      max_suffix_len < 0 || max_query_len < 0 || !std::isfinite(softmax_scale))
    return PKV_ERR_INVALID_ARG;
  if (block_size != kBlock || (head_dim != 64 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0 || num_tokens == 0) return PKV_OK;
  if (max_query_len < 1 || max_blocks_per_seq < 1) return PKV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_suffix_len) > static_cast<int64_t>(max_blocks_per_seq) * kBlock)
    return PKV_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !out || !query_start_loc || !suffix_lens ||
      !suffix_block_table || (shared_blocks > 0 && !shared_block_table))
    return PKV_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(query_start_loc, 4) || !aligned(suffix_lens, 4) ||
      !aligned(suffix_block_table, 4) || (shared_block_table && !aligned(shared_block_table, 4)) ||
      (lse_out && !aligned(lse_out, 4)) || (error_flag && !aligned(error_flag, 4)))
    return PKV_ERR_INVALID_ARG;
  if (num_seqs > 65535 || num_tokens > 0x7FFFFFFFll) return PKV_ERR_UNSUPPORTED;
  const int64_t num_slots = num_blocks * kBlock;
  if (num_slots > 0x7FFFFFFFll || static_cast<int64_t>(shared_blocks) * kBlock > 0x7FFFFFFFll)
    return PKV_ERR_UNSUPPORTED;
  int S = prefix_splits;
  if (shared_blocks == 0) {
    S = 0;
  } else if (S == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
    S = cascade_split_rule(num_tokens, shared_blocks, num_q_heads, num_kv_heads, head_dim,
                           prefill_packed_supported(head_dim, et,
                                                    num_q_heads / num_kv_heads),
                           dev);
    if (S < 1) return PKV_ERR_CUDA;
  }
  const size_t need = pkv_cascade_workspace_bytes(num_tokens, num_q_heads, head_dim, S);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256))
    return PKV_ERR_WORKSPACE;
  const size_t rows = static_cast<size_t>(S + 1) * num_tokens * num_q_heads;

  AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = q;
  a.out = out;
  a.lse_out = lse_out;
  a.qsl = query_start_loc;
  a.num_seqs = num_seqs;
  a.num_tokens = num_tokens;
  a.hq = num_q_heads;
  a.hkv = num_kv_heads;
  a.group = num_q_heads / num_kv_heads;
  a.scale_log2 = softmax_scale * kLog2e * (et == ElemType::kE4m3 ? k_scale : 1.f);
  a.v_scale = et == ElemType::kE4m3 ? v_scale : 1.f;
  a.ws_o = static_cast<float*>(workspace);
  a.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                      align256(rows * head_dim * sizeof(float)));
  a.flag = error_flag;
  a.num_blocks = num_blocks;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  CUtensorMap kmap, vmap;
  if (!encode_decode_maps(&kmap, &vmap, k_cache, v_cache, num_slots, num_kv_heads, head_dim, et))
    return PKV_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  // tensor cores for the prefix pass (bf16, head_dim 128, a GQA group that
  // divides 128 rows, positive scale); the CUDA-core tiles otherwise
  const bool tc = prefill_packed_supported(head_dim, et,
                                           num_q_heads / num_kv_heads) &&
                  softmax_scale > 0.f;
  // Two independent passes write disjoint partials; the merge reads both.
  // With the tensor-core prefix pass the own-key pass goes first and the
  // prefix pass behind it defers its dependency wait to its CTAs' exits (its
  // inputs are complete once the own-key CTAs release it), so the prefix
  // tiles run in the own-key grid's tail; the CUDA-core prefix pass runs
  // first, in stream order.
  auto own_keys = [&]() -> cudaError_t {
    // 2. each request over its own keys (causal): partial S
    AttnArgs u = a;
    u.seq_lens = suffix_lens;
    u.block_table = suffix_block_table;
    u.max_blocks_per_seq = max_blocks_per_seq;
    u.num_seqs = num_seqs;
    u.max_query_len = max_query_len;
    u.max_seq_len = max_suffix_len;
    u.causal = 1;
    u.num_splits = 1;
    u.long_rows = max_query_len > kDecodeMaxQ ? 1 : 0;
    u.cascade = 2;
    u.cascade_slot = S;
    // (no longest-first order when the deferred prefix pass follows it)
    u.lpt = !tc && num_seqs >= 2 && num_seqs <= kLptMaxSeqs ? 1 : 0;
    return launch_decode(u, kmap, vmap, et, head_dim, /*pdl=*/true, st);
  };
  if (tc) e = own_keys();
  if (e == cudaSuccess && S > 0) {
    // 1. every row over the shared prefix, split S ways: partials 0..S-1
    AttnArgs p = a;
    p.block_table = shared_block_table;
    p.max_blocks_per_seq = shared_blocks;
    p.num_seqs = 1;
    p.max_query_len = static_cast<int>(num_tokens);
    p.max_seq_len = shared_blocks * kBlock;
    p.causal = 0;
    p.num_splits = S;
    p.long_rows = 1;
    p.cascade = 1;
    p.prefix_len = shared_blocks * kBlock;
    p.defer_wait = tc ? 1 : 0;
    if (tc) {
      CUtensorMap qmap, kmap_sw, vmap_sw;
      if (!encode_q_map(&qmap, q, num_tokens, num_q_heads, head_dim, p.group) ||
          !encode_cache_map(&kmap_sw, k_cache, num_slots, num_kv_heads, head_dim, et, true) ||
          !encode_cache_map(&vmap_sw, v_cache, num_slots, num_kv_heads, head_dim, et, true))
        return PKV_ERR_CUDA;
      e = launch_prefill(p, qmap, kmap_sw, vmap_sw, head_dim, et, st);
    } else {
      e = launch_decode(p, kmap, vmap, et, head_dim, /*pdl=*/true, st);
    }
  }
  if (e == cudaSuccess && !tc) e = own_keys();
  if (e == cudaSuccess) {
    // 3. merge the S + 1 partials of every row
    AttnArgs c = a;
    c.num_splits = S + 1;
    c.cascade = 3;
    e = launch_combine(c, et, head_dim, st);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

pkv_status pkv_cascade_attention(const void* q, const void* k_cache, const void* v_cache,
                                 void* out, float* lse_out, const int32_t* query_start_loc,
                                 const int32_t* suffix_lens, const int32_t* suffix_block_table,
                                 int max_blocks_per_seq, const int32_t* shared_block_table,
                                 int shared_blocks, int num_seqs, int64_t num_tokens,
                                 int max_query_len, int max_suffix_len, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size,
                                 float softmax_scale, int prefix_splits, void* workspace,
                                 size_t workspace_bytes, int32_t* error_flag, int64_t num_blocks,
                                 pkv_dtype dtype, void* stream) {
  if (!valid_dtype(dtype)) return PKV_ERR_INVALID_ARG;
  return cascade_call(q, k_cache, v_cache, out, lse_out, query_start_loc, suffix_lens,
                      suffix_block_table, max_blocks_per_seq, shared_block_table, shared_blocks,
                      num_seqs, num_tokens, max_query_len, max_suffix_len, num_q_heads,
                      num_kv_heads, head_dim, block_size, softmax_scale, prefix_splits, workspace,
                      workspace_bytes, error_flag, num_blocks,
                      dtype == PKV_BF16 ? ElemType::kBf16 : ElemType::kF32, 1.f, 1.f, stream);
}

pkv_status pkv_cascade_attention_e4m3(
    const void* q, const void* k_cache, const void* v_cache, void* out, float* lse_out,
    const int32_t* query_start_loc, const int32_t* suffix_lens, const int32_t* suffix_block_table,
    int max_blocks_per_seq, const int32_t* shared_block_table, int shared_blocks, int num_seqs,
    int64_t num_tokens, int max_query_len, int max_suffix_len, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, float softmax_scale, float k_scale, float v_scale,
    int prefix_splits, void* workspace, size_t workspace_bytes, int32_t* error_flag,
    int64_t num_blocks, void* stream) {
  if (!valid_scale(k_scale) || !valid_scale(v_scale)) return PKV_ERR_INVALID_ARG;
  return cascade_call(q, k_cache, v_cache, out, lse_out, query_start_loc, suffix_lens,
                      suffix_block_table, max_blocks_per_seq, shared_block_table, shared_blocks,
                      num_seqs, num_tokens, max_query_len, max_suffix_len, num_q_heads,
                      num_kv_heads, head_dim, block_size, softmax_scale, prefix_splits, workspace,
                      workspace_bytes, error_flag, num_blocks, ElemType::kE4m3, k_scale, v_scale,
                      stream);
}

pkv_status pkv_attention_varlen_e4m3_window(
    const void* q, const void* k_cache, const void* v_cache, void* out, float* lse_out,
    const int32_t* query_start_loc, const int32_t* seq_lens, const int32_t* block_table,
    int max_blocks_per_seq, int num_seqs, int64_t num_tokens, int max_query_len, int max_seq_len,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, float softmax_scale,
    float k_scale, float v_scale, int causal, int window, int num_splits, void* workspace,
    size_t workspace_bytes, int32_t* error_flag, int64_t num_blocks, void* stream) {
  if (!valid_scale(k_scale) || !valid_scale(v_scale) || window < 0) return PKV_ERR_INVALID_ARG;
  return attention(q, k_cache, v_cache, out, lse_out, query_start_loc, seq_lens, block_table,
                   max_blocks_per_seq, num_seqs, num_tokens, max_query_len, max_seq_len,
                   num_q_heads, num_kv_heads, head_dim, block_size, softmax_scale, k_scale,
                   v_scale, causal, window, num_splits, workspace, workspace_bytes, error_flag,
                   num_blocks, ElemType::kE4m3, stream);
}

}  // extern "C"
