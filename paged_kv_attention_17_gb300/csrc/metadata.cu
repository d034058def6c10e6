// Host-side flat-batch metadata of one step (no device code).
//
// "Model execution", section "Flattening a step": the runner concatenates the
// scheduled tokens of all requests into one flat batch and hands attention
// query_start_loc (cumulative token offsets), seq_lens (context after this
// step), block_table (physical block ids per request) and slot_mapping (the
// physical slot block_id * block_size + offset of each new token, which sits
// at position computed + k of its request).  A C host builds these arrays
// here before copying them to the device.
#include <cstring>

#include "pkv.h"

extern "C" pkv_status pkv_build_metadata(int num_seqs, const int32_t* computed,
                                         const int32_t* scheduled, const int32_t* block_offsets,
                                         const int32_t* block_ids, int block_size,
                                         int max_blocks_per_seq, int64_t num_tokens,
                                         int32_t* query_start_loc, int32_t* seq_lens,
                                         int32_t* block_table, int64_t* slot_mapping,
                                         int64_t* positions, int32_t* max_query_len,
                                         int32_t* max_seq_len) {
  if (num_seqs < 0 || block_size < 1 || max_blocks_per_seq < 1 || num_tokens < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs > 0 && (!computed || !scheduled || !block_offsets || !query_start_loc ||
                       !seq_lens || !block_table))
    return PKV_ERR_INVALID_ARG;
  if (num_tokens > 0 && !slot_mapping) return PKV_ERR_INVALID_ARG;
  // ---- validate everything before writing anything ----
  int64_t total = 0;
  if (num_seqs > 0 && block_offsets[0] != 0) return PKV_ERR_INVALID_ARG;
  for (int r = 0; r < num_seqs; ++r) {
    const int64_t c = computed[r], s = scheduled[r];
    const int64_t nb = static_cast<int64_t>(block_offsets[r + 1]) - block_offsets[r];
    if (c < 0 || s < 0 || nb < 0 || nb > max_blocks_per_seq) return PKV_ERR_INVALID_ARG;
    if (c + s > 0x7FFFFFFFll) return PKV_ERR_INVALID_ARG;
    if ((c + s + block_size - 1) / block_size > nb) return PKV_ERR_INVALID_ARG;   // blocks cover the context
    if (nb > 0 && !block_ids) return PKV_ERR_INVALID_ARG;
    for (int64_t b = block_offsets[r]; b < block_offsets[r + 1]; ++b)
      if (block_ids[b] < 0) return PKV_ERR_INVALID_ARG;
    total += s;
  }
  if (total != num_tokens || total > 0x7FFFFFFFll) return PKV_ERR_INVALID_ARG;
  // ---- fill ----
  int32_t mq = 0, ms = 0;
  int64_t t = 0;
  if (num_seqs > 0) query_start_loc[0] = 0;
  for (int r = 0; r < num_seqs; ++r) {
    const int32_t c = computed[r], s = scheduled[r];
    const int32_t* blocks = block_ids ? block_ids + block_offsets[r] : nullptr;
    const int nb = block_offsets[r + 1] - block_offsets[r];
    int32_t* row = block_table + static_cast<int64_t>(r) * max_blocks_per_seq;
    std::memset(row, 0, sizeof(int32_t) * max_blocks_per_seq);
    if (nb > 0) std::memcpy(row, blocks, sizeof(int32_t) * nb);
    seq_lens[r] = c + s;
    for (int32_t k = 0; k < s; ++k, ++t) {
      const int64_t pos = static_cast<int64_t>(c) + k;
      slot_mapping[t] = static_cast<int64_t>(blocks[pos / block_size]) * block_size + pos % block_size;
      if (positions) positions[t] = pos;
    }
    query_start_loc[r + 1] = static_cast<int32_t>(t);
    mq = s > mq ? s : mq;
    ms = c + s > ms ? c + s : ms;
  }
  if (max_query_len) *max_query_len = mq;
  if (max_seq_len) *max_seq_len = ms;
  return PKV_OK;
}
