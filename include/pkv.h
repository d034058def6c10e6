/*
 * pkv.h - C ABI of the paged KV attention library for GB300 (sm_103a).
 *
 * What it computes.  Exact softmax attention of every new token of a flat,
 * variable-length serving batch over its request's context, where the context
 * K/V live in a paged cache of 16-token blocks named by per-request block
 * tables, plus the slot-mapped write of the new tokens' K/V into that cache.
 * The batch description follows "Model execution" (vLLM internals notes),
 * section "Flattening a step": query_start_loc, seq_lens, block_table and
 * slot_mapping; the method follows "Inside the engine: kernels, CUDA graphs
 * and the life of a request", sections "Never materialise the TxT matrix"
 * (online softmax), "Prefill has a full grid; decode at batch 1 has almost
 * none" (split-KV partials merged by a second reduction kernel) and
 * "Attention over a block table, not a contiguous tensor" (16-token blocks
 * gathered through a block table).
 *
 * Conventions for every entry point.
 *   - Device pointers are CUDA device addresses on the current device; the
 *     caller allocates and owns every buffer.  The library never allocates,
 *     frees or synchronises: each call validates its host arguments, enqueues
 *     kernels on `stream` (a cudaStream_t; NULL = legacy default stream) and
 *     returns.  All pointers to tensors must be 16-byte aligned.
 *   - Host-checkable errors return a status and enqueue nothing.
 *   - Data-dependent errors (a block ID or slot outside the cache, a request
 *     with more new tokens than context, a query_start_loc that is not a
 *     valid prefix sum) cannot be seen on the host without a sync.  Kernels
 *     skip the offending access, never trap, and OR a PKV_FLAG_* bit into
 *     *error_flag (a device int32 the caller zeroes and reads later) when
 *     error_flag is non-NULL.  Outputs of the affected rows are unspecified.
 *   - Tensors are dense and row-major in the shapes given; the KV cache is
 *     two tensors (K and V), each [num_blocks, block_size, num_kv_heads,
 *     head_dim], i.e. [num_slots, num_kv_heads, head_dim] with
 *     slot = block_id * block_size + offset.
 *   - Supported: block_size 16; head_dim 64 or 128; num_q_heads a multiple of
 *     num_kv_heads; dtype PKV_F32 or PKV_BF16 (same dtype for Q, K, V and
 *     the output), or an 8-bit E4M3 cache with bf16 Q and output through the
 *     _e4m3 entry points.  Arithmetic is fp32 with fp32 accumulation (the
 *     tensor-core prefill rounds P to bf16 for its P.V product).
 *
 * Entry points: pkv_write / pkv_write_e4m3 (slot-mapped write), pkv_stage_inputs
 * (a step's packed inputs copied to the device), pkv_num_splits
 * and pkv_workspace_bytes (split-KV sizing), pkv_attention_varlen and its
 * variants _window (sliding window), _e4m3 (8-bit cache), _e4m3_window and
 * _noalloc (no caller workspace), pkv_write_attention_varlen / _e4m3 (write
 * and attend in one call, the write folded into the decode kernel for decode
 * steps), pkv_cascade_splits / pkv_cascade_workspace_bytes /
 * pkv_cascade_attention / _e4m3 (requests sharing a block-aligned prefix),
 * pkv_build_metadata (the step's flat-batch metadata, host only) and
 * pkv_status_string.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad size or count */
    PKV_ERR_UNSUPPORTED = 2,    /* valid request this build does not implement */
    PKV_ERR_WORKSPACE = 3,      /* workspace missing or smaller than required */
    PKV_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
    PKV_ERR_DEVICE_CHECK = 5,   /* reserved for callers mapping *error_flag */
    PKV_ERR_DEVICE_TIMEOUT = 6  /* reserved for callers mapping *error_flag */
} pkv_status;

typedef enum { PKV_F32 = 0, PKV_BF16 = 1 } pkv_dtype;

/* Bits a kernel ORs into *error_flag. */
#define PKV_FLAG_BAD_BLOCK   1  /* block_table entry outside [0, num_blocks) */
#define PKV_FLAG_BAD_SLOT    2  /* slot_mapping entry >= num_blocks * block_size */
#define PKV_FLAG_BAD_LENGTHS 4  /* q_len > seq_len, q_len > max_query_len,
                                   seq_len > max_blocks_per_seq * block_size, or
                                   query_start_loc not a prefix sum ending at
                                   num_tokens */
#define PKV_FLAG_TIMEOUT     8  /* a pipeline wait gave up (about 2 s bound) */

/* Requests with at most this many new tokens take the split-KV decode path;
 * longer ones take the tiled prefill path. */
#define PKV_DECODE_MAX_QLEN 4

/*
 * pkv_write - store each new token's K and V at its slot.
 *
 * "Model execution", section "Flattening a step": slot_mapping gives, per new
 * token, the physical slot block_id * block_size + offset its K and V go to;
 * "Inside the engine ...", section "Attention over a block table ...": the
 * KV-write kernel scatters into non-contiguous blocks.
 *
 *   k_new, v_new   device, [num_tokens, num_kv_heads, head_dim], dtype.
 *   slot_mapping   device int64 [num_tokens]; a negative slot (a padding
 *                  token) is skipped; a slot >= num_blocks * block_size is
 *                  skipped and flagged PKV_FLAG_BAD_SLOT.
 *   k_cache, v_cache  device, [num_blocks, block_size, num_kv_heads, head_dim].
 *   error_flag     device int32 or NULL.
 * Slots not named by slot_mapping keep their contents.  Two tokens naming
 * the same slot leave either one's row there (unspecified which).
 * num_tokens == 0 is a no-op returning PKV_OK.
 */
pkv_status pkv_write(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                     int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_blocks,
                     int block_size, int num_kv_heads, int head_dim, pkv_dtype dtype,
                     int32_t* error_flag, void* stream);

/*
 * pkv_write_e4m3 - pkv_write into an 8-bit E4M3 cache.
 *
 * "Model execution", section "Where it breaks" (an FP8 KV cache is a backend
 * feature) and "Anatomy of a serving engine", the FP8-cache exercise of its
 * KV-memory arithmetic: the cache holds one byte per element.  The pages fix
 * no format; this library reads it as E4M3 (sign, 4 exponent bits with bias
 * 7, 3 mantissa bits; subnormals m/8 * 2^-6; largest finite 448; no
 * infinities; S.1111.111 is NaN) with one fp32 scale per cache tensor: a
 * stored code c stands for scale * value(c).  Element x is stored as the
 * nearest code (ties to the even mantissa, magnitudes beyond 448 saturate to
 * 448) of x / scale, the division correctly rounded in fp32.
 *
 *   k_new, v_new   device, [num_tokens, num_kv_heads, head_dim], src_dtype
 *                  (PKV_F32 or PKV_BF16).
 *   k_cache, v_cache  device uint8 [num_blocks, block_size, num_kv_heads,
 *                  head_dim].
 *   k_scale, v_scale  finite, > 0.
 *   num_kv_heads * head_dim must be a multiple of 16 (else
 *   PKV_ERR_UNSUPPORTED).  slot_mapping, error_flag and the rest as pkv_write.
 */
pkv_status pkv_write_e4m3(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                          int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_blocks,
                          int block_size, int num_kv_heads, int head_dim, pkv_dtype src_dtype,
                          float k_scale, float v_scale, int32_t* error_flag, void* stream);

/*
 * pkv_stage_inputs - copy a step's packed inputs into device memory.
 *
 * "Inside the engine: kernels, CUDA graphs and the life of a request",
 * section on CUDA graphs (a captured step runs on fixed buffers, so each
 * step's inputs are copied into them first), and "Model execution", section
 * "Flattening a step" (the step's inputs are copied to the device
 * asynchronously; nothing waits for them on the host).  One kernel copies
 * nbytes from src to dst with the device's own loads: src may be pinned host
 * memory mapped into the device's address space (the loads cross the host
 * link) or device memory.  The kernel lets the next kernel on the stream
 * launch at once, and that kernel's dependency wait returns only after the
 * copy is complete, so a step's attention kernels overlap their set-up with
 * the transfer.  It starts copying after earlier work on the stream ends.
 *
 *   dst     device memory, 16-byte aligned, nbytes long.
 *   src     device-accessible memory, 16-byte aligned, nbytes long, not
 *           overlapping dst.
 *   nbytes  a multiple of 16 (else PKV_ERR_INVALID_ARG); 0 is a no-op.
 * Returns PKV_OK, PKV_ERR_INVALID_ARG (null or misaligned pointer, bad size)
 * or PKV_ERR_CUDA (launch failure).
 */
pkv_status pkv_stage_inputs(void* dst, const void* src, int64_t nbytes, void* stream);

/*
 * pkv_num_splits - how many KV splits the decode path should use.
 *
 * "Inside the engine ...", section "Prefill has a full grid; decode at batch 1
 * has almost none": split the KV axis when there are too few query rows to
 * fill the GPU; at high batch the grid is already full and the split is
 * turned off.  With U = num_seqs x num_kv_heads x row tiles of decode work
 * units and C the decode CTAs device `device` holds at once (SM count x
 * resident CTAs per SM), T = floor(7 C / 8): max(1, floor(T / U)), so one
 * wave of split CTAs leaves some SMs free for the combine kernel and the next
 * launch to start early (1 once the grid is nearly full);
 * never fewer than 8 blocks (128 keys) per split nor more than 64 splits.
 * Returns 0 for invalid arguments or device.
 */
int pkv_num_splits(int num_seqs, int max_query_len, int max_seq_len, int num_q_heads,
                   int num_kv_heads, int head_dim, int device);

/*
 * pkv_workspace_bytes - device workspace pkv_attention_varlen needs.
 *
 * Holds the split-KV partials of the decode path: for every split, request,
 * decode row (< PKV_DECODE_MAX_QLEN) and query head, an fp32 partial output
 * [head_dim] and its log-sum-exp.  0 when num_splits <= 1.
 */
size_t pkv_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int num_splits);

/*
 * pkv_attention_varlen - attention of a flat varlen batch over the paged cache.
 *
 * For request r (0 <= r < num_seqs), n = query_start_loc[r+1] -
 * query_start_loc[r] new tokens occupy rows query_start_loc[r]..+n-1 of q and
 * out, and L = seq_lens[r] is its context after this step (its new tokens
 * already written, e.g. by pkv_write).  New token i is at position
 * p = L - n + i; with causal != 0 it attends keys 0..p, otherwise all L keys.
 * Key j of request r is cache row block_table[r * max_blocks_per_seq + j/16]
 * * 16 + j % 16, kv head h / (num_q_heads / num_kv_heads) for query head h.
 *   out[t, h, :] = sum_j softmax_j(softmax_scale * q[t,h,:] . k_j) v_j
 * computed as an online softmax over key tiles ("Never materialise the TxT
 * matrix"); requests with n <= PKV_DECODE_MAX_QLEN take the split-KV decode
 * kernel (partials merged by a log-sum-exp combine kernel when num_splits >
 * 1), longer ones the tiled prefill kernel: on tensor cores for bf16 at
 * head_dim 64 or 128 (two query heads of a KV head per CTA, or with an odd
 * GQA group two query tiles of one head; an E4M3 cache through
 * pkv_attention_varlen_e4m3 at head_dim 128), else on the decode kernel's
 * CUDA-core 16-row tiles.
 *
 *   q, out            device [num_tokens, num_q_heads, head_dim], dtype.
 *   lse_out           device fp32 [num_tokens, num_q_heads] or NULL: natural-log
 *                     log-sum-exp of each row's scaled scores (-inf if the row
 *                     sees no key).
 *   k_cache, v_cache  device [num_blocks, 16, num_kv_heads, head_dim], dtype.
 *   query_start_loc   device int32 [num_seqs + 1], nondecreasing, [0] = 0,
 *                     [num_seqs] <= num_tokens (rows of q/out past it, such
 *                     as a captured graph's padding rows, are neither read
 *                     nor written).
 *   seq_lens          device int32 [num_seqs].
 *   block_table       device int32 [num_seqs, max_blocks_per_seq].
 *   max_query_len     host: >= every n (bounds the prefill grid).
 *   max_seq_len       host: >= every L, <= 16 * max_blocks_per_seq (sizes the
 *                     split heuristic and the pre-launch L2 warm-up; a larger
 *                     value returns PKV_ERR_INVALID_ARG).  A seq_len beyond the
 *                     table row is flagged on the device (PKV_FLAG_BAD_LENGTHS).
 *   num_splits        0 = pkv_num_splits(...); else 1..64.
 *   workspace         device, >= pkv_workspace_bytes(num_seqs, num_q_heads,
 *                     head_dim, splits) bytes, 256-byte aligned; may be NULL
 *                     when that is 0.  Contents need no initialisation.
 * Rows of requests with n == 0 are absent; a request with L == 0 and n == 0
 * is a no-op.  Returns PKV_OK once the kernels are enqueued.
 */
pkv_status pkv_attention_varlen(const void* q, const void* k_cache, const void* v_cache,
                                void* out, float* lse_out, const int32_t* query_start_loc,
                                const int32_t* seq_lens, const int32_t* block_table,
                                int max_blocks_per_seq, int num_seqs, int64_t num_tokens,
                                int max_query_len, int max_seq_len, int num_q_heads,
                                int num_kv_heads, int head_dim, int block_size,
                                float softmax_scale, int causal, int num_splits,
                                void* workspace, size_t workspace_bytes, int32_t* error_flag,
                                int64_t num_blocks, pkv_dtype dtype, void* stream);

/*
 * pkv_write_attention_varlen - pkv_write then pkv_attention_varlen, as one
 * call.
 *
 * The same two steps ("Model execution", section "Flattening a step": the
 * new tokens' K/V go to their slots, then attention reads the cache).  When
 * every request is decode-class (max_query_len <= PKV_DECODE_MAX_QLEN) the
 * write rides in the decode kernel: each CTA stores the new-token rows it is
 * about to read (a bounded barrier orders the stores before its TMA loads of
 * them), so the step is one launch fewer.  Otherwise pkv_write runs first.
 *   k_new, v_new, slot_mapping: as pkv_write (q's dtype).  The other
 *   arguments as pkv_attention_varlen.  On the fused path only the tokens of
 *   rows below query_start_loc[num_seqs] are stored (padding rows carry slot
 *   -1 anyway); a slot past the cache is skipped and flagged
 *   PKV_FLAG_BAD_SLOT.  The cache contents after the call are those of the
 *   two separate calls.
 */
pkv_status pkv_write_attention_varlen(
    const void* k_new, const void* v_new, const int64_t* slot_mapping, const void* q,
    void* k_cache, void* v_cache, void* out, float* lse_out, const int32_t* query_start_loc,
    const int32_t* seq_lens, const int32_t* block_table, int max_blocks_per_seq, int num_seqs,
    int64_t num_tokens, int max_query_len, int max_seq_len, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, float softmax_scale, int causal, int num_splits,
    void* workspace, size_t workspace_bytes, int32_t* error_flag, int64_t num_blocks,
    pkv_dtype dtype, void* stream);

/*
 * pkv_attention_varlen_window - pkv_attention_varlen with a sliding window.
 *
 * "Anatomy of a serving engine", section "Where it breaks": sliding-window
 * attention is a variant some backends support; the pages give no
 * definition.  Reading taken: with window W > 0 the new token at position
 * p = L - n + i sees only keys j with p - W < j (the W most recent
 * positions, itself included), on top of the causal limit j <= p (or j < L
 * with causal == 0).  window == 0 is pkv_attention_varlen exactly, and so is
 * any window >= max_seq_len (it excludes no key; the call runs as window 0).  Key
 * blocks wholly below a tile's window start are not read, and the automatic
 * split count is sized for a context of window + PKV_DECODE_MAX_QLEN keys.
 * Windows shorter than 128 keys run every request on the split-KV kernel's
 * CUDA-core tiles (fp32 P) instead of the tensor-core prefill.
 *   window  >= 0 (negative: PKV_ERR_INVALID_ARG).
 * Everything else as pkv_attention_varlen.
 */
pkv_status pkv_attention_varlen_window(const void* q, const void* k_cache, const void* v_cache,
                                       void* out, float* lse_out,
                                       const int32_t* query_start_loc, const int32_t* seq_lens,
                                       const int32_t* block_table, int max_blocks_per_seq,
                                       int num_seqs, int64_t num_tokens, int max_query_len,
                                       int max_seq_len, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, float softmax_scale,
                                       int causal, int window, int num_splits, void* workspace,
                                       size_t workspace_bytes, int32_t* error_flag,
                                       int64_t num_blocks, pkv_dtype dtype, void* stream);

/*
 * pkv_attention_varlen_e4m3 - pkv_attention_varlen over an E4M3 cache.
 *
 * The cache format of pkv_write_e4m3: key j stands for k_scale * value(code),
 * value j for v_scale * value(code), so
 *   out[t, h, :] = v_scale * sum_j softmax_j(softmax_scale * k_scale *
 *                  q[t,h,:] . value(K code_j)) value(V code_j)
 * (lse_out: the natural-log log-sum-exp of those scaled scores).  At head_dim
 * 128 the contractions run on tensor cores with fp32 accumulation and P
 * rounded to f16 for P.V.  V codes are widened exactly to f16.  K codes are
 * widened too, with q scaled by a power of two into f16, in split decode
 * launches without a window (the latency-bound form, which fetches each
 * split's first block speculatively) and in tiles of 16 rows; otherwise they
 * enter E4M3 MMAs as they are, against each q row scaled by a power of two
 * and split into two E4M3 terms (exact for every element within 2^9 of
 * the row's largest).  That is the decode kernel's mma.sync tiles for decode
 * rows; longer requests take the tcgen05 prefill tiles (codes widened in
 * shared memory, each q row rewritten as f16 scaled so its largest magnitude
 * lies in [2^14, 2^15)).  At head_dim 64 the codes are widened to fp32 in
 * registers on CUDA cores.
 *   q, out            device bf16 [num_tokens, num_q_heads, head_dim].
 *   k_cache, v_cache  device uint8 [num_blocks, 16, num_kv_heads, head_dim].
 *   k_scale, v_scale  finite, > 0 (else PKV_ERR_INVALID_ARG).
 * Everything else as pkv_attention_varlen, workspace included: requests with
 * n > PKV_DECODE_MAX_QLEN take the tensor-core prefill where the bf16 call's
 * would at head_dim 128 (a positive softmax_scale, no window below 128 keys),
 * else the decode kernel's CUDA-core tiles.
 */
pkv_status pkv_attention_varlen_e4m3(const void* q, const void* k_cache, const void* v_cache,
                                     void* out, float* lse_out, const int32_t* query_start_loc,
                                     const int32_t* seq_lens, const int32_t* block_table,
                                     int max_blocks_per_seq, int num_seqs, int64_t num_tokens,
                                     int max_query_len, int max_seq_len, int num_q_heads,
                                     int num_kv_heads, int head_dim, int block_size,
                                     float softmax_scale, float k_scale, float v_scale, int causal,
                                     int num_splits, void* workspace, size_t workspace_bytes,
                                     int32_t* error_flag, int64_t num_blocks, void* stream);

/*
 * pkv_attention_varlen_e4m3_window - pkv_attention_varlen_e4m3 with a sliding
 * window: the row at position p keeps keys j with p - window < j, on top of
 * the causal limit, as pkv_attention_varlen_window.
 *   window  >= 0 (0: no window; negative: PKV_ERR_INVALID_ARG).
 * Everything else as pkv_attention_varlen_e4m3.
 */
pkv_status pkv_attention_varlen_e4m3_window(
    const void* q, const void* k_cache, const void* v_cache, void* out, float* lse_out,
    const int32_t* query_start_loc, const int32_t* seq_lens, const int32_t* block_table,
    int max_blocks_per_seq, int num_seqs, int64_t num_tokens, int max_query_len, int max_seq_len,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, float softmax_scale,
    float k_scale, float v_scale, int causal, int window, int num_splits, void* workspace,
    size_t workspace_bytes, int32_t* error_flag, int64_t num_blocks, void* stream);

/*
 * pkv_write_attention_varlen_e4m3 - pkv_write_e4m3 then
 * pkv_attention_varlen_e4m3, as one call: the write rides in the decode
 * kernel (quantising bf16 rows with k_scale / v_scale as pkv_write_e4m3
 * does) when every request is decode-class, as for
 * pkv_write_attention_varlen.  k_new, v_new: bf16 [num_tokens,
 * num_kv_heads, head_dim].  Other arguments as pkv_attention_varlen_e4m3.
 */
pkv_status pkv_write_attention_varlen_e4m3(
    const void* k_new, const void* v_new, const int64_t* slot_mapping, const void* q,
    void* k_cache, void* v_cache, void* out, float* lse_out, const int32_t* query_start_loc,
    const int32_t* seq_lens, const int32_t* block_table, int max_blocks_per_seq, int num_seqs,
    int64_t num_tokens, int max_query_len, int max_seq_len, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, float softmax_scale, float k_scale, float v_scale, int causal,
    int num_splits, void* workspace, size_t workspace_bytes, int32_t* error_flag,
    int64_t num_blocks, void* stream);

/*
 * pkv_attention_varlen_noalloc - pkv_attention_varlen without a caller
 * workspace.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory (for example a plain C host program
 * whose device memory is owned by another runtime's caching allocator, or a
 * path that must never block in cudaMalloc/cudaFree).  The split-KV partials
 * live in a fixed 8 MiB array compiled into the library (held on every GPU
 * that loads it until the process exits); the call allocates nothing.
 *   Arguments are those of pkv_attention_varlen minus the workspace.  With
 *   num_splits == 0 the automatic split count is lowered until its partials
 *   (pkv_workspace_bytes) fit in 8 MiB; an explicit num_splits whose partials
 *   exceed 8 MiB returns PKV_ERR_WORKSPACE and enqueues nothing.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current): make it before any
 *   stream capture.  Host threads may make first calls concurrently (the
 *   cached address is atomic).  All calls on a device share the array, so
 *   calls whose kernels overlap on the GPU race; serialise them.
 */
pkv_status pkv_attention_varlen_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                        void* out, float* lse_out,
                                        const int32_t* query_start_loc, const int32_t* seq_lens,
                                        const int32_t* block_table, int max_blocks_per_seq,
                                        int num_seqs, int64_t num_tokens, int max_query_len,
                                        int max_seq_len, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, float softmax_scale,
                                        int causal, int num_splits, int32_t* error_flag,
                                        int64_t num_blocks, pkv_dtype dtype, void* stream);

/*
 * Shared-prefix (cascade) attention.
 *
 * "Anatomy of a serving engine", section "Capacity belongs to the KV cache
 * manager": paged blocks let requests share the blocks of a common prefix.
 * Here every request of the batch starts with the same shared_blocks blocks
 * (P = 16 * shared_blocks keys, named by shared_block_table) followed by its
 * own suffix_lens[r] keys (suffix_block_table row r); its context is
 * L = P + suffix_lens[r] and its n new tokens are the last n of them, all in
 * its own part (n <= suffix_lens[r], else PKV_FLAG_BAD_LENGTHS).  The result
 * is that of pkv_attention_varlen (causal) with the table shared ++ own.
 * It is computed as the key axis split in two ("Inside the engine ...",
 * section "Prefill has a full grid; decode at batch 1 has almost none": a
 * split of the keys changes nothing about the result): every row of the
 * batch over the prefix at once (all prefix keys are visible to every new
 * row; the prefix is read from HBM once for all requests, split
 * prefix_splits ways over the key axis), each request over its own keys,
 * and a log-sum-exp merge of the prefix_splits + 1 partials per row.  The
 * prefix pass runs on the tensor cores for bf16 at head_dim 64 or 128 (E4M3
 * caches at 128, pkv_cascade_attention_e4m3) with an even GQA group that
 * divides 128 (each 128-row tile holds 128 / group tokens with their whole
 * group, so one K/V tile feeds every head of the KV head) and a positive
 * softmax_scale, else on the split-KV kernel's CUDA-core tiles; the own-key
 * pass runs on the decode kernel and the merge on CUDA cores.
 */

/* pkv_cascade_splits - prefix splits for num_tokens rows over shared_blocks
 * blocks: max(1, min(floor(T / U), cap, 63)) with T = floor(7 x SMs / 8).
 * Tensor-core prefix pass (bf16, head_dim 64 or 128, even GQA group dividing
 * 128): U = num_kv_heads x ceil(group x num_tokens / 256) row tiles, cap =
 * ceil(shared_blocks / 32) - each split at least four 128-key tiles (fewer
 * leave the pass short of its pipelined steady state).  CUDA-core pass
 * (otherwise): U = num_kv_heads x ceil(group x num_tokens / 16), cap =
 * floor(shared_blocks / 8).  0 when shared_blocks == 0; -1 for invalid
 * arguments or device. */
int pkv_cascade_splits(int64_t num_tokens, int shared_blocks, int num_q_heads, int num_kv_heads,
                       int head_dim, pkv_dtype dtype, int device);

/* pkv_cascade_workspace_bytes - device workspace pkv_cascade_attention needs:
 * fp32 partial outputs [prefix_splits + 1][num_tokens][num_q_heads][head_dim]
 * and their log-sum-exps, each 256-byte aligned. */
size_t pkv_cascade_workspace_bytes(int64_t num_tokens, int num_q_heads, int head_dim,
                                   int prefix_splits);

/*
 * pkv_cascade_attention - attention of a batch sharing a block-aligned prefix.
 *
 *   q, out, lse_out, query_start_loc, num_seqs, num_tokens, max_query_len,
 *   heads, head_dim, block_size, softmax_scale, error_flag, num_blocks,
 *   dtype, stream: as pkv_attention_varlen.
 *   suffix_lens         device int32 [num_seqs]: keys after the prefix.
 *   suffix_block_table  device int32 [num_seqs, max_blocks_per_seq]: the
 *                       blocks of those keys.
 *   shared_block_table  device int32 [shared_blocks] (NULL when 0 blocks).
 *   max_suffix_len      host, >= every suffix_lens[r] and <= 16 *
 *                       max_blocks_per_seq (else PKV_ERR_INVALID_ARG).
 *   prefix_splits       0 = pkv_cascade_splits(...); else 1..63.
 *   workspace           device, >= pkv_cascade_workspace_bytes(num_tokens,
 *                       num_q_heads, head_dim, splits), 256-byte aligned
 *                       (splits = 0 when shared_blocks == 0).
 * Rows of out past query_start_loc[num_seqs] are not written (the prefix
 * pass reads every q row below num_tokens).
 */
pkv_status pkv_cascade_attention(const void* q, const void* k_cache, const void* v_cache,
                                 void* out, float* lse_out, const int32_t* query_start_loc,
                                 const int32_t* suffix_lens, const int32_t* suffix_block_table,
                                 int max_blocks_per_seq, const int32_t* shared_block_table,
                                 int shared_blocks, int num_seqs, int64_t num_tokens,
                                 int max_query_len, int max_suffix_len, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size,
                                 float softmax_scale, int prefix_splits, void* workspace,
                                 size_t workspace_bytes, int32_t* error_flag, int64_t num_blocks,
                                 pkv_dtype dtype, void* stream);

/*
 * pkv_cascade_attention_e4m3 - pkv_cascade_attention over an E4M3 cache (the
 * format of pkv_write_e4m3; k_scale, v_scale finite and > 0, else
 * PKV_ERR_INVALID_ARG).  q and out are bf16.  At head_dim 128 the prefix
 * pass runs on the tensor-core prefill tiles where the bf16 call's would
 * (even GQA group dividing 128, positive softmax_scale; codes widened to f16,
 * q rows scaled to f16 by powers of two) and prefix_splits 0 takes
 * pkv_cascade_splits(..., PKV_BF16, ...); otherwise it runs on the split-KV
 * kernel's CUDA-core tiles and takes pkv_cascade_splits(..., PKV_F32, ...).
 * The own-key pass runs on the decode kernel (tensor cores at head_dim 128).
 * Everything else as pkv_cascade_attention.
 */
pkv_status pkv_cascade_attention_e4m3(
    const void* q, const void* k_cache, const void* v_cache, void* out, float* lse_out,
    const int32_t* query_start_loc, const int32_t* suffix_lens, const int32_t* suffix_block_table,
    int max_blocks_per_seq, const int32_t* shared_block_table, int shared_blocks, int num_seqs,
    int64_t num_tokens, int max_query_len, int max_suffix_len, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, float softmax_scale, float k_scale, float v_scale,
    int prefix_splits, void* workspace, size_t workspace_bytes, int32_t* error_flag,
    int64_t num_blocks, void* stream);

/*
 * pkv_build_metadata - the flat-batch metadata of one step, on the host.
 *
 * "Model execution", section "Flattening a step": the scheduled tokens of all
 * requests form one flat batch; query_start_loc holds the cumulative token
 * offsets, seq_lens the context after this step (computed + scheduled),
 * block_table each request's physical blocks, and slot_mapping the slot
 * block_id * block_size + offset of new token k of request r, which sits at
 * position computed[r] + k.  Host memory only; no CUDA call.
 *   computed, scheduled  host int32 [num_seqs], >= 0.
 *   block_offsets        host int32 [num_seqs + 1], [0] = 0, nondecreasing:
 *                        request r's blocks are block_ids[block_offsets[r] ..
 *                        block_offsets[r + 1]), at least ceil((computed +
 *                        scheduled) / block_size) of them, ids >= 0.
 *   max_blocks_per_seq   width of block_table, >= every request's block count.
 *   num_tokens           must equal the sum of scheduled.
 *   Outputs (host, caller-allocated): query_start_loc int32 [num_seqs + 1],
 *   seq_lens int32 [num_seqs], block_table int32 [num_seqs,
 *   max_blocks_per_seq] (unused entries 0), slot_mapping int64 [num_tokens],
 *   positions int64 [num_tokens] or NULL, max_query_len / max_seq_len host
 *   int32 or NULL.
 * Every argument is checked before anything is written; a violation returns
 * PKV_ERR_INVALID_ARG and writes nothing.
 */
pkv_status pkv_build_metadata(int num_seqs, const int32_t* computed, const int32_t* scheduled,
                              const int32_t* block_offsets, const int32_t* block_ids,
                              int block_size, int max_blocks_per_seq, int64_t num_tokens,
                              int32_t* query_start_loc, int32_t* seq_lens, int32_t* block_table,
                              int64_t* slot_mapping, int64_t* positions, int32_t* max_query_len,
                              int32_t* max_seq_len);

/* Static, human-readable name of a status code. */
const char* pkv_status_string(pkv_status status);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
