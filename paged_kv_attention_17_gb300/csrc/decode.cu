// Split-KV decode attention over the paged cache, and the log-sum-exp combine.
//
// "Inside the engine: kernels, CUDA graphs and the life of a request":
//   * "Never materialise the TxT matrix" - K/V tiles stream past the query rows
//     while a running max m and denominator l are kept; the accumulator is
//     rescaled by e^(m_old - m_new) whenever the max moves.
//   * "Prefill has a full grid; decode at batch 1 has almost none" - with few
//     query rows the KV axis is split, each split runs the same online softmax
//     and a second reduction kernel combines the partials.
//   * "Attention over a block table, not a contiguous tensor" - every
//     16-token block is fetched through the request's block table.
//
// Design (GB300):
//   * One CTA = (split, kv head, row tile of one request).  The rows of a tile
//     are the GQA group's query heads x the request's new tokens, so every K/V
//     byte fetched from HBM feeds all query heads that share the kv head.
//   * Every warp streams its own blocks (b0 + w, b0 + w + warps, ...) through
//     its own ring of shared-memory stages, one 16-token block of K and of V
//     per stage with a "K full" and a "V full" mbarrier each (one waiter, so
//     parity waits cannot alias): it issues a block's TMA boxes from several
//     lanes at once (the TMA unit serves boxes from many issuing threads in
//     parallel, while one thread's boxes go one after another), computes its
//     scores as soon as K lands, and refills the stage with its block P
//     further on as soon as it has read it.  Block ids come from the table in
//     windows of 32 tiles, one per lane, the next window loaded ahead.
//   * Tensor-core build (bf16 caches, and E4M3 caches of head_dim 128): the
//     tile's rows are the M dimension of mma.sync m16n8k16 for both Q.K^T
//     and P.V (K and V read from 128B-swizzled stages by ldmatrix, or as E4M3
//     codes widened to f16 in registers), with a lagged reference max per row;
//     four warps and a 96 KB ring, so two CTAs fit on an SM.
//   * CUDA-core build (fp32 caches, E4M3 at head_dim 64): a register-q path
//     for one token of a 4-head group (each lane dots a 16-dim slice of the
//     four q rows with packed fp32 FMAs, a transpose-reduce over 8 lanes) and
//     a generic path (lanes own keys, q staged in shared memory).
//   * Before the programmatic-dependent-launch wait (while the previous
//     kernel finishes) the CTA sets up its barriers, prefetches the tensor
//     maps and warms L2 with the K/V blocks it will most likely read; every
//     input it then uses is read after the wait.
//   * In split launches each warp's first block is loaded right after the
//     wait from the block id read before it, and kept only if the metadata
//     and table read after the wait confirm it; otherwise the warp lets that
//     fill land and its stage's phases run one ahead.
//   * Each warp keeps its own (m, l, acc); the warps are merged through shared
//     memory at the end (same algebra as the split merge).
//   * Bounded mbarrier waits: a stuck pipeline sets PKV_FLAG_TIMEOUT and exits.
//   * Variants over the same pipeline: E4M3 caches (k/v scales folded into
//     the score scale and the epilogue); sliding windows (a tile's range
//     starts at its first row's window, each row masks below its own); the
//     cascade passes (every row of the batch over a shared prefix, or a
//     request's own keys, written as fp32 partials); and the fused write
//     (warp 0 stores the step's new K/V rows this CTA reads, and a block
//     holding one is loaded only after a barrier says they are stored).
#include <type_traits>

#include "common.cuh"

namespace pkv {

// Element type of the cache (float, bf16 or an E4M3 code) and of q / out
// (the same, except bf16 for E4M3 caches).
template <typename T>
constexpr bool kIsE4m3 = std::is_same<T, e4m3_t>::value;
template <typename T>
struct QType {
  using type = T;
};
template <>
struct QType<e4m3_t> {
  using type = __nv_bfloat16;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Packed fp32 pairs (fma.rn.f32x2 / mul.rn.f32x2 on sm_100+): two lanes of
// fp32 arithmetic per instruction.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(f32x2 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ void fma2(f32x2& acc, f32x2 a, f32x2 b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ void mul2(f32x2& acc, f32x2 a) {
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(acc) : "l"(a));
}
__device__ __forceinline__ f32x2 bf16x2_to_f32x2(uint32_t w) { return pack2(bf16_lo(w), bf16_hi(w)); }

// ---- warp-level tensor-core helpers (mma.sync m16n8k16, ldmatrix) ----
// D += A.B for a 16x16 A (four .b32 registers: rows g and g+8, k 2q..2q+1 and
// 2q+8..2q+9 for lane 4g+q) and a 16x8 B (two registers: k 2q..2q+1 and
// 2q+8..2q+9, column g); D rows g (d0, d1) and g+8 (d2, d3), columns 2q, 2q+1.
template <bool F16>
__device__ __forceinline__ void mma16816(float& d0, float& d1, float& d2, float& d3,
                                         uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Four 8x8 16-bit matrices from shared memory: lane l gives the address of
// row l % 8 of matrix l / 8; register i receives matrix i (plain: row l / 4,
// columns 2(l % 4), +1; .trans: the transposed matrix's).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
// Transpose of an 8x8 16-bit matrix held one .b32 (row l / 4, columns
// 2 (l % 4), +1) per lane: lane l receives the same slots of the transpose.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// two E4M3 codes (low 16 bits, element 0 in the low byte) -> f16x2, exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t h2;
  asm("{\n\t.reg .b16 c, u;\n\tmov.b32 {c, u}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
      : "=r"(h2)
      : "r"(two_codes));
  return h2;
}
// four E4M3 codes (a word, element 0 in the low byte) -> f16x2 of codes 0, 1
// and of codes 2, 3: the word's 16-bit halves feed the conversions directly
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four_codes, uint32_t& lo,
                                                  uint32_t& hi) {
  asm("{\n\t.reg .b16 c0, c1;\n\tmov.b32 {c0, c1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, c0;\n\tcvt.rn.f16x2.e4m3x2 %1, c1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(four_codes));
}
// (lo, hi) -> bf16x2 / f16x2, round to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float f16_lo(uint32_t w) {
  float f;
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, l;\n\t}"
      : "=f"(f)
      : "r"(w));
  return f;
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
  float f;
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, h;\n\t}"
      : "=f"(f)
      : "r"(w));
  return f;
}

// D += A.B for a 16x32 A and a 32x8 B of E4M3 codes (fp32 accumulation):
// lane 4g+q holds A rows g (a0, a2) and g+8 (a1, a3), k 4q..4q+3 (a0, a1) and
// 16+4q..16+4q+3 (a2, a3), four codes a register, element 0 in the low byte;
// B column g, k 4q..4q+3 (b0) and 16+4q.. (b1); D as for mma16816.
__device__ __forceinline__ void mma16832_e4m3(float& d0, float& d1, float& d2, float& d3,
                                              uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four values x0..x3 (each with at most 8 significant bits, magnitudes below
// 2^8) as two E4M3 words, element 0 in the low byte: hi is x rounded to E4M3,
// lo the remainder x - hi rounded to E4M3.  The remainder has at most 4
// significant bits and x's last bit, so hi + lo = x exactly when that bit is
// on E4M3's 2^-9 grid (|x| >= 2^-2); below, |hi + lo - x| <= 2^-10.
__device__ __forceinline__ void e4m3_split4(float x0, float x1, float x2, float x3,
                                            uint32_t& hi, uint32_t& lo) {
  uint32_t h01, h23, l01, l23;
  asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tcvt.u32.u16 %0, t;\n\t}"
      : "=r"(h01) : "f"(x1), "f"(x0));
  asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tcvt.u32.u16 %0, t;\n\t}"
      : "=r"(h23) : "f"(x3), "f"(x2));
  hi = h01 | (h23 << 16);
  uint32_t f01, f23;                                   // hi widened back (exactly) to f16
  e4m3x4_to_f16x2x2(hi, f01, f23);
  const float r0 = x0 - f16_lo(f01), r1 = x1 - f16_hi(f01);
  const float r2 = x2 - f16_lo(f23), r3 = x3 - f16_hi(f23);
  asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tcvt.u32.u16 %0, t;\n\t}"
      : "=r"(l01) : "f"(r1), "f"(r0));
  asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tcvt.u32.u16 %0, t;\n\t}"
      : "=r"(l23) : "f"(r3), "f"(r2));
  lo = l01 | (l23 << 16);
}

// Tensor-core (mma.sync m16n8k16) build of the decode kernel: bf16 caches
// (head_dim 64 or 128) and E4M3 caches of head_dim 128.  The GQA group's
// rows (up to 16 per tile) are the M dimension of both contractions, so one
// K/V tile feeds every query head of its kv head through the tensor cores
// and a 16-key block costs a warp about a hundred instructions instead of
// several hundred of CUDA-core FMAs.  fp32 caches and E4M3 at head_dim 64
// keep the CUDA-core build.
template <typename T, int D>
constexpr bool kMmaBuild = (sizeof(T) == 2 && (D == 64 || D == 128)) || (kIsE4m3<T> && D == 128);

template <typename T, int D, int R = 4>
struct DecodeCfg {
  static constexpr bool kMma = kMmaBuild<T, D>;
  static constexpr int kRowBytes = D * static_cast<int>(sizeof(T));
  static constexpr int kHalfChunks = kRowBytes / 32;      // 16-byte chunks per half key row
  // CUDA-core build: K and V each arrive as one unswizzled TMA box per block
  // (16 rows of the head's kRowBytes); the register-q path has the 8 lanes of
  // a quarter-warp read 8 consecutive 16-byte chunks of one key row, the
  // generic path rotates each lane's chunk order by its key, so neither
  // conflicts on shared-memory banks.  Tensor-core build: the rows' 128-byte
  // column slices land slice-major ([slice][16 rows][128 B], 128B-swizzled),
  // so the ldmatrix row reads of 8 consecutive keys hit 8 distinct bank
  // groups; one 4-D box (column, slot, slice, head) brings all slices of a
  // block, since the copy unit takes a warp's boxes one at a time (~37 ns
  // each), which bounds a block's issue, not its bytes.
  static constexpr int kBoxes = 1;                          // boxes per block of K (of V)
  static constexpr int kBoxBytes = kMma ? kBlock * 128 : kBlock * kRowBytes;  // per column slice
  static constexpr int kStageBytes = 2 * kBlock * kRowBytes;   // one block of K and of V
  // Consumer (compute) warps per CTA, plus one TMA producer warp.  CUDA-core
  // build: 11 + 1 warps (three per SM sub-partition, 168 registers each) for
  // 4-row tiles, whose register-q path fits that budget; wider tiles keep
  // 255 registers with 7 + 1 warps; one CTA per SM.  Tensor-core build: a 96
  // KB ring, so two CTAs fit on an SM and the next launch's CTAs become
  // resident (and warm L2) while this one streams; 6 + 1 warps (two stages of
  // bf16 per warp), or 7 + 1 over an E4M3 cache, whose half-size stages still
  // give each warp three and whose longer per-block path gains from the extra
  // warp (8 + 1 would leave 96 registers a thread).
  static constexpr int kWarps = kMma ? (kIsE4m3<T> ? 7 : 6) : (R == 4 ? 11 : 7);
  static constexpr int kRingBudget = kMma ? 98304 : 196608;
  static constexpr int kStagesRaw = kRingBudget / (kWarps * kStageBytes);
  static constexpr int kStagesPerWarp = kStagesRaw < 1 ? 1 : (kStagesRaw > 6 ? 6 : kStagesRaw);
  static constexpr int kStages = kWarps * kStagesPerWarp;
  static constexpr int kMinBlocksPerSm = kMma ? 2 : 1;
  // Blocks per CTA warmed into L2 before the dependent-launch wait.  CUDA-core
  // build: each consumer warp's first block (warming more floods the memory
  // queues that the previous kernel's last loads wait in, with one CTA per
  // SM).  Tensor-core build: a split launch's whole range up to this cap (its
  // CTAs are resident beside the previous launch's), else the first ring fill.
  static constexpr int kPrefetchBlocks = kMma ? 64 : kWarps;
  static constexpr int kConsumerThreads = kWarps * 32;
  static constexpr int kThreads = kConsumerThreads + 32;  // + one TMA producer warp
  // producer lanes: one per (consumer warp, K or V, 128-byte box), so every
  // TMA box of a block is issued by a thread of its own
  static constexpr int kIssueLanes = kWarps * 2 * kBoxes;
  static_assert(kIssueLanes <= 32, "one producer lane per box");
  static constexpr int kDPL = D / 32;                     // output columns per lane
  static constexpr int kPairs = kDPL / 2;
  static_assert((kHalfChunks & (kHalfChunks - 1)) == 0, "chunks per half row: power of two");
  static_assert(!kMma || kRowBytes % 128 == 0, "tensor-core build: rows of whole 128-byte slices");
};

template <typename T, int D, int R>
struct DecodeSmem {
  using C = DecodeCfg<T, D, R>;
  static constexpr int kStageArea = C::kStages * C::kStageBytes;
  static constexpr int kMergeBytes = C::kWarps * R * (D + 3) * 4;   // m, l, l~, acc per row
  static constexpr int kRingBytes = kStageArea > kMergeBytes ? kStageArea : kMergeBytes;
  // CUDA-core build: q rows as fp32; tensor-core build: the tile's q rows as
  // loaded (bf16), rows padded by 16 bytes so the fragment reads of 8 rows
  // hit distinct banks, or (E4M3 cache, E4M3 contraction of K) the rows' hi
  // codes, their lo codes (D + 16 bytes a row each) and a score scale per row
  static constexpr int kQRowBytes = D * 2 + 16;
  static constexpr int kQCodeRowBytes = D + 16;
  static constexpr int kQCodeBytes = C::kMma && kIsE4m3<T> ? 2 * R * kQCodeRowBytes + R * 4 : 0;
  static constexpr int kQOff = kRingBytes;
  static constexpr int kQBytes =
      C::kMma ? (kQCodeBytes > R * kQRowBytes ? kQCodeBytes : R * kQRowBytes) : R * D * 4;
  static constexpr int kPOff = kQOff + kQBytes;
  static constexpr int kBarOff = kPOff + (C::kMma ? 0 : C::kWarps * kBlock * R * 8);
  // kfull[], vfull[], empty[], then per consumer warp the barrier and the
  // verdict of its speculative first block
  static constexpr int kSpecOff = kBarOff + 3 * C::kStages * 8;
  // then the barrier of the fused KV write
  static constexpr int kWrOff = kSpecOff + C::kWarps * 8 + (C::kWarps * 4 + 7) / 8 * 8;
  static constexpr int kBytes = kWrOff + 8;
  static constexpr int kAlloc = kBytes + 1024;            // slack to align the base to 1 KB
};

// Position of q element (row, d) in shared memory.  fp32 and E4M3 caches:
// plain rows.  bf16: a 16-byte key chunk holds 8 elements whose fp32 q
// counterparts (32 bytes) are stored as two 16-byte halves in separate
// regions, so the rotated chunk reads of 8 lanes hit 8 distinct bank groups.
template <typename T, int D>
__device__ __forceinline__ int q_index(int row, int d) {
  if constexpr (sizeof(T) == 4 || kIsE4m3<T>) {
    return row * D + d;
  } else {
    const int c = d >> 3, w = d & 7;
    return row * D + (w >> 2) * (D / 2) + c * 4 + (w & 3);
  }
}

template <typename T>
__device__ __forceinline__ float load_elem(const void* base, int64_t idx) {
  if constexpr (sizeof(T) == 4) {
    return __ldg(static_cast<const float*>(base) + idx);
  } else {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
  }
}

template <typename T>
__device__ __forceinline__ void store_elem(void* base, int64_t idx, float v) {
  if constexpr (sizeof(T) == 4) {
    static_cast<float*>(base)[idx] = v;
  } else {
    static_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
  }
}

// Workspace row of (split, request, decode row, q head).
__device__ __forceinline__ int64_t ws_row(const AttnArgs& a, int s, int r, int i, int h) {
  return ((static_cast<int64_t>(s) * a.num_seqs + r) * kDecodeMaxQ + i) * a.hq + h;
}

// Workspace row of a partial: by (split, request, decode row) in a plain call,
// by (slot, flat token t) in the cascade passes.
__device__ __forceinline__ int64_t part_row(const AttnArgs& a, int s, int r, int64_t t, int i,
                                            int h) {
  return a.cascade ? (static_cast<int64_t>(s) * a.num_tokens + t) * a.hq + h
                   : ws_row(a, s, r, i, h);
}

// Longest-first dispatch of an unsplit launch (at most kLptMaxSeqs requests):
// the request whose rank, by decreasing seq_len (ties by index), equals
// `rank`.  After the dependency wait every CTA computes the same ranking from
// the same seq_lens, so the ranks are a bijection onto the requests; the
// request's query_start_loc pair and seq_len, loaded in the same round trip,
// are returned too.  Before the wait (hint = true, L2-only loads of values
// that may still change) the result only steers the L2 warm-up.  Keys are
// unique (length in the high bits, reversed index in the low nine), so a
// request's rank is the number of keys above its own.  Called by every thread.
__device__ __forceinline__ int request_by_length_rank(const AttnArgs& a, int rank, bool hint,
                                                      int& q0, int& q1, int& len) {
  __shared__ uint32_t s_key[kLptMaxSeqs];
  __shared__ int s_len[kLptMaxSeqs];
  __shared__ int s_qsl[kLptMaxSeqs + 1];
  __shared__ int s_pick;
  const int n = a.num_seqs;
  for (int i = threadIdx.x; i <= n; i += blockDim.x) {
    s_qsl[i] = hint ? __ldcg(a.qsl + i) : __ldg(a.qsl + i);
    if (i < n) {
      const int L = hint ? __ldcg(a.seq_lens + i) : __ldg(a.seq_lens + i);
      s_len[i] = L;
      s_key[i] = (static_cast<uint32_t>(min(max(L, 0), (1 << 22) - 1)) << 9) |
                 static_cast<uint32_t>(511 - i);
    }
  }
  if (threadIdx.x == 0) s_pick = rank;     // (every rank is taken below)
  __syncthreads();
  for (int c = threadIdx.x; c < n; c += blockDim.x) {
    const uint32_t kc = s_key[c];
    int above = 0;
    for (int j = 0; j < n; ++j) above += s_key[j] > kc ? 1 : 0;
    if (above == rank) s_pick = c;
  }
  __syncthreads();
  const int r = s_pick;
  q0 = s_qsl[r];
  q1 = s_qsl[r + 1];
  len = s_len[r];
  __syncthreads();                          // the arrays are reused by a second call
  return r;
}

// A lane's kDPL consecutive floats of a partial row in one vector store (the
// row is D floats and the lane's slice starts at a multiple of kDPL floats).
template <int kDPL>
__device__ __forceinline__ void store_partial(float* dst, const float (&o)[kDPL]) {
  if constexpr (kDPL == 4) {
    *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
  } else if constexpr (kDPL == 2) {
    *reinterpret_cast<float2*>(dst) = make_float2(o[0], o[1]);
  } else {
#pragma unroll
    for (int e = 0; e < kDPL; ++e) dst[e] = o[e];
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// this thread's generic-proxy global stores before its later async-proxy (TMA) reads
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// V columns lane*kDPL .. +kDPL-1 of one cached row, as fp32 pairs.
template <typename T, int D>
__device__ __forceinline__ void load_v_pairs(const uint8_t* vrow, int lane,
                                             f32x2 (&v)[DecodeCfg<T, D>::kPairs]) {
  using C = DecodeCfg<T, D>;
  if constexpr (sizeof(T) == 4) {
    if constexpr (C::kPairs == 1) {
      v[0] = *reinterpret_cast<const f32x2*>(vrow + lane * 8);
    } else {
      const ulonglong2 t = *reinterpret_cast<const ulonglong2*>(vrow + lane * 16);
      v[0] = t.x;
      v[1] = t.y;
    }
  } else if constexpr (kIsE4m3<T>) {
    if constexpr (C::kPairs == 1) {
      const float2 f = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(vrow + lane * 2));
      v[0] = pack2(f.x, f.y);
    } else {
      const uint32_t c4 = *reinterpret_cast<const uint32_t*>(vrow + lane * 4);
      const float2 f0 = e4m3x2_to_float2(c4 & 0xffffu), f1 = e4m3x2_to_float2(c4 >> 16);
      v[0] = pack2(f0.x, f0.y);
      v[1] = pack2(f1.x, f1.y);
    }
  } else {
    if constexpr (C::kPairs == 1) {
      v[0] = bf16x2_to_f32x2(*reinterpret_cast<const uint32_t*>(vrow + lane * 4));
    } else {
      const uint2 t = *reinterpret_cast<const uint2*>(vrow + lane * 8);
      v[0] = bf16x2_to_f32x2(t.x);
      v[1] = bf16x2_to_f32x2(t.y);
    }
  }
}

// SPEC: build with the speculative first blocks (used for split launches of
// 4-row tiles; unsplit launches run the build without, which measures faster)
template <typename T, int D, int R, bool SPEC>
__global__ void __launch_bounds__(DecodeCfg<T, D, R>::kThreads, DecodeCfg<T, D, R>::kMinBlocksPerSm)
    decode_kernel(const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const AttnArgs a) {
  using C = DecodeCfg<T, D, R>;
  using Sm = DecodeSmem<T, D, R>;
  constexpr int P = C::kStagesPerWarp;
  constexpr int W = C::kWarps;
  // Register-q path for one token of a 4-query-head GQA group (CUDA-core
  // build); every other CUDA-core shape takes the generic path below.
  using QT = typename QType<T>::type;                  // q / out element type
  constexpr bool kMma = C::kMma;                      // tensor-core build (see DecodeCfg)
  constexpr bool kFast = !kMma && (sizeof(T) == 2 || kIsE4m3<T>) && R == 4;
  constexpr int kFastChunks = D / 64;                 // 16-byte q chunks per row and lane
  // speculative first blocks (below) for the 4-row tiles of split launches,
  // where each CTA's first block is on the critical path
  constexpr bool kSpec = SPEC && R == 4;
  // whether this CTA may speculate (same answer on every thread)
  const bool spec_possible =
      kSpec && a.num_splits > 1 && blockIdx.y == 0 && a.window == 0 && a.cascade == 0;
  constexpr int kPWarpFloats = kBlock * R * 2;        // p_s floats per warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* q_s = reinterpret_cast<float*>(smem + Sm::kQOff);
  float* p_s = reinterpret_cast<float*>(smem + Sm::kPOff);   // [warp][key][row] (p, p)
  uint64_t* kfull = reinterpret_cast<uint64_t*>(smem + Sm::kBarOff);   // K of a stage landed
  uint64_t* vfull = kfull + C::kStages;                                 // V of a stage landed
  uint64_t* empty = vfull + C::kStages;                                 // stage released
  uint64_t* spec_bar = reinterpret_cast<uint64_t*>(smem + Sm::kSpecOff);
  int* spec_state = reinterpret_cast<int*>(spec_bar + C::kWarps);
  uint64_t* wr_bar = reinterpret_cast<uint64_t*>(smem + Sm::kWrOff);   // fused write stored

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool producer = warp == W;
  // producer lane -> (consumer warp pw, box part pp: K boxes, then V boxes)
  const int pw = lane / (2 * C::kBoxes), pp = lane % (2 * C::kBoxes);
  const bool p_act = producer && lane < C::kIssueLanes;
  const int g = blockIdx.x % a.hkv;
  const int s = blockIdx.x / a.hkv;
  const int z = blockIdx.y;
  // the request: blockIdx.z, or (longest-first launches) the request of that
  // rank by length, hinted before the wait and settled after it
  int hq0 = 0, hq1 = 0, hlen = 0;
  const int r_grid = a.lpt ? request_by_length_rank(a, blockIdx.z, true, hq0, hq1, hlen)
                           : static_cast<int>(blockIdx.z);

  // ---- set-up that reads no input: under programmatic dependent launch it
  //      overlaps the tail of the previous kernel in the stream ----
  if (producer && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&vfull[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < W; ++i) mbar_init(&spec_bar[i], 1);
    mbar_init(wr_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int32_t* table_hint = a.block_table + static_cast<int64_t>(r_grid) * a.max_blocks_per_seq;
  // the split range a context of max_seq_len keys gives (the pre-launch hint)
  const int nb_spec = min((a.max_seq_len + kBlock - 1) / kBlock, a.max_blocks_per_seq);
  const int per_spec = a.num_splits > 1 ? (nb_spec + a.num_splits - 1) / a.num_splits : nb_spec;
  const int spec_b0 = min(s * per_spec, nb_spec);
  int32_t e_hint = 0;                  // producer lane: hinted entry of warp pw's first block
  bool hint_ok = false;
  if (z == 0 && a.window == 0 && a.cascade == 0) {
    // ---- L2 warm-up while the previous kernel finishes: the K/V blocks this
    //      split will most likely read (the hinted split range, cut at the
    //      request's length, the table row and a cap).  A block of the cache
    //      holds every KV head's rows contiguously, and the CTAs of the split
    //      (one per KV head) read the same blocks, so CTA g warms every
    //      hkv-th block of the range whole, K and V, with one bulk prefetch
    //      each: a few operations of the asynchronous copy unit instead of a
    //      line-by-line stream of load-unit requests, which the loads after
    //      the wait would queue behind.  The table and lengths read here may
    //      still change before the wait, so they only steer prefetches: every
    //      value used below is re-read after the wait, and L2 stays coherent
    //      with the previous kernel's writes.  Only the first row tile of a
    //      request warms L2 (the others share its blocks or exit at once). ----
    // L2-only loads (ld.global.cg): nothing read before the wait may sit in L1,
    // where the read-only loads after the wait could find a stale copy
    const int len_hint = min(max(__ldcg(a.seq_lens + r_grid), 0), a.max_seq_len);
    const int n_hint = __ldcg(a.qsl + r_grid + 1) - __ldcg(a.qsl + r_grid);
    const bool runs_here = n_hint >= 1 && (n_hint <= kDecodeMaxQ || a.long_rows);
    // tensor-core build without a split: the blocks of the first ring fill
    const int pf_cap = kMma && a.num_splits == 1 ? C::kStages : C::kPrefetchBlocks;
    const int sb1 = !runs_here ? spec_b0
                               : min(min(min(spec_b0 + per_spec, (len_hint + kBlock - 1) / kBlock),
                                         spec_b0 + pf_cap),
                                     nb_spec);
    if (p_act && spec_possible && spec_b0 + pw < sb1) {
      e_hint = __ldcg(table_hint + spec_b0 + pw);
      hint_ok = true;
    }
    if (!producer && warp == 0) {
      const int64_t block_bytes = static_cast<int64_t>(kBlock) * a.hkv * C::kRowBytes;
      for (int bb = spec_b0 + g + a.hkv * lane; bb < sb1; bb += 32 * a.hkv) {
        const int32_t id = __ldcg(table_hint + bb);
        if (id < 0 || id >= a.num_blocks) continue;
        bulk_prefetch_l2(static_cast<const uint8_t*>(a.k_cache) + id * block_bytes,
                         static_cast<uint32_t>(block_bytes));
        bulk_prefetch_l2(static_cast<const uint8_t*>(a.v_cache) + id * block_bytes,
                         static_cast<uint32_t>(block_bytes));
      }
    }
  }

  // where this request's rows start in q (an address hint, read L2-only)
  const int q0_hint = kMma && !producer && a.cascade != 1 ? __ldcg(a.qsl + r_grid) : 0;

  // ---- inputs only after the wait ----
  pdl_wait_primary();
  pdl_launch_dependents();
  // longest request first: the grid's CTAs start in block-index order, so an
  // unsplit launch of requests of unequal length ends with a tail of long
  // ones unless blockIdx.z is read as a rank of the requests by length
  int lq0 = 0, lq1 = 0, llen = 0;
  const int r = a.lpt ? request_by_length_rank(a, blockIdx.z, false, lq0, lq1, llen) : r_grid;
  const int32_t* table = a.block_table + static_cast<int64_t>(r) * a.max_blocks_per_seq;
  // The request's metadata and the table entries of the hinted split range
  // are the first loads after the wait (everything after depends on them);
  // the speculative q rows and K/V boxes go out behind them.
  // cascade prefix pass: one request holding every row of the batch, over the
  // prefix_len shared keys
  const bool prefix_pass = a.cascade == 1;
  const int md_q0 = prefix_pass ? 0 : (a.lpt ? lq0 : ld_early(a.qsl + r));
  const int md_q1 = prefix_pass ? static_cast<int>(a.num_tokens)
                                : (a.lpt ? lq1 : ld_early(a.qsl + r + 1));
  const int md_L = prefix_pass ? a.prefix_len : (a.lpt ? llen : ld_early(a.seq_lens + r));
  // the table entries of warp pw's first two blocks of the hinted split range:
  // the verdict on the speculative block and the first loads need no second
  // round trip when the real range starts at the hinted block
  const bool spec_v0 = p_act && spec_b0 + pw < nb_spec;
  const bool spec_v1 = p_act && spec_b0 + pw + W < nb_spec;
  const int32_t spec_e0 = spec_v0 ? ld_early(table + spec_b0 + pw) : 0;
  const int32_t spec_e1 = spec_v1 ? ld_early(table + spec_b0 + pw + W) : 0;
  // Tensor-core build: the q rows of this tile are loaded at once from the
  // hinted start (token index kept inside q, so every load is in bounds) in
  // 16-byte pieces by all consumer threads, in flight together with the
  // metadata; reloaded below if the metadata puts the rows elsewhere, then
  // staged in shared memory, where each lane picks its fragment words.
  constexpr int kMT = kMma ? D / 16 : 1;               // k-steps of Q.K^T
  // E4M3 cache: K's codes enter the MMAs as they are (m16n8k32 E4M3 against
  // q split into two E4M3 terms) in tiles of up to 8 rows, where the
  // per-block path dominates; the speculative form (split launches without
  // a window: latency-bound) keeps the shorter q set-up of f16 MMAs over
  // widened codes
  constexpr bool kF8Mma = kMma && kIsE4m3<T> && !SPEC && R <= 8;
  constexpr bool kHi = R == 16;                        // M-rows 8..15 are tile rows
  constexpr int kHR = kHi ? 2 : 1;                     // M-row halves this lane holds
  constexpr int kQChunks = R * D / 8;                  // 16-byte pieces of the tile's q rows
  constexpr int kQLd = kMma ? (kQChunks + C::kConsumerThreads - 1) / C::kConsumerThreads : 1;
  const int g8 = lane >> 2, kq = lane & 3;
  uint4 qld[kQLd];
  auto load_q = [&](int q0v) {
#pragma unroll
    for (int u = 0; u < kQLd; ++u) {
      const int idx = threadIdx.x + u * C::kConsumerThreads;
      if (idx < kQChunks) {
        const int rr = blockIdx.y * R + idx / (D / 8);
        const int64_t tok = min(max(static_cast<int64_t>(q0v) + rr / a.group, int64_t{0}),
                                a.num_tokens - 1);
        qld[u] = ld_early_v4(static_cast<const QT*>(a.q) +
                             (tok * a.hq + g * a.group + rr % a.group) * D + (idx % (D / 8)) * 8);
      }
    }
  };
  if constexpr (kMma) {
    if (!producer) load_q(q0_hint);
  }
  // Producer lane (pw, pp) issues box pp of each block of consumer warp pw:
  // TMA boxes from many issuing threads proceed in parallel, while one
  // thread's boxes go one after another.  The first box of K (of V) posts its
  // barrier's byte count.
  const uint64_t pol = l2_policy_evict_first();
  auto issue_box = [&](int st, int row) {
    const bool v = pp >= C::kBoxes;
    uint64_t* bar = v ? &vfull[st] : &kfull[st];
    mbar_arrive_expect_tx(bar, kBlock * C::kRowBytes);
    uint8_t* dst = smem + st * C::kStageBytes + (v ? kBlock * C::kRowBytes : 0);
    if constexpr (C::kMma && C::kRowBytes > 128)   // several 128-byte slices: the 4-D map
      tma_load_4d(dst, v ? &vmap : &kmap, bar, 0, row, 0, g, pol);
    else
      tma_load_3d(dst, v ? &vmap : &kmap, bar, 0, g, row, pol);
  };
  // Speculative first block: warp pw's first block of the hinted split range
  // goes into its stage 0 at once - the K/V data is read after the wait,
  // only the block id comes from the hint.  It is kept (used) only if the
  // metadata and table read below confirm that block id as the warp's first;
  // otherwise the fill is wasted and that stage's phases shift by one.  An
  // out-of-range hint loads rows -16..-1, which TMA fills with zeros without
  // reading memory.
  const bool spec_issued = p_act && spec_possible && hint_ok;
  if (spec_issued)
    issue_box(pw * P, (e_hint >= 0 && e_hint < a.num_blocks) ? e_hint * kBlock : -kBlock);
  // every exit from here on first lets a speculative load land (bounded)
  auto drain_spec = [&]() {
    if (spec_issued) mbar_wait(pp >= C::kBoxes ? &vfull[pw * P] : &kfull[pw * P], 0);
  };
  const int q0 = md_q0, q1 = md_q1;
  const int n = q1 - q0;
  const int L = md_L;
  if (n == 0) {
    drain_spec();
    return;
  }
  if (n < 0 || q0 < 0 || q1 > a.num_tokens || (n > L && !prefix_pass) || n > a.max_query_len) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && z == 0) raise_flag(a.flag, PKV_FLAG_BAD_LENGTHS);
    drain_spec();
    return;
  }
  const bool decode_class = n <= kDecodeMaxQ || prefix_pass;
  if (!decode_class && !a.long_rows) {                // the prefill kernel owns it
    drain_spec();
    return;
  }
  const bool split_mode = decode_class && a.num_splits > 1;
  if (!split_mode && s != 0) {
    drain_spec();
    return;
  }
  const int group = a.group;
  const int rows_total = group * n;
  const int rho0 = z * R;
  if (rho0 >= rows_total) {
    drain_spec();
    return;
  }
  const int nrows = min(R, rows_total - rho0);
  const int i_last = (rho0 + nrows - 1) / group;
  const int kv_len = a.causal ? (L - n + i_last + 1) : L;
  const int nblk = (kv_len + kBlock - 1) / kBlock;
  if (nblk > a.max_blocks_per_seq) {
    if (threadIdx.x == 0) raise_flag(a.flag, PKV_FLAG_BAD_LENGTHS);
    drain_spec();
    return;
  }
  // sliding window: the tile's first row sees keys from key_lo on, later rows
  // from further on; blocks below key_lo are never read
  const int key_lo = a.window > 0 ? max(0, L - n + rho0 / group - a.window + 1) : 0;
  const int blk_lo = min(key_lo / kBlock, nblk);
  int b0 = blk_lo, b1 = nblk;
  if (split_mode) {
    const int per = (nblk - blk_lo + a.num_splits - 1) / a.num_splits;
    b0 = blk_lo + min(s * per, nblk - blk_lo);
    b1 = min(b0 + per, nblk);
  }
  if (b0 >= b1) {
    // empty split: partial (o = 0, lse = -inf) so the combine weighs it 0
    for (int rho = warp; rho < nrows && warp < C::kWarps; rho += C::kWarps) {
      const int rr = rho0 + rho;
      const int64_t w = part_row(a, s, r, q0 + rr / group, rr / group, g * group + rr % group);
#pragma unroll
      for (int e = 0; e < C::kDPL; ++e) a.ws_o[w * D + lane * C::kDPL + e] = 0.f;
      if (lane == 0) a.ws_lse[w] = -INFINITY;
    }
    drain_spec();
    return;
  }
  const int key_end = min(kv_len, b1 * kBlock);       // keys of this split: [b0*16, key_end)
  // fused write: the new-token rows this CTA reads, positions [fw_lo, fw_hi)
  // (head g); warp 0 stores them, and a block holding one is loaded only
  // after that (wr_bar)
  const int fw_lo = a.fuse_write ? max(L - n, b0 * kBlock) : 0;
  const int fw_hi = a.fuse_write ? key_end : 0;
  const int nt = b1 - b0;                              // one block per stage
  const int my_tiles = nt > warp ? (nt - warp + W - 1) / W : 0;

  // q elements this thread stages (generic path), loaded before the causal
  // limits are worked out so the loads are in flight meanwhile
  constexpr int kQPer = kFast || kMma ? 1 : (R * D + C::kConsumerThreads - 1) / C::kConsumerThreads;
  QT qraw[kQPer];
  if constexpr (!kFast && !kMma) {
#pragma unroll
    for (int u = 0; u < kQPer; ++u) {
      const int e = threadIdx.x + u * C::kConsumerThreads;
      const int rho = e / D, d = e % D;
      if (!producer && e < R * D && rho < nrows) {
        const int rr = rho0 + rho;
        const int64_t t = q0 + rr / group;
        const int h = g * group + rr % group;
        qraw[u] = static_cast<const QT*>(a.q)[(t * a.hq + h) * D + d];
      } else {
        qraw[u] = QT(0.f);
      }
    }
  }

  float m[R], l[R];
  f32x2 acc[R][C::kPairs];
#pragma unroll
  for (int rho = 0; rho < R; ++rho) {
    m[rho] = -INFINITY;
    l[rho] = 0.f;
#pragma unroll
    for (int e = 0; e < C::kPairs; ++e) acc[rho][e] = 0ull;
  }

  const int kl = lane & (kBlock - 1);                  // key of this lane within a block
  const int half = lane >> 4;                          // which half of the key row it dots

  // ---- register-q path state: lane = (key group kg of 4 keys, D slice dc).
  //      The slice is chunks dc and dc + 8 of each row (16 dims for D = 128),
  //      so the 8 lanes of a group read 8 distinct bank groups of one row. ----
  const int kg = lane >> 3, dc = lane & 7;
  const int fb2 = (dc >> 2) & 1, fb1 = (dc >> 1) & 1, fb0 = dc & 1;
  const int my_r = 2 * fb2 + fb1;                      // row this lane owns after reduction
  const int kk0 = kg * 4 + 2 * fb0;                    // first of its two keys in a block
  f32x2 qr[kFast ? 4 : 1][kFast ? 4 * kFastChunks : 1];
  f32x2 acc2[kFast ? C::kDPL : 1][2];                  // [column][row pair (0,1) | (2,3)]
  float m_mine = -INFINITY, l_mine = 0.f;
  int lim_mine = 0, lo_mine = 0;
  // visible keys of each row: lo[rho] <= key < lim[rho] (causal limit, and the
  // sliding window's start, which is <= 0 without a window)
  const int wlo = a.window > 0 ? L - n - a.window + 1 : -(1 << 30);   // window start of row i: wlo + i
  int lim[R], lo[R];
#pragma unroll
  for (int rho = 0; rho < R; ++rho) {
    lim[rho] = min(key_end, a.causal ? (L - n + (rho0 + rho) / group + 1) : L);
    lo[rho] = wlo + (rho0 + rho) / group;
  }

  // ---- tensor-core build state.  Both contractions are taken transposed,
  //      S^T = K.Q^T and O^T = V^T.P^T, so the 16 keys of a block (and 16
  //      dims of O) fill the M dimension and the tile's rows the N dimension
  //      (8 per n-tile h; 16-row tiles have two): lane 4*g8 + kq holds the B
  //      operand of Q^T for rows 8h + g8 per 16-dim k-step, and for rows
  //      8h + 2kq + e (e = 0, 1) the running max (log2 domain, a lagged
  //      reference: moved only when a block's max passes it by more than
  //      kLag, so p <= 2^kLag), its partial sums of p (fp32: the row's mass,
  //      for the LSE and the split weights) and of p as rounded into the
  //      16-bit P operand (the accumulator's own normaliser, so the output is
  //      an exact weighted average of V rows), and the O^T accumulator per
  //      16-dim m-tile. ----
  constexpr int kMD = kMma ? D / 16 : 1;               // m-tiles of O^T (16 dims each)
  constexpr float kLag = 8.f;
  // B operands of S^T = K.Q^T: [t][rows 8h + g8: k lo, k hi per h]; E4M3
  // cache: [u] the hi words and [kMT / 2 + u] the lo words of k32-step u
  uint32_t qa[kMT][2 * kHR];
  float oacc[kMD][kHR][4];                             // O^T: dims g8 (c0, c1), g8 + 8 (c2, c3)
  float mm[kHR][2], ll[kHR][2], lr[kHR][2];
  int mlim[kHR][2], mlo[kHR][2];
  // log2-domain score scale of this lane's accumulator columns (rows
  // 8h + 2kq + e); per row for E4M3 caches, whose q rows carry their own
  // power-of-two scaling
  float rs[kHR][2];
#pragma unroll
  for (int hr = 0; hr < kHR; ++hr)
#pragma unroll
    for (int e = 0; e < 2; ++e) rs[hr][e] = a.scale_log2;
#pragma unroll
  for (int hr = 0; hr < kHR; ++hr)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      mm[hr][e] = -INFINITY;
      ll[hr][e] = 0.f;
      lr[hr][e] = 0.f;
      const int i_row = (rho0 + 8 * hr + 2 * kq + e) / group;   // token (padding rows too)
      mlim[hr][e] = min(key_end, a.causal ? (L - n + i_row + 1) : L);
      mlo[hr][e] = wlo + i_row;
    }
#pragma unroll
  for (int mt = 0; mt < kMD; ++mt)
#pragma unroll
    for (int hr = 0; hr < kHR; ++hr)
#pragma unroll
      for (int c = 0; c < 4; ++c) oacc[mt][hr][c] = 0.f;

  if (producer) {
    // ---- TMA producer: lane (pw, pp) issues box pp of every block of
    //      consumer warp pw (blocks b0 + pw + W j).  It polls the "empty"
    //      barrier of the warp's next stage without blocking and issues its
    //      box as soon as the stage is released; the lanes of ready stages
    //      issue together.  The compute warps never stall behind the TMA
    //      unit. ----
    const int tiles = (p_act && nt > pw) ? (nt - pw + W - 1) / W : 0;
    auto entry_of = [&](int jj) -> int32_t {
      return jj < tiles ? ld_early(table + b0 + pw + W * jj) : 0;
    };
    // a speculative first block holding new-token rows of a fused write was
    // loaded before they were stored: discard it
    const int sb = b0 + pw;
    const bool spec_clash = fw_lo < fw_hi && sb * kBlock < fw_hi && (sb + 1) * kBlock > fw_lo;
    const bool spec_ok = spec_b0 == b0;                 // the real range starts at the hint
    int32_t e_cur = spec_ok && spec_v0 ? spec_e0 : entry_of(0);
    int32_t e_next = spec_ok && spec_v1 ? spec_e1 : entry_of(1);
    // verdict on the speculative first block: 0 none, 1 used as tile 0,
    // 2 wasted (stage 0's phases then run one ahead of its tiles)
    const bool used = spec_issued && spec_ok && spec_v0 && tiles > 0 && spec_e0 == e_hint &&
                      !spec_clash;
    const int verdict = !spec_issued ? 0 : (used ? 1 : 2);
    if (verdict == 2) {
      // a wasted fill lands before the verdict is published (the consumer's
      // parity waits on stage 0 rely on it), bounded like every wait
      if (!mbar_wait(pp >= C::kBoxes ? &vfull[pw * P] : &kfull[pw * P], 0))
        raise_flag(a.flag, PKV_FLAG_TIMEOUT);
    }
    __syncwarp();
    if (spec_possible && p_act && pp == 0) {
      spec_state[pw] = verdict;
      mbar_arrive(&spec_bar[pw]);
    }
    if (used && pp == 0 && (e_hint < 0 || e_hint >= a.num_blocks))
      raise_flag(a.flag, PKV_FLAG_BAD_BLOCK);
    const int shift0 = verdict == 2;
    int jj = 0;
    if (used) {
      jj = 1;
      e_cur = e_next;
      e_next = entry_of(2);
    }
    unsigned long long t_progress = 0;
    while (__any_sync(0xffffffffu, jj < tiles)) {
      bool ready = false;
      if (jj < tiles) {
        const int st = pw * P + jj % P;
        ready = jj < P || mbar_ready(&empty[st], ((jj / P) - 1) & 1);
        // a wasted speculative fill must land before stage 0 is filled again
        if (ready && jj == 0 && shift0)
          ready = mbar_ready(&kfull[st], 0) && mbar_ready(&vfull[st], 0);
        // a block holding rows of the fused write only once they are stored
        if (ready && fw_lo < fw_hi) {
          const int bi = b0 + pw + W * jj;
          if (bi * kBlock < fw_hi && (bi + 1) * kBlock > fw_lo) ready = mbar_ready(wr_bar, 0);
        }
        if (ready) {
          int id = e_cur;
          if (id < 0 || id >= a.num_blocks) {
            if (pp == 0) raise_flag(a.flag, PKV_FLAG_BAD_BLOCK);
            id = 0;
          }
          if (jj >= P) fence_proxy_async_smem();   // the warp's reads of the stage before a refill
          issue_box(st, id * kBlock);
          ++jj;
          e_cur = e_next;
          e_next = entry_of(jj + 1);
        }
      }
      if (__any_sync(0xffffffffu, ready)) {
        t_progress = 0;
      } else {
        // nothing released yet: back off briefly; give up after ~2 s without progress
        const unsigned long long now = globaltimer();
        if (t_progress == 0) t_progress = now;
        if (now - t_progress > kWaitLimitNs) {
          if (lane == 0) raise_flag(a.flag, PKV_FLAG_TIMEOUT);
          break;
        }
        __nanosleep(32);
      }
    }
    // every box this lane issued has landed before the merge reuses the ring
    // (a no-op unless a consumer gave up early); bounded like every wait
    for (int q = 0; p_act && q < P; ++q) {
      const int c = (jj > q ? (jj - q + P - 1) / P : 0) + (q == 0 ? shift0 : 0);  // fills of stage q
      if (c > 0 && !mbar_wait(pp >= C::kBoxes ? &vfull[pw * P + q] : &kfull[pw * P + q], (c - 1) & 1))
        break;
    }
    __syncwarp();
  } else {
    if constexpr (kMma) {
      // ---- q (loaded right after the wait): reloaded if the metadata puts
      //      the rows elsewhere, staged in shared memory, and each lane's B
      //      operand words picked for rows 8h + g8 (zero past the tile's
      //      rows).  E4M3 cache: each q row is scaled by a power of two
      //      bringing its max|q| into [2^7, 2^8) and split into two E4M3
      //      terms (hi + lo: exact for every element within 2^9 of the row's
      //      largest, off by at most 2^-17 of it below that), so K's codes
      //      enter the MMAs as they are; the row's score scale takes the
      //      inverse power. ----
      if (q0 != (prefix_pass ? 0 : q0_hint)) load_q(q0);
      uint8_t* qst = smem + Sm::kQOff;
      if constexpr (kF8Mma) {
        // E4M3 contraction: the 16 threads holding a row's 8-element chunks (a
        // half-warp) find its max|q|, scale it by 2^-e into [2^7, 2^8) and
        // split each chunk into hi + lo E4M3 codes; a row past the
        // tile's rows is zeros.  Code rows: hi at qst, lo R rows further,
        // then the rows' log2-domain score scales.
        static_assert(D / 8 == 16, "a q row is one half-warp's chunks");
        float* rscale = reinterpret_cast<float*>(qst + 2 * R * Sm::kQCodeRowBytes);
#pragma unroll
        for (int u = 0; u < kQLd; ++u) {
          const int idx = threadIdx.x + u * C::kConsumerThreads;
          const bool in = idx < kQChunks;
          const uint4 v = in ? qld[u] : make_uint4(0u, 0u, 0u, 0u);
          const float x[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                              bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
          float mx = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(x[i]));
#pragma unroll
          for (int o = 1; o < 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (in) {
            const int rho = idx / (D / 8), c = idx % (D / 8);
            const int ex = (__float_as_int(mx) >> 23) & 0xff;
            // max|q| in [2^E, 2^(E+1)): e = E - 7 (clamped so 2^-e and 2^e
            // are normal floats; a zero row takes e = 0); a row holding an
            // infinity or a NaN gets a NaN scale, so its scores are NaN
            const int e = mx > 0.f ? max(-120, min(120, ex - 127 - 7)) : 0;
            const float qs = __int_as_float((127 - e) << 23);      // 2^-e
            uint32_t h0 = 0u, h1 = 0u, l0 = 0u, l1 = 0u;
            if (rho < nrows) {
              e4m3_split4(x[0] * qs, x[1] * qs, x[2] * qs, x[3] * qs, h0, l0);
              e4m3_split4(x[4] * qs, x[5] * qs, x[6] * qs, x[7] * qs, h1, l1);
            }
            *reinterpret_cast<uint2*>(qst + rho * Sm::kQCodeRowBytes + 8 * c) =
                make_uint2(h0, h1);
            *reinterpret_cast<uint2*>(qst + (R + rho) * Sm::kQCodeRowBytes + 8 * c) =
                make_uint2(l0, l1);
            if (c == 0)
              rscale[rho] = rho < nrows && ex == 0xff
                                ? __int_as_float(0x7fc00000)
                                : a.scale_log2 * __int_as_float((127 + (rho < nrows ? e : 0)) << 23);
          }
        }
      } else {
#pragma unroll
        for (int u = 0; u < kQLd; ++u) {
          const int idx = threadIdx.x + u * C::kConsumerThreads;
          if (idx < kQChunks)
            *reinterpret_cast<uint4*>(qst + (idx / (D / 8)) * Sm::kQRowBytes + (idx % (D / 8)) * 16) =
                qld[u];
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(C::kConsumerThreads) : "memory");
      uint32_t qw[kHR][kMT][2];
#pragma unroll
      for (int hr = 0; hr < kHR; ++hr) {
        const int rho = g8 + 8 * hr;
        const uint8_t* qrow = qst + rho * Sm::kQRowBytes;
#pragma unroll
        for (int t = 0; t < kMT; ++t) {
          if (kF8Mma || rho >= nrows) {
            qw[hr][t][0] = qw[hr][t][1] = 0u;                // (kF8Mma: the code rows below)
          } else if constexpr (kIsE4m3<T>) {
            // dims 32kq + 4t .. +3
            const uint2 v = *reinterpret_cast<const uint2*>(qrow + (32 * kq + 4 * t) * 2);
            qw[hr][t][0] = v.x;
            qw[hr][t][1] = v.y;
          } else {
            // dims 16t + 2kq, +1 and 16t + 8 + 2kq, +1
            qw[hr][t][0] = *reinterpret_cast<const uint32_t*>(qrow + (16 * t + 2 * kq) * 2);
            qw[hr][t][1] = *reinterpret_cast<const uint32_t*>(qrow + (16 * t + 8 + 2 * kq) * 2);
          }
        }
      }
      if constexpr (kF8Mma) {
        // the lane's B words: row 8h + g8, dims 32kq .. 32kq + 31 of the hi
        // and lo code rows (word t: dims 32kq + 4t .. +3, k32-step t / 2, B
        // register t % 2); the scales of its accumulator columns, rows
        // 8h + 2kq + e
        const float* rscale = reinterpret_cast<const float*>(qst + 2 * R * Sm::kQCodeRowBytes);
#pragma unroll
        for (int hr = 0; hr < kHR; ++hr) {
          const int rho = g8 + 8 * hr;
          uint4 w[2][2] = {{make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)},
                           {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)}};
          if (rho < nrows) {
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2)
#pragma unroll
              for (int h = 0; h < 2; ++h)
                w[s2][h] = lds128(smem_u32(qst + (s2 * R + rho) * Sm::kQCodeRowBytes + 32 * kq + 16 * h));
          }
#pragma unroll
          for (int t = 0; t < kMT; ++t) {
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
              const uint4& c4 = w[s2][t >> 2];
              const uint32_t word = (t & 3) == 0 ? c4.x : (t & 3) == 1 ? c4.y : (t & 3) == 2 ? c4.z : c4.w;
              qa[s2 * (kMT / 2) + (t >> 1)][2 * hr + (t & 1)] = word;
            }
          }
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int rc = 8 * hr + 2 * kq + e2;
            rs[hr][e2] = rc < R ? rscale[rc] : a.scale_log2;
          }
        }
      } else if constexpr (kIsE4m3<T>) {
        // f16 contraction: the tile's q scaled by a power of two bringing its
        // max|q| into [2^14, 2^15), where f16 holds every bf16 element within
        // 2^31 of that maximum exactly; the score scale takes the inverse
        float mx = 0.f;
#pragma unroll
        for (int hr = 0; hr < kHR; ++hr)
#pragma unroll
          for (int t = 0; t < kMT; ++t)
#pragma unroll
            for (int u = 0; u < 2; ++u)
              mx = fmaxf(mx, fmaxf(fabsf(bf16_lo(qw[hr][t][u])), fabsf(bf16_hi(qw[hr][t][u]))));
        mx = warp_max(mx);
        int e = 0;
        if (mx > 0.f && mx <= 3.0e38f) e = ((__float_as_int(mx) >> 23) & 0xff) - 127 - 14;
        e = max(-100, min(100, e));
        const float qs = __int_as_float((127 - e) << 23);          // 2^-e
        const float sscale = a.scale_log2 * __int_as_float((127 + e) << 23);
#pragma unroll
        for (int hr = 0; hr < kHR; ++hr) {
#pragma unroll
          for (int t = 0; t < kMT; ++t)
#pragma unroll
            for (int u = 0; u < 2; ++u)
              qa[t][2 * hr + u] =
                  pack_f16x2(bf16_lo(qw[hr][t][u]) * qs, bf16_hi(qw[hr][t][u]) * qs);
          rs[hr][0] = rs[hr][1] = sscale;
        }
      } else {
#pragma unroll
        for (int hr = 0; hr < kHR; ++hr)
#pragma unroll
          for (int t = 0; t < kMT; ++t) {
            qa[t][2 * hr] = qw[hr][t][0];
            qa[t][2 * hr + 1] = qw[hr][t][1];
          }
      }
    } else if constexpr (kFast) {
      // this lane's q slice of all four rows straight from global memory (no
      // CTA-wide staging), pre-scaled into the log2 domain
      uint4 qv[4][kFastChunks];
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4) {
        const int rr = rho0 + r4;
        const int64_t qrow =
            (static_cast<int64_t>(q0 + rr / group) * a.hq + g * group + rr % group) * D;
#pragma unroll
        for (int cc = 0; cc < kFastChunks; ++cc)
          qv[r4][cc] = r4 < nrows ? __ldg(reinterpret_cast<const uint4*>(
                                        static_cast<const QT*>(a.q) + qrow +
                                        (kIsE4m3<T> ? (D / 8) * dc + 8 * cc : 8 * (dc + 8 * cc))))
                                  : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4)
#pragma unroll
        for (int cc = 0; cc < kFastChunks; ++cc) {
          const uint32_t wq[4] = {qv[r4][cc].x, qv[r4][cc].y, qv[r4][cc].z, qv[r4][cc].w};
#pragma unroll
          for (int p2 = 0; p2 < 4; ++p2)
            qr[r4][cc * 4 + p2] =
                pack2(bf16_lo(wq[p2]) * a.scale_log2, bf16_hi(wq[p2]) * a.scale_log2);
        }
#pragma unroll
      for (int c = 0; c < C::kDPL; ++c) acc2[c][0] = acc2[c][1] = 0ull;
      lim_mine = min(key_end, a.causal ? (L - n + (rho0 + my_r) / group + 1) : L);
      lo_mine = wlo + (rho0 + my_r) / group;
    } else {
      // ---- stage q rows (pre-scaled into the log2 domain), consumer warps only ----
#pragma unroll
      for (int u = 0; u < kQPer; ++u) {
        const int e = threadIdx.x + u * C::kConsumerThreads;
        if (e < R * D) q_s[q_index<T, D>(e / D, e % D)] = static_cast<float>(qraw[u]) * a.scale_log2;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(C::kConsumerThreads) : "memory");
    }
    // ---- fused write (warp 0): the K/V rows of head g of the new tokens this
    //      CTA reads; every CTA reading a row stores the same bytes first ----
    if (fw_lo < fw_hi && warp == 0) {
      // a chunk: 16 bytes of the new row (8 bf16 -> 8 codes for E4M3 caches)
      constexpr int kChunks = kIsE4m3<T> ? D / 8 : C::kRowBytes / 16;
      const int p_first = L - n;
      const int count = (fw_hi - fw_lo) * 2 * kChunks;
      const int64_t num_slots = a.num_blocks * kBlock;
      for (int c = lane; c < count; c += 32) {
        const int64_t t = q0 + (fw_lo - p_first) + c / (2 * kChunks);
        const int part = (c / kChunks) & 1;                  // 0: K, 1: V
        const int ch = c % kChunks;
        const int64_t slot = __ldg(a.slots + t);
        if (slot < 0) continue;                              // padding: nothing stored
        if (slot >= num_slots) {
          raise_flag(a.flag, PKV_FLAG_BAD_SLOT);
          continue;
        }
        uint8_t* cache = static_cast<uint8_t*>(const_cast<void*>(part ? a.v_cache : a.k_cache));
        if constexpr (kIsE4m3<T>) {
          // codes of value / scale: fp32 division, nearest code, saturating
          const uint4 x = __ldg(reinterpret_cast<const uint4*>(
                                    static_cast<const uint8_t*>(part ? a.v_new : a.k_new) +
                                    (t * a.hkv + g) * D * 2) + ch);
          const float sc = part ? a.wv_scale : a.wk_scale;
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
          uint32_t c2[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            c2[i] = float2_to_e4m3x2(__fdiv_rn(bf16_lo(w[i]), sc), __fdiv_rn(bf16_hi(w[i]), sc));
          *(reinterpret_cast<uint2*>(cache + (slot * a.hkv + g) * C::kRowBytes) + ch) =
              make_uint2(c2[0] | (c2[1] << 16), c2[2] | (c2[3] << 16));
        } else {
          const uint4* src = reinterpret_cast<const uint4*>(
                                 static_cast<const uint8_t*>(part ? a.v_new : a.k_new) +
                                 (t * a.hkv + g) * C::kRowBytes) + ch;
          *(reinterpret_cast<uint4*>(cache + (slot * a.hkv + g) * C::kRowBytes) + ch) =
              __ldg(src);
        }
      }
      // the stores before the producer's TMA (async proxy) loads of them
      fence_proxy_async_global();
      __syncwarp();
      if (lane == 0) mbar_arrive(wr_bar);
    }
    // the producer's verdict on this warp's speculative first block
    int shift0 = 0;
    if (spec_possible && my_tiles > 0) {
      if (!mbar_wait(&spec_bar[warp], 0)) {
        if (lane == 0) raise_flag(a.flag, PKV_FLAG_TIMEOUT);
      }
      // "wasted" is published only once that fill (phase 0 of stage 0) has
      // landed, so stage 0 is then in phase 1 or just past it, and the
      // parity-1 wait for tile 0 cannot pass early
      shift0 = spec_state[warp] == 2 ? 1 : 0;
    }
    for (int j = 0; j < my_tiles; ++j) {
      const int blk = b0 + warp + W * j;
      const int st = warp * P + (j % P);
      const int ph = (j / P + (j % P == 0 ? shift0 : 0)) & 1;   // phase of this fill
      const bool got = mbar_wait(&kfull[st], ph);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) raise_flag(a.flag, PKV_FLAG_TIMEOUT);
        break;
      }
      const uint8_t* ks = smem + st * C::kStageBytes;
      const uint8_t* vs = ks + kBlock * C::kRowBytes;
      const int key0 = blk * kBlock;
      const int nvalid = min(kBlock, key_end - key0);

      if constexpr (kMma) {
        constexpr bool kF16 = kIsE4m3<T>;              // f16 MMAs over widened E4M3 codes
        const uint32_t ks_u = smem_u32(ks), vs_u = smem_u32(vs);
        const int r8 = lane & 7, mi = lane >> 3;      // ldmatrix: row r8 of matrix mi
        // ---- S^T = K.Q^T: rows of the accumulator are the block's keys (g8,
        //      g8 + 8), columns the tile's rows; even and odd k-steps
        //      accumulate separately (independent MMA chains), then add ----
        float sc[2][kHR][4];                           // [k-step parity][n-tile][c]
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int hr = 0; hr < kHR; ++hr)
#pragma unroll
            for (int c = 0; c < 4; ++c) sc[u][hr][c] = 0.f;
        auto mma_s = [&](int t, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
#pragma unroll
          for (int hr = 0; hr < kHR; ++hr)
            mma16816<kF16>(sc[t & 1][hr][0], sc[t & 1][hr][1], sc[t & 1][hr][2], sc[t & 1][hr][3],
                           a0, a1, a2, a3, qa[t][2 * hr], qa[t][2 * hr + 1]);
        };
        if constexpr (kF8Mma) {
          // lane's codes: key rows g8 and g8 + 8, bytes 32kq .. 32kq + 31
          // (16-byte chunks 2kq, 2kq + 1, placed at chunk ^ (row % 8)).
          // k32-step u takes words 2u (k 4kq..) and 2u + 1 (k 16 + 4kq..) of
          // each row as they are: the codes are the A operand, against the hi
          // and lo terms of q in two independent accumulator chains
          uint4 kc[2][2];
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              kc[j][h] = lds128(ks_u + (g8 + 8 * j) * 128 + (((2 * kq + h) ^ g8) << 4));
          auto word = [&](const uint4& c4, int w) {
            return w == 0 ? c4.x : w == 1 ? c4.y : w == 2 ? c4.z : c4.w;
          };
#pragma unroll
          for (int u = 0; u < kMT / 2; ++u) {
            const int t0 = 2 * u, t1 = 2 * u + 1;
            const uint32_t a0 = word(kc[0][t0 >> 2], t0 & 3), a1 = word(kc[1][t0 >> 2], t0 & 3);
            const uint32_t a2 = word(kc[0][t1 >> 2], t1 & 3), a3 = word(kc[1][t1 >> 2], t1 & 3);
#pragma unroll
            for (int hr = 0; hr < kHR; ++hr) {
              mma16832_e4m3(sc[0][hr][0], sc[0][hr][1], sc[0][hr][2], sc[0][hr][3], a0, a1, a2,
                            a3, qa[u][2 * hr], qa[u][2 * hr + 1]);
              mma16832_e4m3(sc[1][hr][0], sc[1][hr][1], sc[1][hr][2], sc[1][hr][3], a0, a1, a2,
                            a3, qa[kMT / 2 + u][2 * hr], qa[kMT / 2 + u][2 * hr + 1]);
            }
          }
        } else if constexpr (kIsE4m3<T>) {
          // lane's codes: key rows g8 and g8 + 8, bytes 32kq .. 32kq + 31
          // (16-byte chunks 2kq, 2kq + 1, placed at chunk ^ (row % 8)),
          // widened to f16 k-step by k-step
          uint4 kc[2][2];
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              kc[j][h] = lds128(ks_u + (g8 + 8 * j) * 128 + (((2 * kq + h) ^ g8) << 4));
#pragma unroll
          for (int t = 0; t < kMT; ++t) {
            auto word = [&](const uint4& c4) {
              return (t & 3) == 0 ? c4.x : (t & 3) == 1 ? c4.y : (t & 3) == 2 ? c4.z : c4.w;
            };
            const uint32_t w0 = word(kc[0][t >> 2]), w1 = word(kc[1][t >> 2]);
            uint32_t a0, a1, a2, a3;
            e4m3x4_to_f16x2x2(w0, a0, a2);
            e4m3x4_to_f16x2x2(w1, a1, a3);
            mma_s(t, a0, a1, a2, a3);
          }
        } else {
          // matrix mi: keys 8 (mi & 1) .. +7, 16-byte chunk 2 (t % 4) + (mi >> 1)
          // of 128-byte slice t / 4
          const uint32_t krow = ks_u + (8 * (mi & 1) + r8) * 128;
#pragma unroll
          for (int t = 0; t < kMT; ++t) {
            uint32_t ka[4];
            ldsm_x4(ka, krow + (t >> 2) * C::kBoxBytes + (((2 * (t & 3) + (mi >> 1)) ^ r8) << 4));
            mma_s(t, ka[0], ka[1], ka[2], ka[3]);
          }
        }
        // ---- scores in the log2 domain, masked (keys past the split range,
        //      the causal limit, the window start); lane holds keys g8 (c0,
        //      c1) and g8 + 8 (c2, c3) of rows 8h + 2kq + e ----
        const int kA = key0 + g8, kB = key0 + g8 + 8;
        bool all_in = nvalid == kBlock;
#pragma unroll
        for (int hr = 0; hr < kHR; ++hr)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            all_in = all_in && key0 >= mlo[hr][e] && key0 + kBlock <= mlim[hr][e];
        all_in = __all_sync(0xffffffffu, all_in);
        float x[kHR][4];
#pragma unroll
        for (int hr = 0; hr < kHR; ++hr)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int e = c & 1, key = c < 2 ? kA : kB;
            const float v = (sc[0][hr][c] + sc[1][hr][c]) * rs[hr][e];
            x[hr][c] = all_in || (key < mlim[hr][e] && key >= mlo[hr][e]) ? v : -INFINITY;
          }
        // ---- online softmax with a lagged reference max per row: a row's 16
        //      keys sit on the 8 lanes of its kq ----
        float bm[kHR][2];
        bool need = false;
#pragma unroll
        for (int hr = 0; hr < kHR; ++hr)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float v = fmaxf(x[hr][e], x[hr][2 + e]);
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
            bm[hr][e] = v;
            need = need || v > mm[hr][e] + kLag;
          }
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int hr = 0; hr < kHR; ++hr)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const bool nd = bm[hr][e] > mm[hr][e] + kLag;
              const float al = nd ? ex2(mm[hr][e] - bm[hr][e]) : 1.f;   // 0 when mm was -inf
              mm[hr][e] = nd ? bm[hr][e] : mm[hr][e];
              ll[hr][e] *= al;
              lr[hr][e] *= al;
#pragma unroll
              for (int mt = 0; mt < kMD; ++mt) {
                oacc[mt][hr][e] *= al;
                oacc[mt][hr][2 + e] *= al;
              }
            }
        }
        // P^T (B operand of O^T += V^T.P^T) per n-tile: p of keys g8 | g8 + 8
        // for rows 2kq, 2kq + 1 packed into 16-bit pairs, then transposed so
        // each lane holds row g8's keys 2kq, 2kq+1 | 8+2kq, 9+2kq
        uint32_t pb[kHR][2];
#pragma unroll
        for (int hr = 0; hr < kHR; ++hr) {
          float p[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float m = mm[hr][c & 1];
            p[c] = ex2(x[hr][c] - (m == -INFINITY ? 0.f : m));
          }
          uint32_t pk[2];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if constexpr (kF16) {
              pk[j] = pack_f16x2(p[2 * j], p[2 * j + 1]);
              lr[hr][0] += f16_lo(pk[j]);
              lr[hr][1] += f16_hi(pk[j]);
            } else {
              pk[j] = pack_bf16x2(p[2 * j], p[2 * j + 1]);
              lr[hr][0] += bf16_lo(pk[j]);
              lr[hr][1] += bf16_hi(pk[j]);
            }
            ll[hr][0] += p[2 * j];
            ll[hr][1] += p[2 * j + 1];
            pb[hr][j] = movmatrix_t(pk[j]);
          }
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&vfull[st], ph))) {
          if (lane == 0) raise_flag(a.flag, PKV_FLAG_TIMEOUT);
          break;
        }
        // ---- O^T += V^T.P^T over 16-dim m-tiles ----
        auto mma_o = [&](int mt, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
#pragma unroll
          for (int hr = 0; hr < kHR; ++hr)
            mma16816<kF16>(oacc[mt][hr][0], oacc[mt][hr][1], oacc[mt][hr][2], oacc[mt][hr][3], a0,
                           a1, a2, a3, pb[hr][0], pb[hr][1]);
        };
        if constexpr (kIsE4m3<T>) {
          // lane's codes: keys 2kq, 2kq+1, 2kq+8, 2kq+9, dims 16 g8 .. +15 (one
          // 16-byte chunk each); m-tile mt takes its rows g8 and g8 + 8 as
          // dims 16 g8 + 2 mt and 16 g8 + 2 mt + 1, so a byte shuffle pairs
          // the two keys of each dim
          uint4 vc[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int kv = 2 * kq + (i & 1) + 8 * (i >> 1);
            vc[i] = lds128(vs_u + kv * 128 + ((g8 ^ (kv & 7)) << 4));
            // keys past the split range may hold anything (even NaN codes)
            if (nvalid < kBlock && kv >= nvalid) vc[i] = make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            auto word = [&](const uint4& c4) {
              return w == 0 ? c4.x : w == 1 ? c4.y : w == 2 ? c4.z : c4.w;
            };
            const uint32_t a0 = word(vc[0]), a1 = word(vc[1]), b0 = word(vc[2]), b1 = word(vc[3]);
            const uint32_t alo = prmt(a0, a1, 0x5140), ahi = prmt(a0, a1, 0x7362);
            const uint32_t blo = prmt(b0, b1, 0x5140), bhi = prmt(b0, b1, 0x7362);
            uint32_t x0, x1, y0, y1;
            e4m3x4_to_f16x2x2(alo, x0, x1);
            e4m3x4_to_f16x2x2(blo, y0, y1);
            mma_o(2 * w, x0, x1, y0, y1);
            e4m3x4_to_f16x2x2(ahi, x0, x1);
            e4m3x4_to_f16x2x2(bhi, y0, y1);
            mma_o(2 * w + 1, x0, x1, y0, y1);
          }
        } else {
          // matrix mi (.trans): keys 8 (mi >> 1) .. +7, chunk 2 (mt % 4) + (mi & 1)
          // of 128-byte slice mt / 4
          const uint32_t vrow = vs_u + (8 * (mi >> 1) + r8) * 128;
          // keys past the split range may hold anything: zero their V
          uint32_t mk0 = 0xffffffffu, mk1 = 0xffffffffu;
          if (nvalid < kBlock) {
            mk0 = (2 * kq < nvalid ? 0x0000ffffu : 0u) | (2 * kq + 1 < nvalid ? 0xffff0000u : 0u);
            mk1 = (2 * kq + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * kq + 9 < nvalid ? 0xffff0000u : 0u);
          }
#pragma unroll
          for (int mt = 0; mt < kMD; ++mt) {
            uint32_t va[4];
            ldsm_x4_t(va, vrow + (mt >> 2) * C::kBoxBytes +
                              (((2 * (mt & 3) + (mi & 1)) ^ r8) << 4));
            mma_o(mt, va[0] & mk0, va[1] & mk0, va[2] & mk1, va[3] & mk1);
          }
        }
      } else if constexpr (kFast) {
        // ---- scores: partial dots of 4 keys x 4 rows over this lane's slice ----
        f32x2 part[4][4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
          for (int r = 0; r < 4; ++r) part[t][r] = 0ull;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int key = kg * 4 + t;
          const uint8_t* krow = ks + key * C::kRowBytes;
          if constexpr (kIsE4m3<T>) {
            // this lane's D/8 consecutive codes of the key (16 or 8 bytes)
            uint32_t w[D / 32];
            if constexpr (D == 128) {
              const uint4 kc = *reinterpret_cast<const uint4*>(krow + dc * 16);
              w[0] = kc.x; w[1] = kc.y; w[2] = kc.z; w[3] = kc.w;
            } else {
              const uint2 kc = *reinterpret_cast<const uint2*>(krow + dc * 8);
              w[0] = kc.x; w[1] = kc.y;
            }
#pragma unroll
            for (int i = 0; i < D / 32; ++i) {
              const float2 f0 = e4m3x2_to_float2(w[i] & 0xffffu);
              const float2 f1 = e4m3x2_to_float2(w[i] >> 16);
              const f32x2 ka = pack2(f0.x, f0.y), kb = pack2(f1.x, f1.y);
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                fma2(part[t][r], qr[r][2 * i], ka);
                fma2(part[t][r], qr[r][2 * i + 1], kb);
              }
            }
          } else {
#pragma unroll
          for (int cc = 0; cc < kFastChunks; ++cc) {
            const int chunk = dc + 8 * cc;
            const uint4 kc = *reinterpret_cast<const uint4*>(krow + chunk * 16);
            const f32x2 k01 = bf16x2_to_f32x2(kc.x), k23 = bf16x2_to_f32x2(kc.y);
            const f32x2 k45 = bf16x2_to_f32x2(kc.z), k67 = bf16x2_to_f32x2(kc.w);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              fma2(part[t][r], qr[r][cc * 4 + 0], k01);
              fma2(part[t][r], qr[r][cc * 4 + 1], k23);
              fma2(part[t][r], qr[r][cc * 4 + 2], k45);
              fma2(part[t][r], qr[r][cc * 4 + 3], k67);
            }
          }
          }
        }
        // ---- transpose-reduce over the 8 slice lanes (xor 4, 2, 1): values
        //      v = row * 4 + key end up summed, two per lane (row my_r, keys
        //      kk0 and kk0 + 1) ----
        float sv[16];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float2 x = unpack2(part[t][r]);
            sv[r * 4 + t] = x.x + x.y;
          }
        float s8[8], s4[4], s2[2];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float send = fb2 ? sv[i] : sv[i + 8], keep = fb2 ? sv[i + 8] : sv[i];
          s8[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float send = fb1 ? s8[i] : s8[i + 4], keep = fb1 ? s8[i + 4] : s8[i];
          s4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float send = fb0 ? s4[i] : s4[i + 2], keep = fb0 ? s4[i + 2] : s4[i];
          s2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
        }
        // ---- online softmax of row my_r (the 8 lanes holding it share m) ----
        const float x0 = key0 + kk0 < lim_mine && key0 + kk0 >= lo_mine ? s2[0] : -INFINITY;
        const float x1 =
            key0 + kk0 + 1 < lim_mine && key0 + kk0 + 1 >= lo_mine ? s2[1] : -INFINITY;
        float mx = fmaxf(x0, x1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mnew = fmaxf(m_mine, mx);
        const float msafe = mnew == -INFINITY ? 0.f : mnew;
        const float alpha = ex2(m_mine - msafe);
        const float p0 = ex2(x0 - msafe), p1 = ex2(x1 - msafe);
        l_mine = l_mine * alpha + (p0 + p1);
        m_mine = mnew;
        float* pw = p_s + warp * kPWarpFloats;           // [16 keys][4 rows], then alpha[4]
        pw[kk0 * 4 + my_r] = p0;
        pw[(kk0 + 1) * 4 + my_r] = p1;
        if (kg == 0 && fb0 == 0) pw[kBlock * 4 + my_r] = alpha;
        __syncwarp();
        const ulonglong2 al = *reinterpret_cast<const ulonglong2*>(pw + kBlock * 4);
#pragma unroll
        for (int c = 0; c < C::kDPL; ++c) {
          mul2(acc2[c][0], al.x);
          mul2(acc2[c][1], al.y);
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&vfull[st], ph))) {
          if (lane == 0) raise_flag(a.flag, PKV_FLAG_TIMEOUT);
          break;
        }
        // ---- P.V: lane owns columns lane*kDPL.., rows paired in each FMA ----
        auto pv_fast = [&](int jj) {
          const ulonglong2 pp = *reinterpret_cast<const ulonglong2*>(pw + jj * 4);
          f32x2 v[C::kPairs];
          load_v_pairs<T, D>(vs + jj * C::kRowBytes, lane, v);
#pragma unroll
          for (int e = 0; e < C::kPairs; ++e) {
            const float2 vf = unpack2(v[e]);
            const f32x2 va = pack2(vf.x, vf.x), vb = pack2(vf.y, vf.y);
            fma2(acc2[2 * e][0], pp.x, va);
            fma2(acc2[2 * e][1], pp.y, va);
            fma2(acc2[2 * e + 1][0], pp.x, vb);
            fma2(acc2[2 * e + 1][1], pp.y, vb);
          }
        };
        if (nvalid == kBlock) {
#pragma unroll
          for (int jj = 0; jj < kBlock; ++jj) pv_fast(jj);
        } else {
#pragma unroll 4
          for (int jj = 0; jj < nvalid; ++jj) pv_fast(jj);
        }
      } else {
      // ---- scores: lane owns key key0 + kl, half of its row; halves summed by shuffle ----
      f32x2 sc2[R];
#pragma unroll
      for (int rho = 0; rho < R; ++rho) sc2[rho] = 0ull;
      const uint8_t* krow = ks + kl * C::kRowBytes;      // this key's row
#pragma unroll
      for (int c = 0; c < C::kHalfChunks; ++c) {
        // 16-byte chunk of the full row, order rotated by the key (bank spread)
        const int chunk = half * C::kHalfChunks + ((c + kl) & (C::kHalfChunks - 1));
        const uint4 kc = *reinterpret_cast<const uint4*>(krow + chunk * 16);
        if constexpr (sizeof(T) == 4) {
          const f32x2 k01 = pack2(__uint_as_float(kc.x), __uint_as_float(kc.y));
          const f32x2 k23 = pack2(__uint_as_float(kc.z), __uint_as_float(kc.w));
#pragma unroll
          for (int rho = 0; rho < R; ++rho) {
            const ulonglong2 qa = *reinterpret_cast<const ulonglong2*>(q_s + rho * D + chunk * 4);
            fma2(sc2[rho], qa.x, k01);
            fma2(sc2[rho], qa.y, k23);
          }
        } else if constexpr (kIsE4m3<T>) {
          // 16 codes = dims 16 chunk .. 16 chunk + 15
          const uint32_t w[4] = {kc.x, kc.y, kc.z, kc.w};
          f32x2 kp[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f0 = e4m3x2_to_float2(w[i] & 0xffffu);
            const float2 f1 = e4m3x2_to_float2(w[i] >> 16);
            kp[2 * i] = pack2(f0.x, f0.y);
            kp[2 * i + 1] = pack2(f1.x, f1.y);
          }
#pragma unroll
          for (int rho = 0; rho < R; ++rho) {
            const ulonglong2* qp = reinterpret_cast<const ulonglong2*>(q_s + rho * D + chunk * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const ulonglong2 qq = qp[i];
              fma2(sc2[rho], qq.x, kp[2 * i]);
              fma2(sc2[rho], qq.y, kp[2 * i + 1]);
            }
          }
        } else {
          const f32x2 k01 = bf16x2_to_f32x2(kc.x), k23 = bf16x2_to_f32x2(kc.y);
          const f32x2 k45 = bf16x2_to_f32x2(kc.z), k67 = bf16x2_to_f32x2(kc.w);
#pragma unroll
          for (int rho = 0; rho < R; ++rho) {
            const ulonglong2 qa = *reinterpret_cast<const ulonglong2*>(q_s + rho * D + chunk * 4);
            const ulonglong2 qb =
                *reinterpret_cast<const ulonglong2*>(q_s + rho * D + D / 2 + chunk * 4);
            fma2(sc2[rho], qa.x, k01);
            fma2(sc2[rho], qa.y, k23);
            fma2(sc2[rho], qb.x, k45);
            fma2(sc2[rho], qb.y, k67);
          }
        }
      }

      // ---- online softmax update (per row; m uniform over the warp).  Every
      //      row of the tile is computed (rows past nrows have q = 0 and are
      //      never stored), so the rows' shuffle and exp chains interleave ----
      const int key = key0 + kl;
      float* pw = p_s + ((warp * kBlock + kl) * R) * 2;
      float sv[R], mx[R];
#pragma unroll
      for (int rho = 0; rho < R; ++rho) {
        const float2 t2 = unpack2(sc2[rho]);
        sv[rho] = t2.x + t2.y;
      }
#pragma unroll
      for (int rho = 0; rho < R; ++rho) sv[rho] += __shfl_xor_sync(0xffffffffu, sv[rho], 16);
#pragma unroll
      for (int rho = 0; rho < R; ++rho) {
        sv[rho] = key < lim[rho] && key >= lo[rho] ? sv[rho] : -INFINITY;
        mx[rho] = sv[rho];
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
#pragma unroll
        for (int rho = 0; rho < R; ++rho)
          mx[rho] = fmaxf(mx[rho], __shfl_xor_sync(0xffffffffu, mx[rho], o));
      }
#pragma unroll
      for (int rho = 0; rho < R; ++rho) {
        const float mnew = fmaxf(m[rho], mx[rho]);
        const float msafe = mnew == -INFINITY ? 0.f : mnew;
        const float alpha = ex2(m[rho] - msafe);
        const float p = ex2(sv[rho] - msafe);
        l[rho] = l[rho] * alpha + (half == 0 ? p : 0.f);
        m[rho] = mnew;
        const f32x2 a2 = pack2(alpha, alpha);
#pragma unroll
        for (int e = 0; e < C::kPairs; ++e) mul2(acc[rho][e], a2);
        if (half == 0) *reinterpret_cast<float2*>(pw + rho * 2) = make_float2(p, p);
      }
      __syncwarp();

      if (!__all_sync(0xffffffffu, mbar_wait(&vfull[st], ph))) {
        if (lane == 0) raise_flag(a.flag, PKV_FLAG_TIMEOUT);
        break;
      }
      // ---- P.V: lane owns output columns lane*kDPL .. +kDPL-1 ----
      auto pv_key = [&](int jj) {
        const float* pr = p_s + ((warp * kBlock + jj) * R) * 2;
        f32x2 pp[R];
#pragma unroll
        for (int r2 = 0; r2 < R; r2 += 2) {
          const ulonglong2 t = *reinterpret_cast<const ulonglong2*>(pr + r2 * 2);
          pp[r2] = t.x;
          pp[r2 + 1] = t.y;
        }
        f32x2 v[C::kPairs];
        load_v_pairs<T, D>(vs + jj * C::kRowBytes, lane, v);
#pragma unroll
        for (int rho = 0; rho < R; ++rho) {
#pragma unroll
          for (int e = 0; e < C::kPairs; ++e) fma2(acc[rho][e], pp[rho], v[e]);
        }
      };
      if (nvalid == kBlock) {
        // a full block: fully unrolled, so its loads are issued ahead of the FMAs
#pragma unroll
        for (int jj = 0; jj < kBlock; ++jj) pv_key(jj);
      } else {
#pragma unroll 4
        for (int jj = 0; jj < nvalid; ++jj) pv_key(jj);
      }
      }  // generic path
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);   // stage free for the producer
    }
  }  // consumer warps

  // ---- merge the warps' states (shared memory reused) ----
  __syncthreads();
  float* mw = reinterpret_cast<float*>(smem);
  float* lw = mw + C::kWarps * R;                      // row mass (fp32 sum of p)
  float* lrw = lw + C::kWarps * R;                     // the accumulator's normaliser
  float* aw = lrw + C::kWarps * R;
  if (kMma && !producer) {
    // rows 8h + 2kq + e of this warp: l summed over the row's eight lanes;
    // accumulator slot c of m-tile mt is dim 16 mt + g8 (+ 8 for c >= 2) for
    // a bf16 cache, 16 g8 + 2 mt (+ 1 for c >= 2) for an E4M3 cache
#pragma unroll
    for (int hr = 0; hr < kHR; ++hr)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float lt = ll[hr][e], lrt = lr[hr][e];
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          lt += __shfl_xor_sync(0xffffffffu, lt, o);
          lrt += __shfl_xor_sync(0xffffffffu, lrt, o);
        }
        const int rho = 8 * hr + 2 * kq + e;
        if (rho < R) {
          if (g8 == 0) {
            mw[warp * R + rho] = mm[hr][e];
            lw[warp * R + rho] = lt;
            lrw[warp * R + rho] = lrt;
          }
#pragma unroll
          for (int mt = 0; mt < kMD; ++mt)
#pragma unroll
            for (int hi = 0; hi < 2; ++hi) {
              const int dim = kIsE4m3<T> ? 16 * g8 + 2 * mt + hi : 16 * mt + g8 + 8 * hi;
              aw[(warp * R + rho) * D + dim] = oacc[mt][hr][2 * hi + e];
            }
        }
      }
  }
  if (kFast && !producer) {
    float lt = l_mine + __shfl_xor_sync(0xffffffffu, l_mine, 1);
    lt += __shfl_xor_sync(0xffffffffu, lt, 8);
    lt += __shfl_xor_sync(0xffffffffu, lt, 16);
    if (kg == 0 && fb0 == 0) {
      mw[warp * R + my_r] = m_mine;
      lw[warp * R + my_r] = lt;
    }
#pragma unroll
    for (int c = 0; c < C::kDPL; ++c) {
      const float2 a01 = unpack2(acc2[c][0]), a23 = unpack2(acc2[c][1]);
      aw[(warp * R + 0) * D + lane * C::kDPL + c] = a01.x;
      aw[(warp * R + 1) * D + lane * C::kDPL + c] = a01.y;
      aw[(warp * R + 2) * D + lane * C::kDPL + c] = a23.x;
      aw[(warp * R + 3) * D + lane * C::kDPL + c] = a23.y;
    }
  }
#pragma unroll
  for (int rho = 0; rho < R; ++rho) {
    if (!kFast && !kMma && !producer && rho < nrows) {
      const float lt = warp_sum(l[rho]);
      if (lane == 0) {
        mw[warp * R + rho] = m[rho];
        lw[warp * R + rho] = lt;
      }
#pragma unroll
      for (int e = 0; e < C::kPairs; ++e)
        *reinterpret_cast<float2*>(aw + (warp * R + rho) * D + lane * C::kDPL + 2 * e) =
            unpack2(acc[rho][e]);
    }
  }
  __syncthreads();
  for (int rho = warp; rho < nrows && !producer; rho += W) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) M = fmaxf(M, mw[w * R + rho]);
    float o[C::kDPL];
#pragma unroll
    for (int e = 0; e < C::kDPL; ++e) o[e] = 0.f;
    float lsum = 0.f, lnorm = 0.f;   // row mass; the accumulator's normaliser
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < C::kWarps; ++w) {
        const float f = ex2(mw[w * R + rho] - M);
        lsum = fmaf(f, lw[w * R + rho], lsum);
        if constexpr (kMma) lnorm = fmaf(f, lrw[w * R + rho], lnorm);
        // the lane's slice in one shared-memory load (aw starts 3 x W x R
        // floats in, a multiple of 16 bytes; rows are D floats)
        const float* src = aw + (w * R + rho) * D + lane * C::kDPL;
        if constexpr (C::kDPL == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          o[0] = fmaf(f, v.x, o[0]);
          o[1] = fmaf(f, v.y, o[1]);
          o[2] = fmaf(f, v.z, o[2]);
          o[3] = fmaf(f, v.w, o[3]);
        } else {
#pragma unroll
          for (int e = 0; e < C::kDPL; ++e) o[e] = fmaf(f, src[e], o[e]);
        }
      }
    }
    if constexpr (!kMma) lnorm = lsum;
    const float inv = lnorm > 0.f ? a.v_scale / lnorm : 0.f;   // v_scale: E4M3 caches
    const float lse2 = lsum > 0.f ? M + lg2(lsum) : -INFINITY;
    const int rr = rho0 + rho;
    const int i = rr / group;
    const int h = g * group + rr % group;
    if (split_mode || a.cascade != 0) {
      // a split partial, or a cascade partial (prefix split s, or the own-key
      // slot of a request)
      const int64_t w = part_row(a, a.cascade == 2 ? a.cascade_slot : s, r, q0 + i, i, h);
#pragma unroll
      for (int e = 0; e < C::kDPL; ++e) o[e] *= inv;
      store_partial<C::kDPL>(a.ws_o + w * D + lane * C::kDPL, o);
      if (lane == 0) a.ws_lse[w] = lse2;
    } else {
      const int64_t t = q0 + i;
      const int64_t base = (t * a.hq + h) * D + lane * C::kDPL;
      if constexpr (sizeof(QT) == 2 && C::kDPL == 4) {
        // four bf16 outputs of the lane in one 8-byte store
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + base) =
            make_uint2(pack_bf16x2(o[0] * inv, o[1] * inv), pack_bf16x2(o[2] * inv, o[3] * inv));
      } else {
#pragma unroll
        for (int e = 0; e < C::kDPL; ++e) store_elem<QT>(a.out, base + e, o[e] * inv);
      }
      if (a.lse_out != nullptr && lane == 0) a.lse_out[t * a.hq + h] = lse2 * kLn2;
    }
  }
}

// Decode rows per request the combine grid covers: no row index reaches
// max_query_len, and decode-class requests have at most kDecodeMaxQ.
__host__ __device__ __forceinline__ int combine_rows(int max_query_len) {
  return max_query_len < 1 ? 1 : (max_query_len > kDecodeMaxQ ? kDecodeMaxQ : max_query_len);
}

// Log-sum-exp merge of the split partials: for each (request, decode row,
// q head), M = max_s lse_s, w_s = 2^(lse_s - M), o = sum_s w_s o_s / sum_s w_s.
// One CTA of 4 warps per row: warp w takes splits s = w, w + 4, ...; all of a
// warp's partial loads are issued before any is used.
template <typename T, int D>
__global__ void __launch_bounds__(128) combine_kernel(const AttnArgs a) {
  constexpr int kDPL = D / 32;
  // per-warp sums, rows padded to keep each lane's slice 16-byte aligned
  __shared__ __align__(16) float red[4][D + 4];
  // the next kernel may launch at once; its dependency wait still returns only
  // after this grid completes
  pdl_launch_dependents();
  pdl_wait_primary();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t item = blockIdx.x;
  const int h = static_cast<int>(item % a.hq);
  const int64_t ri = item / a.hq;
  const int qrows = combine_rows(a.max_query_len);
  const int i = static_cast<int>(ri % qrows);
  const int r = static_cast<int>(ri / qrows);
  if (r >= a.num_seqs) return;
  const int S = a.num_splits;                          // <= kMaxSplits = 64
  // workspace row of partial s, by (request, decode row)
  auto prow = [&](int sp) -> int64_t { return ws_row(a, sp, r, i, h); };
  // Partials are loaded before the row is known to exist (rows of requests
  // that are not decode-class hold stale data and are simply not stored), so
  // the metadata and workspace loads are in flight together.
  const int q0 = __ldg(a.qsl + r);
  const int q1 = __ldg(a.qsl + r + 1);
  const int L = __ldg(a.seq_lens + r);
  const float l0 = lane < S ? a.ws_lse[prow(lane)] : -INFINITY;
  const float l1 = lane + 32 < S ? a.ws_lse[prow(lane + 32)] : -INFINITY;
  constexpr int kMaxPer = kMaxSplits / 4;
  float part[kMaxPer][kDPL];
#pragma unroll
  for (int u = 0; u < kMaxPer; ++u) {
    const int sp = warp + 4 * u;
    if (sp < S) {
      // one 16-byte (D 128) or 8-byte (D 64) load per partial: a row is D
      // floats, so the lane's slice is aligned
      const float* src = a.ws_o + prow(sp) * D + lane * kDPL;
      if constexpr (kDPL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        part[u][0] = v.x;
        part[u][1] = v.y;
        part[u][2] = v.z;
        part[u][3] = v.w;
      } else if constexpr (kDPL == 2) {
        const float2 v = *reinterpret_cast<const float2*>(src);
        part[u][0] = v.x;
        part[u][1] = v.y;
      } else {
#pragma unroll
        for (int e = 0; e < kDPL; ++e) part[u][e] = src[e];
      }
    }
  }
  {
    const int n = q1 - q0;
    if (n <= 0 || n > kDecodeMaxQ || i >= n || q0 < 0 || q1 > a.num_tokens || n > L) return;
  }
  float M = warp_max(fmaxf(l0, l1));
  const float w0 = M == -INFINITY ? 0.f : ex2(l0 - M);
  const float w1 = M == -INFINITY ? 0.f : ex2(l1 - M);
  const float wsum = warp_sum(w0 + w1);
  float o[kDPL];
#pragma unroll
  for (int e = 0; e < kDPL; ++e) o[e] = 0.f;
#pragma unroll
  for (int u = 0; u < kMaxPer; ++u) {
    const int sp = warp + 4 * u;
    if (sp < S) {
      const float f = __shfl_sync(0xffffffffu, sp < 32 ? w0 : w1, sp & 31);
#pragma unroll
      for (int e = 0; e < kDPL; ++e) o[e] = fmaf(f, part[u][e], o[e]);
    }
  }
#pragma unroll
  for (int e = 0; e < kDPL; ++e) red[warp][lane * kDPL + e] = o[e];
  __syncthreads();
  if (warp != 0) return;
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int64_t t = q0 + i;
  const int64_t base = (t * a.hq + h) * D + lane * kDPL;
  float v[kDPL];
  if constexpr (kDPL == 4) {
    float4 s4 = *reinterpret_cast<const float4*>(&red[0][lane * 4]);
#pragma unroll
    for (int w = 1; w < 4; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(&red[w][lane * 4]);
      s4.x += x.x; s4.y += x.y; s4.z += x.z; s4.w += x.w;
    }
    v[0] = s4.x * inv; v[1] = s4.y * inv; v[2] = s4.z * inv; v[3] = s4.w * inv;
  } else {
#pragma unroll
    for (int e = 0; e < kDPL; ++e) {
      const int col = lane * kDPL + e;
      v[e] = (red[0][col] + red[1][col] + red[2][col] + red[3][col]) * inv;
    }
  }
  if constexpr (sizeof(T) == 2 && kDPL == 4) {
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + base) =
        make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
  } else if constexpr (sizeof(T) == 2 && kDPL == 2) {
    *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.out) + base) = pack_bf16x2(v[0], v[1]);
  } else {
#pragma unroll
    for (int e = 0; e < kDPL; ++e) store_elem<T>(a.out, base + e, v[e]);
  }
  if (a.lse_out != nullptr && lane == 0)
    a.lse_out[t * a.hq + h] = wsum > 0.f ? (M + lg2(wsum)) * kLn2 : -INFINITY;
}

// The shared-prefix merge (cascade pass 3): for each (token, q head) row,
// M = max_s lse_s, w_s = 2^(lse_s - M), o = sum_s w_s o_s / sum_s w_s over the
// prefix splits' partials and the request's own-key partial.  One warp per
// row, four rows per CTA: a row's few partials (prefix splits + 1) fit one
// warp's registers, so there is no cross-warp reduction; the lane's slice of
// every partial of a chunk is loaded before any is used.
template <typename T, int D>
__global__ void __launch_bounds__(128) merge_rows_kernel(const AttnArgs a) {
  constexpr int kDPL = D / 32;
  constexpr int kChunk = 16;                           // partial loads in flight per lane
  pdl_launch_dependents();
  pdl_wait_primary();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * 4 + warp;
  if (item >= a.num_tokens * a.hq) return;
  const int64_t tok = item / a.hq;
  const int h = static_cast<int>(item % a.hq);
  const int S = a.num_splits;                          // <= kMaxSplits = 64
  auto prow = [&](int sp) -> int64_t {
    return (static_cast<int64_t>(sp) * a.num_tokens + tok) * a.hq + h;
  };
  auto load = [&](int sp, float (&v)[kDPL]) {
    const float* src = a.ws_o + prow(sp) * D + lane * kDPL;
    if constexpr (kDPL == 4) {
      const float4 x = *reinterpret_cast<const float4*>(src);
      v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2*>(src);
      v[0] = x.x; v[1] = x.y;
    }
  };
  const int q1 = __ldg(a.qsl + a.num_seqs);
  const float l0 = lane < S ? a.ws_lse[prow(lane)] : -INFINITY;
  const float l1 = lane + 32 < S ? a.ws_lse[prow(lane + 32)] : -INFINITY;
  float part[kChunk][kDPL];
#pragma unroll
  for (int u = 0; u < kChunk; ++u)
    if (u < S) load(u, part[u]);
  if (tok >= q1) return;                               // padding rows: no own-key partial
  const float M = warp_max(fmaxf(l0, l1));
  const float w0 = M == -INFINITY ? 0.f : ex2(l0 - M);
  const float w1 = M == -INFINITY ? 0.f : ex2(l1 - M);
  const float wsum = warp_sum(w0 + w1);
  float o[kDPL];
#pragma unroll
  for (int e = 0; e < kDPL; ++e) o[e] = 0.f;
  for (int c0 = 0; c0 < S; c0 += kChunk) {
    if (c0 > 0) {
#pragma unroll
      for (int u = 0; u < kChunk; ++u)
        if (c0 + u < S) load(c0 + u, part[u]);
    }
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      const int sp = c0 + u;
      if (sp < S) {
        const float f = __shfl_sync(0xffffffffu, sp < 32 ? w0 : w1, sp & 31);
#pragma unroll
        for (int e = 0; e < kDPL; ++e) o[e] = fmaf(f, part[u][e], o[e]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int64_t base = (tok * a.hq + h) * D + lane * kDPL;
  if constexpr (sizeof(T) == 2 && kDPL == 4) {
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + base) =
        make_uint2(pack_bf16x2(o[0] * inv, o[1] * inv), pack_bf16x2(o[2] * inv, o[3] * inv));
  } else if constexpr (sizeof(T) == 2) {
    *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.out) + base) =
        pack_bf16x2(o[0] * inv, o[1] * inv);
  } else {
#pragma unroll
    for (int e = 0; e < kDPL; ++e) store_elem<T>(a.out, base + e, o[e] * inv);
  }
  if (a.lse_out != nullptr && lane == 0)
    a.lse_out[tok * a.hq + h] = wsum > 0.f ? (M + lg2(wsum)) * kLn2 : -INFINITY;
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
template <typename T, int D, int R, bool SPEC = false>
static cudaError_t ensure_smem_attr() {
  using Sm = DecodeSmem<T, D, R>;
  static unsigned done = 0;                 // one bit per device already configured
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 32 && ((done >> dev) & 1u)) return cudaSuccess;
  e = cudaFuncSetAttribute(decode_kernel<T, D, R, SPEC>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, Sm::kAlloc);
  // the tensor-core build runs two CTAs per SM: ask for the largest
  // shared-memory carveout
  if (e == cudaSuccess && DecodeCfg<T, D, R>::kMma)
    e = cudaFuncSetAttribute(decode_kernel<T, D, R, SPEC>,
                             cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e == cudaSuccess && dev < 32) done |= 1u << dev;
  return e;
}

template <typename T, int D, int R, bool SPEC>
static cudaError_t launch_decode_t(const AttnArgs& a, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, int row_tiles, bool pdl,
                                   cudaStream_t stream) {
  using C = DecodeCfg<T, D, R>;
  using Sm = DecodeSmem<T, D, R>;
  cudaError_t e = ensure_smem_attr<T, D, R, SPEC>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.hkv * a.num_splits), static_cast<unsigned>(row_tiles),
                     static_cast<unsigned>(a.num_seqs));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = Sm::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<T, D, R, SPEC>, kmap, vmap, a);
}

template <typename T, int D>
static cudaError_t launch_decode_d(const AttnArgs& a, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, int R, int row_tiles, bool pdl,
                                   cudaStream_t stream) {
  switch (R) {
    case 4:
      // speculative first blocks only for split launches without a window
      // (their hinted block range ignores it)
      return a.num_splits > 1 && a.window == 0 && a.cascade == 0
                 ? launch_decode_t<T, D, 4, true>(a, kmap, vmap, row_tiles, pdl, stream)
                 : launch_decode_t<T, D, 4, false>(a, kmap, vmap, row_tiles, pdl, stream);
    case 8: return launch_decode_t<T, D, 8, false>(a, kmap, vmap, row_tiles, pdl, stream);
    default: return launch_decode_t<T, D, 16, false>(a, kmap, vmap, row_tiles, pdl, stream);
  }
}

// Resident decode CTAs per SM the split rule plans for: two for the
// tensor-core build, one for the CUDA-core build.
int decode_ctas_per_sm(ElemType et, int head_dim) {
  const bool mma = (et == ElemType::kBf16 && (head_dim == 64 || head_dim == 128)) ||
                   (et == ElemType::kE4m3 && head_dim == 128);
  return mma ? 2 : 1;
}

// Whether the decode kernel for this cache type and head_dim takes its K/V
// boxes in the 128B-swizzled layout (the tensor-core build) rather than as
// whole unswizzled rows.
bool decode_swizzled(ElemType et, int head_dim) {
  if (et == ElemType::kBf16) return head_dim == 64 || head_dim == 128;
  if (et == ElemType::kE4m3) return head_dim == 128;
  return false;
}

// Rows per CTA tile: one token's GQA group rounded up to 4/8/16 rows, so a
// single-token decode always takes the tile shape it needs (requests with a
// few new tokens get one tile per token); 16 when the CUDA-core path also
// runs long requests.
int decode_rows_per_tile(int group, int max_query_len, bool long_rows) {
  (void)max_query_len;
  if (long_rows) return 16;
  return group <= 4 ? 4 : (group <= 8 ? 8 : 16);
}

cudaError_t launch_decode(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          ElemType et, int head_dim, bool pdl, cudaStream_t stream) {
  const int R = decode_rows_per_tile(a.group, a.max_query_len, a.long_rows != 0);
  const int qmax = a.long_rows ? a.max_query_len : min(a.max_query_len, kDecodeMaxQ);
  const int row_tiles = (a.group * (qmax < 1 ? 1 : qmax) + R - 1) / R;
  if (row_tiles > 65535 || a.num_seqs > 65535) return cudaErrorInvalidConfiguration;
  if (et == ElemType::kBf16) {
    return head_dim == 128 ? launch_decode_d<__nv_bfloat16, 128>(a, kmap, vmap, R, row_tiles, pdl, stream)
                           : launch_decode_d<__nv_bfloat16, 64>(a, kmap, vmap, R, row_tiles, pdl, stream);
  }
  if (et == ElemType::kE4m3) {
    return head_dim == 128 ? launch_decode_d<e4m3_t, 128>(a, kmap, vmap, R, row_tiles, pdl, stream)
                           : launch_decode_d<e4m3_t, 64>(a, kmap, vmap, R, row_tiles, pdl, stream);
  }
  return head_dim == 128 ? launch_decode_d<float, 128>(a, kmap, vmap, R, row_tiles, pdl, stream)
                         : launch_decode_d<float, 64>(a, kmap, vmap, R, row_tiles, pdl, stream);
}

// The combine writes out in the query's type: bf16 for bf16 and E4M3 caches.
cudaError_t launch_combine(const AttnArgs& a, ElemType et, int head_dim, cudaStream_t stream) {
  const int64_t items = a.cascade == 3
                            ? a.num_tokens * a.hq
                            : static_cast<int64_t>(a.num_seqs) * combine_rows(a.max_query_len) * a.hq;
  if (items < 1 || items > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(items));
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.cascade == 3) {
    // one warp per (token, head) row, four rows per CTA
    cfg.gridDim = dim3(static_cast<unsigned>((items + 3) / 4));
    if (et != ElemType::kF32)
      return head_dim == 128 ? cudaLaunchKernelEx(&cfg, merge_rows_kernel<__nv_bfloat16, 128>, a)
                             : cudaLaunchKernelEx(&cfg, merge_rows_kernel<__nv_bfloat16, 64>, a);
    return head_dim == 128 ? cudaLaunchKernelEx(&cfg, merge_rows_kernel<float, 128>, a)
                           : cudaLaunchKernelEx(&cfg, merge_rows_kernel<float, 64>, a);
  }
  if (et != ElemType::kF32) {
    return head_dim == 128 ? cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16, 128>, a)
                           : cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16, 64>, a);
  }
  return head_dim == 128 ? cudaLaunchKernelEx(&cfg, combine_kernel<float, 128>, a)
                         : cudaLaunchKernelEx(&cfg, combine_kernel<float, 64>, a);
}

}  // namespace pkv
