// Tiled causal prefill on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// "Inside the engine: kernels, CUDA graphs and the life of a request":
//   * "Never materialise the TxT matrix" - a block of queries stays on chip
//     while K/V tiles stream past it; a running max m and denominator l are
//     kept per row and the accumulator is rescaled by e^(m_old - m_new)
//     whenever the max moves;
//   * "Prefill has a full grid ..." - prefill has a tile per 128 queries, so it
//     parallelises without splitting the key axis;
//   * "Attention over a block table, not a contiguous tensor" - every K/V tile
//     is gathered block by block through the request's block table.
//
// One CTA = (tile of 128 query rows of one request, two query heads that share
// a KV head), so every K/V tile feeds two S = Q K^T products.
//   warps 0-3 and 4-7: one softmax warpgroup per query head, one query row per
//     thread - the S row is read from TMEM (four 32-column loads, one wait),
//     masked only on tiles that cross the causal edge, exponentiated in the
//     log2 domain and written back into TMEM as bf16 P, which aliases the
//     first 64 columns of its own S;
//   warp 8: TMA producer - both heads' Q tiles once (64-column boxes, 128B
//     swizzle), then per 128-key tile 8 blocks x 2 column halves of K and of V
//     through the block table into a 2-stage ring, K and V with separate
//     barriers so S can start before V lands;
//   warp 9: allocates 512 TMEM columns (S/P and O per head) and one lane issues
//     tcgen05.mma in a ping-pong order - P0 V(k), S0(k+1), P1 V(k), S1(k+1) - so
//     one head's softmax overlaps the other head's MMAs; P.V takes P straight
//     from TMEM as the A operand, V from shared memory (MN-major).
// Shared-prefix (cascade) mode: the CTA's 256 rows are (token, query head)
// pairs of one KV head - 256 / group tokens of the batch, each with its whole
// GQA group, loaded by one TMA box per 128 rows - over one split of the
// shared prefix's keys, unmasked (every row sits after the prefix); rows
// write fp32 partials (o, log2-domain lse) to the workspace for the merge.
// The running max is a lagged reference: a row moves it (and rescales its O
// accumulator and l) only when a tile's max exceeds it by more than 8 log2
// units, so every p = 2^(s - reference) stays at most 2^8 - far from overflow
// in fp32 and in the bf16 P - and o = acc / l does not depend on which
// reference acc and l share: the same online softmax with fewer O rescales.
//
// E4M3 caches (head_dim 128): a K (or V) tile arrives as 16 KB of 8-bit codes
// in the second half of its 32 KB ring slot, as early as a bf16 tile would,
// and two more warps (10, 11) widen it in place, exactly, to the f16 tile the
// MMAs read (the bf16 tiles' layout), zeroing key rows past the context: each
// thread loads all its codes, the two warps meet at a named barrier, then
// write.  The MMAs run as kind::f16 with f16 operands: each softmax thread
// first rewrites its bf16 Q row in place as f16 scaled by 2^-e, e chosen per
// row so the row's largest magnitude lands in [2^14, 2^15) (exact for every
// element within 2^31 of the largest), and scales its scores back by 2^e
// together with softmax_scale * k_scale; P goes to TMEM as f16 and v_scale
// joins the final 1 / l.
#include <algorithm>

#include "common.cuh"

namespace pkv {

namespace {

constexpr int kQRows = 128;          // query rows per tile
constexpr int kKeys = 128;           // keys per K/V tile (8 blocks)
constexpr int kStages = 2;
constexpr int kHalf = 16384;         // 64 columns of a 128-row 16-bit tile (128-byte rows)
constexpr int kCodeBytes = kKeys * 128;   // one K (or V) tile of E4M3 codes at head_dim 128
static_assert(kCodeBytes == kHalf, "a code tile fills the second half of its ring slot");

// 2 softmax warpgroups + producer warp + MMA warp (+ 2 widening warps for
// E4M3: 12 warps keep three per SM sub-partition and 168 registers a thread)
__host__ __device__ constexpr int threads_for(bool f8) { return f8 ? 384 : 320; }

// shared-memory layout (bytes from a 1024-aligned base)
constexpr int kOffQ = 0;                                  // 2 query tiles x 2 halves
constexpr int kOffKV = 4 * kHalf;                         // stages x (K 2 halves, V 2 halves)
constexpr int kStageBytes = 4 * kHalf;
__host__ __device__ constexpr int off_bar(bool) { return kOffKV + kStages * kStageBytes; }
// q, k_full[], v_full[], k_empty[], v_empty[], s[2], p[2], o[2]; E4M3 adds
// code_full[K, V][stage] and q_ready
__host__ __device__ constexpr int num_bars(bool f8) { return 1 + 4 * kStages + 6 + (f8 ? 5 : 0); }
__host__ __device__ constexpr int off_misc(bool f8) { return off_bar(f8) + num_bars(f8) * 8; }
__host__ __device__ constexpr int smem_alloc(bool f8) { return off_misc(f8) + 32 + 1024; }
static_assert(smem_alloc(true) <= 232448, "E4M3 prefill shared memory");
// TMEM: S_t in columns [128 t, 128 t + 128) - its first 64 columns take P_t
// (bf16 pairs) once the scores are read - and O_t in [256 + 128 t, ...).
constexpr int kTmemCols = 512;
constexpr float kRescaleSlack = 8.f; // log2 units the reference max may lag the true max

// shared-memory matrix descriptor, 128B swizzle (sm_100 format, version 1)
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFF);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// instruction descriptor, kind::f16: A and B both bf16 (or both f16), fp32
// accumulator, M x N
__device__ __forceinline__ uint32_t idesc_f16kind(int m, int n, int b_mn_major, bool f16) {
  const uint32_t ab = f16 ? 0u : (1u << 7) | (1u << 10);
  return (1u << 4) | ab | (static_cast<uint32_t>(b_mn_major) << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(accumulate));
}

// O += A B with A (M x K, bf16 pairs per column) read from TMEM
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Issue a load of 32 consecutive fp32 columns of this thread's TMEM lane; the
// registers are valid only after tmem_wait_ld.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Wait for this thread's outstanding TMEM loads.  The registers pass through
// the wait as operands, so no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  tmem_ld32_issue(taddr, r);
  tmem_wait_ld(r);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

__device__ __forceinline__ float ex2f_(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2f_(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (sm_100+: one instruction for two lanes of fp32 math) and
// a three-input max, to thin out the softmax's instruction stream.
__device__ __forceinline__ unsigned long long pair(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpair(unsigned long long v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ unsigned long long fma_pair(unsigned long long a, unsigned long long b,
                                                       unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long add_pair(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// four E4M3 codes of a word (element 0 in the low byte) -> f16 pairs (0, 1)
// and (2, 3); every E4M3 value is an f16 value, so the widening is exact
__device__ __forceinline__ void widen4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 c0, c1;\n\tmov.b32 {c0, c1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, c0;\n\tcvt.rn.f16x2.e4m3x2 %1, c1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
// 16-byte shared-memory load and store (one 128-bit access a lane)
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
// bf16 pair -> fp32 pair scaled by f (exact: a power of two in range)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float f) {
  return pack_f16(__uint_as_float(w << 16) * f, __uint_as_float(w & 0xFFFF0000u) * f);
}

}  // namespace

// D: head_dim, 128 or 64.  The layouts are those of D = 128 (two 64-column
// halves of Q, K and V, O_t in 128 TMEM columns); D = 64 fills one half of
// each and the first 64 columns of O_t.  F8: an E4M3 cache (D = 128).
template <int D, bool F8>
__global__ void __launch_bounds__(threads_for(F8), 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const AttnArgs a) {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static_assert(!F8 || D == 128, "E4M3 tiles at head_dim 128");
  constexpr int kThreads = threads_for(F8);
  constexpr int kH = D / 64;                             // 64-column halves of a row
  constexpr int kOC = D / 32;                            // 32-column chunks of an O row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + off_bar(F8));
  uint64_t* bar_q = bars;
  // K and V halves of a stage have their own barriers: K(k) is free once
  // S1(k) has run, V(k) only after PV1(k), so K(k+2) can load earlier.
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + kStages;
  uint64_t* k_empty = v_full + kStages;
  uint64_t* v_empty = k_empty + kStages;
  uint64_t* bar_s = bars + 1 + 4 * kStages;              // [tile]
  uint64_t* bar_p = bar_s + 2;                           // [tile]
  uint64_t* bar_o = bar_s + 4;                           // [tile]
  // E4M3: a stage's codes landed ([part * kStages + stage], part 0 K, 1 V;
  // k_full / v_full then mean widened); Q rewritten as f16
  uint64_t* code_full = bars + num_bars(false);
  uint64_t* bar_qr = code_full + 2 * kStages;
  int* misc = reinterpret_cast<int*>(smem + off_misc(F8));   // [0] request, [1] tile, [2] tmem

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool packed = a.cascade == 1;                    // shared-prefix mode
  // The grid is one-dimensional with the head pair (shared-prefix mode: the
  // kv head and prefix split) varying fastest, so every head pair's heaviest
  // query tiles are dispatched in the first waves (longest work first) and
  // the CTAs reading the same K/V tiles run side by side.
  // Tile-pair mode (an odd GQA group, where two query heads of one KV head
  // cannot pair up): both softmax warpgroups take query head h0, over the
  // consecutive query tiles 2u and 2u + 1 of one request.
  const bool pairs = !packed && a.pair_tiles != 0;
  const int ys = packed ? a.hkv * a.num_splits : (pairs ? a.hq : a.hq / 2);
  const int yidx = static_cast<int>(blockIdx.x % static_cast<unsigned>(ys));
  // query heads h0, h0 + 1 (same KV head), or h0 alone in tile-pair mode
  const int h0 = packed ? 0 : (pairs ? yidx : 2 * yidx);
  const int tglob = static_cast<int>(blockIdx.x / static_cast<unsigned>(ys));

  // defer_wait: launched behind the decode kernel of the same call, whose
  // CTAs release this grid only after their own dependency wait, so every
  // input read here is already complete; the wait moves to each CTA's exit,
  // keeping the call complete only when both grids are, and the prefill
  // tiles run in the decode grid's tail
  if (!a.defer_wait) pdl_wait_primary();
  pdl_launch_dependents();

  // ---- which (request, query tile) this CTA owns: warp 0 scans the long
  //      requests' tile counts (ceil(n / 128) for n > the decode bound) ----
  if (packed) {
    if (threadIdx.x == 0) {
      misc[0] = 0;
      misc[1] = tglob;
    }
  } else if (warp == 0) {
    int base = 0, found_r = -1, found_t = 0;
    for (int r0 = 0; r0 < a.num_seqs && found_r < 0; r0 += 32) {
      const int r = r0 + lane;
      int nt = 0;
      if (r < a.num_seqs) {
        const int n = __ldg(a.qsl + r + 1) - __ldg(a.qsl + r);
        nt = n > kDecodeMaxQ ? (n + kQRows - 1) / kQRows : 0;
        if (pairs) nt = (nt + 1) / 2;                    // units: pairs of tiles
      }
      int inc = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      const int total = __shfl_sync(0xffffffffu, inc, 31);
      if (tglob < base + total) {
        const unsigned hit = __ballot_sync(0xffffffffu, base + inc > tglob);
        const int src = __ffs(hit) - 1;
        const int excl = __shfl_sync(0xffffffffu, inc - nt, src);
        const int ntr = __shfl_sync(0xffffffffu, nt, src);
        found_r = r0 + src;
        found_t = ntr - 1 - (tglob - base - excl);        // last (heaviest) tiles first
      }
      base += total;
    }
    if (lane == 0) {
      misc[0] = found_r;
      misc[1] = found_t;
    }
  }
  __syncthreads();
  const int r = misc[0];
  if (r < 0) {                                           // past the last tile
    if (a.defer_wait) pdl_wait_primary();
    return;
  }
  const int tile = misc[1];
  const int q0 = packed ? 0 : __ldg(a.qsl + r);
  const int q1 = packed ? static_cast<int>(a.num_tokens) : __ldg(a.qsl + r + 1);
  const int n = q1 - q0;
  const int L = packed ? a.prefix_len : __ldg(a.seq_lens + r);
  if (q0 < 0 || q1 > a.num_tokens || (n > L && !packed) || n > a.max_query_len) {
    if (threadIdx.x == 0 && h0 == 0) raise_flag(a.flag, PKV_FLAG_BAD_LENGTHS);
    if (a.defer_wait) pdl_wait_primary();
    return;
  }
  const int g = packed ? yidx % a.hkv : h0 / a.group;
  const int split = packed ? yidx / a.hkv : 0;
  const int tok_per_tile = kQRows / a.group;             // packed: tokens per 128-row tile
  // first row of the unit (its first tile), and the unit's last real row
  const int i0 = (pairs ? 2 * tile : tile) * kQRows;
  const int i_hi = min(i0 + (pairs ? 2 : 1) * kQRows, n) - 1;
  const int kv_len = a.causal ? (L - n + i_hi + 1) : L;
  const int nblk_ctx = (kv_len + kBlock - 1) / kBlock;
  if ((L + kBlock - 1) / kBlock > a.max_blocks_per_seq) {
    if (threadIdx.x == 0) raise_flag(a.flag, PKV_FLAG_BAD_LENGTHS);
    if (a.defer_wait) pdl_wait_primary();
    return;
  }
  // sliding window: key tiles wholly below the first row's window start are
  // skipped; kt below counts the remaining tiles from kt_base
  int kt_base =
      a.window > 0 ? max(0, L - n + i0 - a.window + 1) / kKeys : 0;
  int ntk = (kv_len + kKeys - 1) / kKeys - kt_base;
  if (packed) {
    // this CTA's split of the prefix's key tiles
    const int per = (ntk + a.num_splits - 1) / a.num_splits;
    kt_base = min(split * per, ntk);
    ntk = min(per, ntk - kt_base);
    if (ntk <= 0) {
      // an empty split: partial o = 0, lse = -inf for every row it owns
      for (int rr = threadIdx.x; rr < 2 * kQRows; rr += kThreads) {
        const int64_t rho = static_cast<int64_t>(tile) * 2 * kQRows + rr;
        const int64_t tk = rho / a.group;
        if (tk >= a.num_tokens) continue;
        const int64_t w = (static_cast<int64_t>(split) * a.num_tokens + tk) * a.hq +
                          g * a.group + rho % a.group;
        for (int c = 0; c < D; ++c) a.ws_o[w * D + c] = 0.f;
        a.ws_lse[w] = -INFINITY;
      }
      if (a.defer_wait) pdl_wait_primary();
      return;
    }
  }

  // ---- barriers and TMEM ----
  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < kStages; ++s) {
      // E4M3: a stage is full once both widening warps have written it
      mbar_init(&k_full[s], F8 ? 2 : 1);
      mbar_init(&v_full[s], F8 ? 2 : 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_s[i], 1);
      mbar_init(&bar_p[i], kQRows);
      mbar_init(&bar_o[i], 1);
    }
    if (F8) {
      for (int i = 0; i < 2 * kStages; ++i) mbar_init(&code_full[i], 1);
      mbar_init(bar_qr, 2 * kQRows);
    }
    fence_mbar_init();
  }
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&misc[2])),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = static_cast<uint32_t>(misc[2]);
  bool ok = true;

  if (warp == 8) {
    // ================= TMA producer =================
    const uint64_t pol_kv = l2_policy_evict_last();      // K/V tiles are re-read by other CTAs
    const int32_t* table = a.block_table + static_cast<int64_t>(r) * a.max_blocks_per_seq;
    const int oob = static_cast<int>(a.num_blocks * kBlock);   // a slot past the cache
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      mbar_arrive_expect_tx(bar_q, 2 * kH * kHalf);
      const uint64_t pol_q = l2_policy_evict_first();
      for (int t = 0; t < 2; ++t)
        for (int hh = 0; hh < kH; ++hh) {
          if (packed)   // 128 rows = tok_per_tile tokens x the GQA group of KV head g
            tma_load_3d(smem + kOffQ + (2 * t + hh) * kHalf, &qmap, bar_q, hh * 64, g * a.group,
                        (2 * tile + t) * tok_per_tile, pol_q);
          else
            tma_load_3d(smem + kOffQ + (2 * t + hh) * kHalf, &qmap, bar_q, hh * 64,
                        pairs ? h0 : h0 + t, q0 + i0 + (pairs ? t * kQRows : 0), pol_q);
        }
    }
    int kt = 0;
    for (; kt < ntk; ++kt) {
      const int st = kt % kStages;
      const int blk = (kt_base + kt) * (kKeys / kBlock) + (lane & 7);
      int32_t ent = -1;
      if (lane < kKeys / kBlock && blk < nblk_ctx) {
        ent = __ldg(table + blk);
        if (ent < 0 || ent >= a.num_blocks) {
          raise_flag(a.flag, PKV_FLAG_BAD_BLOCK);
          ent = -1;
        }
      }
      const int slot = ent >= 0 ? ent * kBlock : oob;   // past the context: zero fill
      uint8_t* kst = smem + kOffKV + st * kStageBytes;
      // K half of the stage, then its V half, each once its previous tile is
      // done (E4M3: the codes, into the second half of the slot)
      for (int part = 0; part < 2; ++part) {
        uint64_t* fullb = F8 ? &code_full[part * kStages + st]
                             : (part == 0 ? &k_full[st] : &v_full[st]);
        uint64_t* emptyb = part == 0 ? &k_empty[st] : &v_empty[st];
        if (kt >= kStages) {
          uint32_t w = 1;
          if (lane == 0) w = mbar_wait(emptyb, ((kt / kStages) - 1) & 1) ? 1u : 0u;
          if (!__shfl_sync(0xffffffffu, w, 0)) {
            ok = false;
            break;
          }
        }
        if (lane == 0) mbar_arrive_expect_tx(fullb, F8 ? kCodeBytes : kH * kHalf);
        __syncwarp();
        if (lane < kKeys / kBlock) {
          uint8_t* dst = kst + part * 2 * kHalf;
          const CUtensorMap* map = part == 0 ? &kmap : &vmap;
          if constexpr (F8) {
            tma_load_3d(dst + kHalf + lane * (kBlock * 128), map, fullb, 0, g, slot, pol_kv);
          } else {
            for (int hh = 0; hh < kH; ++hh)
              tma_load_3d(dst + hh * kHalf + lane * (kBlock * 128), map, fullb, hh * 64, g, slot,
                          pol_kv);
          }
        }
        __syncwarp();
      }
      if (!ok) break;
    }
    if (!ok && lane == 0) raise_flag(a.flag, PKV_FLAG_TIMEOUT);
    // let every issued load land before the CTA can exit
    if (lane == 0) {
      for (int kk = max(0, kt - kStages); kk < min(kt + 1, ntk); ++kk) {
        const int sk = kk % kStages;
        if (!mbar_wait(F8 ? &code_full[sk] : &k_full[sk], (kk / kStages) & 1)) break;
        if (kk < kt &&
            !mbar_wait(F8 ? &code_full[kStages + sk] : &v_full[sk], (kk / kStages) & 1))
          break;
      }
      mbar_wait(bar_q, 0);
    }
  } else if (warp == 9) {
    // ================= MMA issuer (one lane) =================
    // Per K/V tile k: PV0(k), S0(k+1), PV1(k), S1(k+1).  The tensor pipe runs
    // one issuer's MMAs in order, so S_t(k+1) overwrites the P_t columns only
    // after PV_t(k) has read them; group 0's softmax of tile k+1 overlaps
    // group 1's P.V of tile k and the reverse.
    if (lane == 0) {
      const uint32_t id_s = idesc_f16kind(kQRows, kKeys, 0, F8);
      const uint32_t id_o = idesc_f16kind(kQRows, D, 1, F8);
      // Descriptors are built once; a step only adds its byte offset >> 4 to
      // the start-address field (every address stays below 256 KB, so the
      // 14-bit field never carries).
      const uint32_t kv_addr0 = smem_u32(smem + kOffKV);
      const uint64_t dq = sdesc(smem_u32(smem + kOffQ), 16, 1024);
      const uint64_t dk = sdesc(kv_addr0, 16, 1024);
      const uint64_t dv = sdesc(kv_addr0 + 2 * kHalf, kHalf, 1024);
      auto issue_s = [&](int t, int kt) {                // S_t = Q_t K^T, D / 16 steps
        const uint64_t a0 = dq + static_cast<uint64_t>((t * 2 * kHalf) >> 4);
        const uint64_t b0 = dk + static_cast<uint64_t>(((kt % kStages) * kStageBytes) >> 4);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t off = static_cast<uint64_t>(((k >> 2) * kHalf + (k & 3) * 32) >> 4);
          umma(tbase + t * kKeys, a0 + off, b0 + off, id_s, k > 0);
        }
        umma_commit(&bar_s[t]);
      };
      auto issue_pv = [&](int t, int kt) {               // O_t += P_t V, 128 keys in 8 steps
        const uint64_t b0 = dv + static_cast<uint64_t>(((kt % kStages) * kStageBytes) >> 4);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          umma_ts(tbase + 2 * kKeys + t * 128, tbase + t * kKeys + k * 8,
                  b0 + static_cast<uint64_t>((k * 2048) >> 4), id_o, (kt > 0 || k > 0) ? 1u : 0u);
        umma_commit(&bar_o[t]);
      };
      auto wait_k = [&](int kt) {
        if (!mbar_wait(&k_full[kt % kStages], (kt / kStages) & 1)) return false;
        tc_fence_after();
        return true;
      };
      auto wait_v = [&](int kt) {
        if (!mbar_wait(&v_full[kt % kStages], (kt / kStages) & 1)) return false;
        tc_fence_after();
        return true;
      };
      ok = mbar_wait(F8 ? bar_qr : bar_q, 0) && wait_k(0);
      if (ok) {
        issue_s(0, 0);
        issue_s(1, 0);
        umma_commit(&k_empty[0]);
      }
      for (int kt = 0; ok && kt < ntk; ++kt) {
        const bool more = kt + 1 < ntk;
        if (!mbar_wait(&bar_p[0], kt & 1) || !wait_v(kt)) { ok = false; break; }
        tc_fence_after();
        issue_pv(0, kt);
        if (more) {
          if (!wait_k(kt + 1)) { ok = false; break; }
          issue_s(0, kt + 1);
        }
        if (!mbar_wait(&bar_p[1], kt & 1)) { ok = false; break; }
        tc_fence_after();
        issue_pv(1, kt);
        umma_commit(&v_empty[kt % kStages]);
        if (more) {
          issue_s(1, kt + 1);
          umma_commit(&k_empty[(kt + 1) % kStages]);
        }
      }
      if (!ok) raise_flag(a.flag, PKV_FLAG_TIMEOUT);
    }
    __syncwarp();
  } else if (warp >= 10) {
    if constexpr (F8) {
      // ================= E4M3 widening (warps 10, 11) =================
      // Unit i of thread ct: the 16 codes of 16-byte chunk j of key row
      // r = (ct % 8) + 8 i (the codes 128B-swizzled: chunk j of row r at
      // position j ^ (r % 8)), widened into f16 chunks 2 (j % 4) and
      // 2 (j % 4) + 1 of column half j / 4 of the slot.  The 8 lanes of a
      // shared-memory phase take 8 rows of one chunk: no bank conflicts.  All
      // the codes of a tile are read before any f16 chunk is written over them.
      const int ct = threadIdx.x - 10 * 32;
      const int j = (ct >> 3) & 7, r7 = ct & 7;
      const int c0 = 2 * (j & 3);
      for (int kt = 0; ok && kt < ntk; ++kt) {
        const int st = kt % kStages;
        const int key0 = (kt_base + kt) * kKeys;
        for (int part = 0; part < 2; ++part) {
          uint32_t w = 1;
          if (lane == 0) w = mbar_wait(&code_full[part * kStages + st], (kt / kStages) & 1);
          w = __shfl_sync(0xffffffffu, w, 0);
          // (a wait that gave up reads whatever the slot holds; nothing of it
          // is written before all_ok below stops both warps)
          const uint32_t slot_base =
              smem_u32(smem + kOffKV + st * kStageBytes + part * 2 * kHalf);
          const uint32_t src = slot_base + kHalf + ((j ^ r7) << 4) + r7 * 128;
          uint4 cw[kKeys / 8];
#pragma unroll
          for (int i = 0; i < kKeys / 8; ++i) cw[i] = lds128(src + i * 8 * 128);
          // the two warps meet once every code of the tile is read; a wait
          // that gave up in either stops both together
          uint32_t all_ok;
          asm volatile(
              "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
              "bar.red.and.pred q, 1, 64, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
              : "=r"(all_ok)
              : "r"(w)
              : "memory");
          if (!all_ok) {
            ok = false;
            break;
          }
          const uint32_t dst = slot_base + (j >> 2) * kHalf + r7 * 128;
#pragma unroll
          for (int i = 0; i < kKeys / 8; ++i) {
            const int r = r7 + 8 * i;
            uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0;  // key rows past the context: zero
            if (key0 + r < kv_len) {
              widen4(cw[i].x, o0.x, o0.y);
              widen4(cw[i].y, o0.z, o0.w);
              widen4(cw[i].z, o1.x, o1.y);
              widen4(cw[i].w, o1.z, o1.w);
            }
            sts128(dst + i * 8 * 128 + ((c0 ^ r7) << 4), o0);
            sts128(dst + i * 8 * 128 + (((c0 + 1) ^ r7) << 4), o1);
          }
          // the widened tile is read by the tensor cores (async proxy)
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(part == 0 ? &k_full[st] : &v_full[st]);
        }
      }
      if (!ok && lane == 0) raise_flag(a.flag, PKV_FLAG_TIMEOUT);
    }
  } else {
    // ================= softmax / epilogue: thread = query row of tile t =================
    const int t = warp >> 2;                             // 0: warps 0-3, 1: warps 4-7
    const int row = threadIdx.x - t * kQRows;            // 0..127 == TMEM lane
    const int h = pairs ? h0 : h0 + t;
    const int i0t = i0 + (pairs ? t * kQRows : 0);       // this warpgroup's tile
    const int i_r = i0t + row;
    const int i_eff = min(i_r, n - 1);                   // padding rows mirror the last row
    const int lim = a.causal ? (L - n + i_eff + 1) : L;  // keys < lim are visible
    const int lim_min = a.causal ? min(L - n + i0t + 1, L) : L;  // smallest lim of the tile
    // window start of the row (keys >= lo are visible) and the tile's largest
    const int lo = a.window > 0 ? L - n + i_eff - a.window + 1 : 0;
    const int lo_max = a.window > 0 ? L - n + min(i0t + kQRows, n) - 1 - a.window + 1 : 0;
    const uint32_t lane_base = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t t_s = lane_base + t * kKeys, t_o = lane_base + 2 * kKeys + t * 128;
    float sc = a.scale_log2;
    if constexpr (F8) {
      // this row of Q as f16 scaled by 2^-e, in place (each 16-byte chunk
      // keeps its swizzled position); its scores are scaled back by 2^e
      const bool got = mbar_wait(bar_q, 0);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
      } else {
        // (chunk c visited at position c ^ (row % 8): the 8 rows of a
        // shared-memory phase then hit distinct banks)
        const uint32_t qrow = smem_u32(smem + kOffQ + 2 * t * kHalf + row * 128);
        const int sw = row & 7;
        uint32_t mx = 0;                                 // two |bf16| maxima, as integers
#pragma unroll
        for (int c = 0; c < 2 * 8; ++c) {
          const uint4 v = lds128(qrow + (c >> 3) * kHalf + ((c & 7) ^ sw) * 16);
          mx = __vmaxu2(mx, __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu));
          mx = __vmaxu2(mx, __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
        }
        const uint32_t m16 = max(mx & 0xFFFFu, mx >> 16);
        // largest |q| in [2^E, 2^(E+1)): e = E - 14 (clamped so 2^-e and 2^e
        // are normal floats; a zero row takes the lower bound)
        const int e = min(max(static_cast<int>(m16 >> 7) - 127 - 14, -100), 113);
        const float down = __int_as_float((127 - e) << 23);
#pragma unroll
        for (int c = 0; c < 2 * 8; ++c) {
          const uint32_t pc = qrow + (c >> 3) * kHalf + ((c & 7) ^ sw) * 16;
          uint4 v = lds128(pc);
          v.x = bf16x2_to_f16x2_scaled(v.x, down);
          v.y = bf16x2_to_f16x2_scaled(v.y, down);
          v.z = bf16x2_to_f16x2_scaled(v.z, down);
          v.w = bf16x2_to_f16x2_scaled(v.w, down);
          sts128(pc, v);
        }
        sc *= __int_as_float((127 + e) << 23);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(bar_qr);
      }
    }
    float m = -INFINITY, l = 0.f;
    for (int kt = 0; ok && kt < ntk; ++kt) {
      const bool got = mbar_wait(&bar_s[t], kt & 1);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kKeys];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];         // all four loads in flight, one wait
        tmem_ld32_issue(t_s, r0);
        tmem_ld32_issue(t_s + 32, r1);
        tmem_ld32_issue(t_s + 64, r2);
        tmem_ld32_issue(t_s + 96, r3);
        tmem_wait_ld(r0);
        tmem_wait_ld(r1);
        tmem_wait_ld(r2);
        tmem_wait_ld(r3);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = __uint_as_float(r0[i]);
          s[32 + i] = __uint_as_float(r1[i]);
          s[64 + i] = __uint_as_float(r2[i]);
          s[96 + i] = __uint_as_float(r3[i]);
        }
      }
      const int key0 = (kt_base + kt) * kKeys;
      if (key0 + kKeys > lim_min || key0 < lo_max) {     // a tile crossing a mask edge
#pragma unroll
        for (int i = 0; i < kKeys; ++i) s[i] = (key0 + i < lim && key0 + i >= lo) ? s[i] : -INFINITY;
      }
      float mx8[8];                                      // 8 independent max chains
#pragma unroll
      for (int j = 0; j < 8; ++j) mx8[j] = fmaxf(s[j], s[j + 8]);
#pragma unroll
      for (int i = 16; i < kKeys; i += 16)               // two new scores per max
#pragma unroll
        for (int j = 0; j < 8; ++j) mx8[j] = max3(mx8[j], s[i + j], s[i + 8 + j]);
      const float mx = max3(max3(mx8[0], mx8[1], mx8[2]), max3(mx8[3], mx8[4], mx8[5]),
                            fmaxf(mx8[6], mx8[7]));
      // Scores are unscaled here; m (scaled log2 domain) is the reference max
      // the accumulator and l are kept relative to.  It moves only when the
      // row max exceeds it by more than kRescaleSlack, so p <= 2^kRescaleSlack
      // and O is rescaled rarely; o = acc / l is unchanged by the choice.
      const float mcand = fmaxf(m, mx * sc);
      const float mnew = (mcand > m + kRescaleSlack) ? mcand : m;
      const float msafe = mnew == -INFINITY ? 0.f : mnew;
      const float alpha = ex2f_(m - msafe);
      // p = 2^(s sc - m): the scaling in packed pairs, 4 independent pair sums
      const unsigned long long scp = pair(sc, sc), nmp = pair(-msafe, -msafe);
      unsigned long long ps4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int j = 0; j < kKeys / 2; ++j) {
        const float2 x = unpair(fma_pair(pair(s[2 * j], s[2 * j + 1]), scp, nmp));
        s[2 * j] = ex2f_(x.x);
        s[2 * j + 1] = ex2f_(x.y);
        ps4[j & 3] = add_pair(ps4[j & 3], pair(s[2 * j], s[2 * j + 1]));
      }
      const float2 sa = unpair(add_pair(add_pair(ps4[0], ps4[1]), add_pair(ps4[2], ps4[3])));
      const float psum = sa.x + sa.y;
      l = l * alpha + psum;
      m = mnew;
      // P row as bf16 pairs into the first 64 columns of this row's S (the
      // scores are all read); the P.V MMA takes it from there as operand A
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          w[j] = F8 ? pack_f16(s[64 * c + 2 * j], s[64 * c + 2 * j + 1])
                    : pack_bf16(s[64 * c + 2 * j], s[64 * c + 2 * j + 1]);
        tmem_st32u(t_s + 32 * c, w);
      }
      if (kt > 0) {
        // the previous P.V of this tile must be done before O is rescaled
        const bool got_o = mbar_wait(&bar_o[t], (kt - 1) & 1);
        if (!__all_sync(0xffffffffu, got_o)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < kOC; ++c) {
            float v[32];
            tmem_ld32(t_o + c * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= alpha;
            tmem_st32(t_o + c * 32, v);
          }
        }
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      // (E4M3: the widening warps zero those rows)
      if (!F8 && t == 0 && kt == ntk - 1) {
        // key rows of the last V tile past the context are zeroed, once the
        // tile's V half has landed (its barrier is separate from K's)
        const bool got_v = mbar_wait(&v_full[kt % kStages], (kt / kStages) & 1);
        if (!__all_sync(0xffffffffu, got_v)) {
          ok = false;
          break;
        }
      }
      if (!F8 && t == 0 && kt == ntk - 1 && key0 + row >= kv_len) {
        uint8_t* vrow = smem + kOffKV + (kt % kStages) * kStageBytes + 2 * kHalf + row * 128;
#pragma unroll
        for (int hh = 0; hh < kH; ++hh)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(vrow + hh * kHalf + c * 16) = make_uint4(0, 0, 0, 0);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(&bar_p[t]);
    }
    // ---- epilogue: O row / l -> output dtype, lse ----
    bool got_o = ok && mbar_wait(&bar_o[t], (ntk - 1) & 1);
    got_o = __all_sync(0xffffffffu, got_o);
    if (!got_o) {
      ok = false;
    } else {
      tc_fence_after();
      const float inv = l > 0.f ? (F8 ? a.v_scale : 1.f) / l : 0.f;
      if (packed) {
        // row (token, head) of the 256-row pair: fp32 partial and log2 lse
        const int64_t rho = (2 * static_cast<int64_t>(tile) + t) * kQRows + row;
        const int64_t tk = rho / a.group;
        const int64_t w = (static_cast<int64_t>(split) * a.num_tokens + tk) * a.hq +
                          g * a.group + rho % a.group;
#pragma unroll
        for (int c = 0; c < kOC; ++c) {
          float v[32];
          tmem_ld32(t_o + c * 32, v);
          if (tk < a.num_tokens) {
            float4* dst = reinterpret_cast<float4*>(a.ws_o + w * D + c * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(v[4 * q] * inv, v[4 * q + 1] * inv, v[4 * q + 2] * inv,
                                   v[4 * q + 3] * inv);
          }
        }
        if (tk < a.num_tokens) a.ws_lse[w] = l > 0.f ? m + lg2f_(l) : -INFINITY;
      } else {
      const bool store = i_r < n;
      __nv_bfloat16* orow =
          static_cast<__nv_bfloat16*>(a.out) + (static_cast<int64_t>(q0 + i_r) * a.hq + h) * D;
#pragma unroll
      for (int c = 0; c < kOC; ++c) {
        float v[32];
        tmem_ld32(t_o + c * 32, v);
        if (store) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_bf16(v[q * 8 + 0] * inv, v[q * 8 + 1] * inv);
            w.y = pack_bf16(v[q * 8 + 2] * inv, v[q * 8 + 3] * inv);
            w.z = pack_bf16(v[q * 8 + 4] * inv, v[q * 8 + 5] * inv);
            w.w = pack_bf16(v[q * 8 + 6] * inv, v[q * 8 + 7] * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + q * 8) = w;
          }
        }
      }
      if (store && a.lse_out != nullptr)
        a.lse_out[static_cast<int64_t>(q0 + i_r) * a.hq + h] =
            l > 0.f ? (m + lg2f_(l)) * kLn2 : -INFINITY;
      }
    }
    if (!ok && lane == 0) raise_flag(a.flag, PKV_FLAG_TIMEOUT);
  }

  // ---- teardown: every TMEM access is done before the columns are freed ----
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase),
                 "r"(kTmemCols));
  if (a.defer_wait) pdl_wait_primary();
}

// The tensor-core path pairs two query heads of one KV head per CTA, or with
// an odd GQA group two query tiles of one head (AttnArgs::pair_tiles).
bool prefill_supported(int head_dim, ElemType et, int group) {
  return ((et == ElemType::kBf16 && (head_dim == 128 || head_dim == 64)) ||
          (et == ElemType::kE4m3 && head_dim == 128)) &&
         group >= 1;
}

// Shared-prefix mode needs an even GQA group whose whole groups fill a
// 128-row tile.
bool prefill_packed_supported(int head_dim, ElemType et, int group) {
  return prefill_supported(head_dim, et, group) && group % 2 == 0 && kQRows % group == 0;
}

cudaError_t launch_prefill(const AttnArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int head_dim, ElemType et,
                           cudaStream_t stream) {
  if (!prefill_supported(head_dim, et, 1)) return cudaErrorInvalidValue;
  const bool f8 = et == ElemType::kE4m3;
  static unsigned done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 32 || !((done >> dev) & 1u)) {
    e = cudaFuncSetAttribute(prefill_kernel<128, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem_alloc(false));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(prefill_kernel<64, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem_alloc(false));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(prefill_kernel<128, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem_alloc(true));
    if (e != cudaSuccess) return e;
    if (dev < 32) done |= 1u << dev;
  }
  // upper bound on the long requests' query tiles: sum ceil(n / 128) <=
  // ceil(N / 128) + (number of long requests); shared-prefix mode: pairs of
  // 128-row (token, head) tiles per KV head, times the prefix splits
  const int64_t long_reqs = std::min<int64_t>(a.num_seqs, a.num_tokens / (kDecodeMaxQ + 1));
  const int64_t tiles = a.cascade == 1
                            ? (a.num_tokens * a.group + 2 * kQRows - 1) / (2 * kQRows)
                            : (a.num_tokens + kQRows - 1) / kQRows + long_reqs;
  const int64_t ys = a.cascade == 1 ? static_cast<int64_t>(a.hkv) * a.num_splits
                                    : (a.pair_tiles ? a.hq : a.hq / 2);
  if (tiles <= 0) return cudaSuccess;
  if (ys < 1 || tiles * ys > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * ys));      // (tile, head pair), pair fastest
  cfg.blockDim = dim3(threads_for(f8));
  cfg.dynamicSmemBytes = smem_alloc(f8);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (f8) return cudaLaunchKernelEx(&cfg, prefill_kernel<128, true>, qmap, kmap, vmap, a);
  return head_dim == 128 ? cudaLaunchKernelEx(&cfg, prefill_kernel<128, false>, qmap, kmap, vmap, a)
                         : cudaLaunchKernelEx(&cfg, prefill_kernel<64, false>, qmap, kmap, vmap, a);
}

}  // namespace pkv
