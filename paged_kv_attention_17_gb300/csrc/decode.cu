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
//   * Each of the CTA's four warps owns a private ring of shared-memory stages
//     (one mbarrier each, so every barrier has exactly one waiter and parity
//     waits cannot alias); its lane 0 issues TMA tensor loads - one 16-row box
//     per block, for K and for V - through the block table, whose entries the
//     warp prefetches 32 at a time, one per lane.
//   * A warp takes whole 32-key stages: lane j owns key j for
//     the dot products (chunk order rotated per lane, conflict-free without
//     swizzle), row max via warp shuffles, exp2 in the log2 domain, then lanes
//     own D/32 output columns for P.V.  Each warp keeps its own (m, l, acc); the
//     warps are merged through shared memory at the end (same algebra as the
//     split merge).
//   * Bounded mbarrier waits: a stuck pipeline sets PKV_FLAG_TIMEOUT and exits.
#include "common.cuh"

namespace pkv {

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

template <typename T, int D>
struct DecodeCfg {
  static constexpr int kRowBytes = D * static_cast<int>(sizeof(T));
  static constexpr int kChunks = kRowBytes / 16;          // 16-byte chunks per key row
  static constexpr int kVec = 16 / static_cast<int>(sizeof(T));
  static constexpr int kTileBlocks = 2;                   // blocks per stage
  static constexpr int kTileKeys = kTileBlocks * kBlock;  // 32: one key per lane
  static constexpr int kStageBytes = 2 * kTileKeys * kRowBytes;   // K + V
  static constexpr int kWarps = 4;                        // consumer warps per CTA
  static constexpr int kStagesRaw = 131072 / (kWarps * kStageBytes);
  static constexpr int kStagesPerWarp = kStagesRaw < 1 ? 1 : (kStagesRaw > 4 ? 4 : kStagesRaw);
  static constexpr int kStages = kWarps * kStagesPerWarp;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kDPL = D / 32;                     // output columns per lane
  static_assert((kChunks & (kChunks - 1)) == 0, "chunks per row must be a power of two");
};

template <typename T, int D, int R>
struct DecodeSmem {
  using C = DecodeCfg<T, D>;
  static constexpr int kStageArea = C::kStages * C::kStageBytes;
  static constexpr int kMergeBytes = C::kWarps * R * (D + 2) * 4;
  static constexpr int kRingBytes = kStageArea > kMergeBytes ? kStageArea : kMergeBytes;
  static constexpr int kQOff = kRingBytes;
  static constexpr int kPOff = kQOff + R * D * 4;
  static constexpr int kBarOff = kPOff + C::kWarps * C::kTileKeys * R * 4;
  static constexpr int kBytes = kBarOff + C::kStages * 8;
  static constexpr int kAlloc = kBytes + 1024;            // slack to align the base to 1 KB
};

// Position of q element (row, d) in shared memory.  fp32: plain rows.  bf16: a
// 16-byte key chunk holds 8 elements whose fp32 q counterparts (32 bytes) are
// stored as two 16-byte halves in separate regions, so the rotated chunk reads
// of 8 lanes hit 8 distinct bank groups.
template <typename T, int D>
__device__ __forceinline__ int q_index(int row, int d) {
  if constexpr (sizeof(T) == 4) {
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

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <typename T, int D, int R>
__global__ void __launch_bounds__(DecodeCfg<T, D>::kThreads)
    decode_kernel(const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const AttnArgs a) {
  using C = DecodeCfg<T, D>;
  using Sm = DecodeSmem<T, D, R>;
  constexpr int P = C::kStagesPerWarp;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* q_s = reinterpret_cast<float*>(smem + Sm::kQOff);
  float* p_s = reinterpret_cast<float*>(smem + Sm::kPOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Sm::kBarOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x % a.hkv;
  const int s = blockIdx.x / a.hkv;
  const int z = blockIdx.y;
  const int r = blockIdx.z;

  // ---- request geometry (uniform over the CTA) ----
  pdl_wait_primary();
  const int q0 = __ldg(a.qsl + r), q1 = __ldg(a.qsl + r + 1);
  const int n = q1 - q0;
  const int L = __ldg(a.seq_lens + r);
  if (n == 0) return;
  if (n < 0 || q0 < 0 || q1 > a.num_tokens || n > L || n > a.max_query_len) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && z == 0) raise_flag(a.flag, PKV_FLAG_BAD_LENGTHS);
    return;
  }
  const bool decode_class = n <= kDecodeMaxQ;
  if (!decode_class && !a.long_rows) return;          // the prefill kernel owns it
  const bool split_mode = decode_class && a.num_splits > 1;
  if (!split_mode && s != 0) return;
  const int rows_total = a.group * n;
  const int rho0 = z * R;
  if (rho0 >= rows_total) return;
  const int nrows = min(R, rows_total - rho0);
  const int i_last = (rho0 + nrows - 1) / a.group;
  const int kv_len = a.causal ? (L - n + i_last + 1) : L;
  const int nblk = (kv_len + kBlock - 1) / kBlock;
  if (nblk > a.max_blocks_per_seq) {
    if (threadIdx.x == 0) raise_flag(a.flag, PKV_FLAG_BAD_LENGTHS);
    return;
  }
  int b0 = 0, b1 = nblk;
  if (split_mode) {
    const int per = (nblk + a.num_splits - 1) / a.num_splits;
    b0 = min(s * per, nblk);
    b1 = min(b0 + per, nblk);
  }
  if (b0 >= b1) {
    // empty split: partial (o = 0, lse = -inf) so the combine weighs it 0
    for (int rho = warp; rho < nrows; rho += C::kWarps) {
      const int rr = rho0 + rho;
      const int64_t w = ws_row(a, s, r, rr / a.group, g * a.group + rr % a.group);
#pragma unroll
      for (int e = 0; e < C::kDPL; ++e) a.ws_o[w * D + lane * C::kDPL + e] = 0.f;
      if (lane == 0) a.ws_lse[w] = -INFINITY;
    }
    return;
  }
  const int ntiles = (b1 - b0 + C::kTileBlocks - 1) / C::kTileBlocks;
  // this warp's tiles: k = warp + kWarps * j, j < my_tiles
  const int my_tiles = ntiles > warp ? (ntiles - warp + C::kWarps - 1) / C::kWarps : 0;

  // ---- barriers first, so the loads can start while q is staged ----
  if (lane == 0) {
    if (warp == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    for (int i = 0; i < P; ++i) mbar_init(&full[warp * P + i], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const uint64_t pol = l2_policy_evict_first();
  const int32_t* table = a.block_table + static_cast<int64_t>(r) * a.max_blocks_per_seq;
  // Block-table entries of this warp's tiles, 16 tiles (32 blocks) per refill:
  // lane l holds block b0 + 2 * (warp + kWarps * (base + l / 2)) + l % 2.
  int32_t entry = 0;
  int entry_base = -1;
  auto issue = [&](int j) {           // warp-uniform call
    if (j >= my_tiles) return;
    if ((j & ~15) != entry_base) {
      entry_base = j & ~15;
      const int kk = warp + C::kWarps * (entry_base + (lane >> 1));
      const int bb = b0 + kk * C::kTileBlocks + (lane & 1);
      entry = (bb < b1) ? __ldg(table + bb) : 0;
    }
    const int k = warp + C::kWarps * j;
    const int first = b0 + k * C::kTileBlocks;
    const int nb = min(C::kTileBlocks, b1 - first);
    int ids[C::kTileBlocks];
#pragma unroll
    for (int u = 0; u < C::kTileBlocks; ++u)
      ids[u] = __shfl_sync(0xffffffffu, entry, ((j & 15) * 2 + u) & 31);
    if (lane == 0) {
      const int st = warp * P + (j % P);
      uint8_t* ks = smem + st * C::kStageBytes;
      uint8_t* vs = ks + C::kTileKeys * C::kRowBytes;
      fence_proxy_async_smem();       // earlier generic reads of this stage before the refill
      mbar_arrive_expect_tx(&full[st], nb * 2 * kBlock * C::kRowBytes);
#pragma unroll
      for (int u = 0; u < C::kTileBlocks; ++u) {
        if (u < nb) {
          int id = ids[u];
          if (id < 0 || id >= a.num_blocks) {
            raise_flag(a.flag, PKV_FLAG_BAD_BLOCK);
            id = 0;
          }
          tma_load_3d(ks + u * kBlock * C::kRowBytes, &kmap, &full[st], 0, g, id * kBlock, pol);
          tma_load_3d(vs + u * kBlock * C::kRowBytes, &vmap, &full[st], 0, g, id * kBlock, pol);
        }
      }
    }
    __syncwarp();
  };
#pragma unroll
  for (int j = 0; j < P; ++j) issue(j);

  // ---- stage q rows (pre-scaled into the log2 domain) ----
  for (int e = threadIdx.x; e < R * D; e += blockDim.x) {
    const int rho = e / D, d = e % D;
    float v = 0.f;
    if (rho < nrows) {
      const int rr = rho0 + rho;
      const int64_t t = q0 + rr / a.group;
      const int h = g * a.group + rr % a.group;
      v = load_elem<T>(a.q, (t * a.hq + h) * D + d) * a.scale_log2;
    }
    q_s[q_index<T, D>(rho, d)] = v;
  }
  __syncthreads();
  pdl_launch_dependents();

  float m[R], l[R], acc[R][C::kDPL];
#pragma unroll
  for (int rho = 0; rho < R; ++rho) {
    m[rho] = -INFINITY;
    l[rho] = 0.f;
#pragma unroll
    for (int e = 0; e < C::kDPL; ++e) acc[rho][e] = 0.f;
  }

  const int pos0 = L - n;                             // position of new token 0
  int j = 0;
  for (; j < my_tiles; ++j) {
    const int k = warp + C::kWarps * j;
    const int st = warp * P + (j % P);
    const bool got = mbar_wait(&full[st], (j / P) & 1);
    if (!__all_sync(0xffffffffu, got)) {
      if (lane == 0) raise_flag(a.flag, PKV_FLAG_TIMEOUT);
      break;
    }
    const uint8_t* ks = smem + st * C::kStageBytes;
    const uint8_t* vs = ks + C::kTileKeys * C::kRowBytes;
    const int key0 = (b0 + k * C::kTileBlocks) * kBlock;
    const int nvalid = min(C::kTileKeys, kv_len - key0);

    // ---- scores: lane owns key key0 + lane ----
    float sc[R];
#pragma unroll
    for (int rho = 0; rho < R; ++rho) sc[rho] = 0.f;
    const uint8_t* krow = ks + lane * C::kRowBytes;
#pragma unroll
    for (int c = 0; c < C::kChunks; ++c) {
      const int idx = (c + lane) & (C::kChunks - 1);
      const uint4 kc = *reinterpret_cast<const uint4*>(krow + idx * 16);
      if constexpr (sizeof(T) == 4) {
        const float k0 = __uint_as_float(kc.x), k1 = __uint_as_float(kc.y);
        const float k2 = __uint_as_float(kc.z), k3 = __uint_as_float(kc.w);
#pragma unroll
        for (int rho = 0; rho < R; ++rho) {
          if (rho < nrows) {
            const float4 qa = *reinterpret_cast<const float4*>(q_s + rho * D + idx * 4);
            sc[rho] = fmaf(qa.x, k0, sc[rho]);
            sc[rho] = fmaf(qa.y, k1, sc[rho]);
            sc[rho] = fmaf(qa.z, k2, sc[rho]);
            sc[rho] = fmaf(qa.w, k3, sc[rho]);
          }
        }
      } else {
        const float k0 = bf16_lo(kc.x), k1 = bf16_hi(kc.x), k2 = bf16_lo(kc.y),
                    k3 = bf16_hi(kc.y);
        const float k4 = bf16_lo(kc.z), k5 = bf16_hi(kc.z), k6 = bf16_lo(kc.w),
                    k7 = bf16_hi(kc.w);
#pragma unroll
        for (int rho = 0; rho < R; ++rho) {
          if (rho < nrows) {
            const float4 qa = *reinterpret_cast<const float4*>(q_s + rho * D + idx * 4);
            const float4 qb = *reinterpret_cast<const float4*>(q_s + rho * D + D / 2 + idx * 4);
            float t0 = sc[rho];
            t0 = fmaf(qa.x, k0, t0);
            t0 = fmaf(qa.y, k1, t0);
            t0 = fmaf(qa.z, k2, t0);
            t0 = fmaf(qa.w, k3, t0);
            t0 = fmaf(qb.x, k4, t0);
            t0 = fmaf(qb.y, k5, t0);
            t0 = fmaf(qb.z, k6, t0);
            t0 = fmaf(qb.w, k7, t0);
            sc[rho] = t0;
          }
        }
      }
    }

    // ---- online softmax update (per row; m uniform over the warp) ----
    const int key = key0 + lane;
    float* pw = p_s + (warp * C::kTileKeys + lane) * R;
#pragma unroll
    for (int rho = 0; rho < R; ++rho) {
      if (rho < nrows) {
        const int lim = a.causal ? (pos0 + (rho0 + rho) / a.group + 1) : L;
        const float sv = key < lim ? sc[rho] : -INFINITY;
        const float mnew = fmaxf(m[rho], warp_max(sv));
        const float msafe = mnew == -INFINITY ? 0.f : mnew;
        const float alpha = ex2(m[rho] - msafe);
        const float p = ex2(sv - msafe);
        l[rho] = l[rho] * alpha + p;
        m[rho] = mnew;
#pragma unroll
        for (int e = 0; e < C::kDPL; ++e) acc[rho][e] *= alpha;
        pw[rho] = p;
      }
    }
    __syncwarp();

    // ---- P.V: lane owns output columns lane*kDPL .. +kDPL-1 ----
#pragma unroll 2
    for (int jj = 0; jj < nvalid; ++jj) {
      const float* pr = p_s + (warp * C::kTileKeys + jj) * R;
      float pv[R];
#pragma unroll
      for (int r4 = 0; r4 < R; r4 += 4) {
        const float4 t4 = *reinterpret_cast<const float4*>(pr + r4);
        pv[r4] = t4.x;
        pv[r4 + 1] = t4.y;
        pv[r4 + 2] = t4.z;
        pv[r4 + 3] = t4.w;
      }
      float vf[C::kDPL];
      const uint8_t* vrow = vs + jj * C::kRowBytes;
      if constexpr (sizeof(T) == 4) {
        if constexpr (C::kDPL == 2) {
          const float2 v2 = *reinterpret_cast<const float2*>(vrow + lane * 8);
          vf[0] = v2.x;
          vf[1] = v2.y;
        } else {
          const float4 v4 = *reinterpret_cast<const float4*>(vrow + lane * 16);
          vf[0] = v4.x;
          vf[1] = v4.y;
          vf[2] = v4.z;
          vf[3] = v4.w;
        }
      } else {
        if constexpr (C::kDPL == 2) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(vrow + lane * 4);
          vf[0] = bf16_lo(w);
          vf[1] = bf16_hi(w);
        } else {
          const uint2 w = *reinterpret_cast<const uint2*>(vrow + lane * 8);
          vf[0] = bf16_lo(w.x);
          vf[1] = bf16_hi(w.x);
          vf[2] = bf16_lo(w.y);
          vf[3] = bf16_hi(w.y);
        }
      }
#pragma unroll
      for (int rho = 0; rho < R; ++rho) {
        if (rho < nrows) {
#pragma unroll
          for (int e = 0; e < C::kDPL; ++e) acc[rho][e] = fmaf(pv[rho], vf[e], acc[rho][e]);
        }
      }
    }
    __syncwarp();
    issue(j + P);                     // refill the stage just consumed
  }
  if (j < my_tiles && lane == 0) {
    // gave up early: let this warp's loads still in flight land before the
    // shared memory is reused (bounded again)
    for (int jj = j; jj < min(my_tiles, j + P); ++jj)
      if (!mbar_wait(&full[warp * P + (jj % P)], (jj / P) & 1)) break;
  }

  // ---- merge the warps' states (shared memory reused) ----
  __syncthreads();
  float* mw = reinterpret_cast<float*>(smem);
  float* lw = mw + C::kWarps * R;
  float* aw = lw + C::kWarps * R;
#pragma unroll
  for (int rho = 0; rho < R; ++rho) {
    if (rho < nrows) {
      const float lt = warp_sum(l[rho]);
      if (lane == 0) {
        mw[warp * R + rho] = m[rho];
        lw[warp * R + rho] = lt;
      }
#pragma unroll
      for (int e = 0; e < C::kDPL; ++e)
        aw[(warp * R + rho) * D + lane * C::kDPL + e] = acc[rho][e];
    }
  }
  __syncthreads();
  for (int rho = warp; rho < nrows; rho += C::kWarps) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) M = fmaxf(M, mw[w * R + rho]);
    float o[C::kDPL];
#pragma unroll
    for (int e = 0; e < C::kDPL; ++e) o[e] = 0.f;
    float lsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < C::kWarps; ++w) {
        const float f = ex2(mw[w * R + rho] - M);
        lsum = fmaf(f, lw[w * R + rho], lsum);
#pragma unroll
        for (int e = 0; e < C::kDPL; ++e)
          o[e] = fmaf(f, aw[(w * R + rho) * D + lane * C::kDPL + e], o[e]);
      }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const float lse2 = lsum > 0.f ? M + lg2(lsum) : -INFINITY;
    const int rr = rho0 + rho;
    const int i = rr / a.group;
    const int h = g * a.group + rr % a.group;
    if (split_mode) {
      const int64_t w = ws_row(a, s, r, i, h);
#pragma unroll
      for (int e = 0; e < C::kDPL; ++e) a.ws_o[w * D + lane * C::kDPL + e] = o[e] * inv;
      if (lane == 0) a.ws_lse[w] = lse2;
    } else {
      const int64_t t = q0 + i;
#pragma unroll
      for (int e = 0; e < C::kDPL; ++e)
        store_elem<T>(a.out, (t * a.hq + h) * D + lane * C::kDPL + e, o[e] * inv);
      if (a.lse_out != nullptr && lane == 0) a.lse_out[t * a.hq + h] = lse2 * kLn2;
    }
  }
}

// One warp per (request, decode row, q head): merge the split partials by
// their log-sum-exp weights, M = max_s lse_s, w_s = 2^(lse_s - M),
// o = sum_s w_s o_s / sum_s w_s.
template <typename T, int D>
__global__ void __launch_bounds__(128) combine_kernel(const AttnArgs a) {
  constexpr int kDPL = D / 32;
  pdl_wait_primary();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * 4 + warp;
  const int h = static_cast<int>(item % a.hq);
  const int64_t ri = item / a.hq;
  const int i = static_cast<int>(ri % kDecodeMaxQ);
  const int r = static_cast<int>(ri / kDecodeMaxQ);
  if (r >= a.num_seqs) return;
  const int q0 = __ldg(a.qsl + r), q1 = __ldg(a.qsl + r + 1);
  const int n = q1 - q0;
  if (n <= 0 || n > kDecodeMaxQ || i >= n || q0 < 0 || q1 > a.num_tokens) return;
  if (n > __ldg(a.seq_lens + r)) return;
  const int S = a.num_splits;
  float M = -INFINITY;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, a.ws_lse[ws_row(a, s, r, i, h)]);
  M = warp_max(M);
  float o[kDPL];
#pragma unroll
  for (int e = 0; e < kDPL; ++e) o[e] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const int64_t w = ws_row(a, s, r, i, h);
      const float f = ex2(a.ws_lse[w] - M);
      wsum += f;
      if (kDPL == 4) {
        const float4 p = *reinterpret_cast<const float4*>(a.ws_o + w * D + lane * 4);
        o[0] = fmaf(f, p.x, o[0]);
        o[1] = fmaf(f, p.y, o[1]);
        o[2 % kDPL] = fmaf(f, p.z, o[2 % kDPL]);
        o[3 % kDPL] = fmaf(f, p.w, o[3 % kDPL]);
      } else {
#pragma unroll
        for (int e = 0; e < kDPL; ++e) o[e] = fmaf(f, a.ws_o[w * D + lane * kDPL + e], o[e]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int64_t t = q0 + i;
#pragma unroll
  for (int e = 0; e < kDPL; ++e) store_elem<T>(a.out, (t * a.hq + h) * D + lane * kDPL + e, o[e] * inv);
  if (a.lse_out != nullptr && lane == 0)
    a.lse_out[t * a.hq + h] = wsum > 0.f ? (M + lg2(wsum)) * kLn2 : -INFINITY;
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
template <typename T, int D, int R>
static cudaError_t launch_decode_t(const AttnArgs& a, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, int row_tiles, bool pdl,
                                   cudaStream_t stream) {
  using C = DecodeCfg<T, D>;
  using Sm = DecodeSmem<T, D, R>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<T, D, R>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Sm::kAlloc);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
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
  return cudaLaunchKernelEx(&cfg, decode_kernel<T, D, R>, kmap, vmap, a);
}

template <typename T, int D>
static cudaError_t launch_decode_d(const AttnArgs& a, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, int R, int row_tiles, bool pdl,
                                   cudaStream_t stream) {
  switch (R) {
    case 4: return launch_decode_t<T, D, 4>(a, kmap, vmap, row_tiles, pdl, stream);
    case 8: return launch_decode_t<T, D, 8>(a, kmap, vmap, row_tiles, pdl, stream);
    default: return launch_decode_t<T, D, 16>(a, kmap, vmap, row_tiles, pdl, stream);
  }
}

// Rows per CTA tile for a launch: the smallest of 4/8/16 holding one request's
// decode rows (group x q_len), 16 when longer requests also run here.
int decode_rows_per_tile(int group, int max_query_len, bool long_rows) {
  const int q = long_rows ? max_query_len : (max_query_len < kDecodeMaxQ ? max_query_len : kDecodeMaxQ);
  const int need = group * (q < 1 ? 1 : q);
  return need <= 4 ? 4 : (need <= 8 ? 8 : 16);
}

cudaError_t launch_decode(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          bool bf16, int head_dim, bool pdl, cudaStream_t stream) {
  const int R = decode_rows_per_tile(a.group, a.max_query_len, a.long_rows != 0);
  const int qmax = a.long_rows ? a.max_query_len : min(a.max_query_len, kDecodeMaxQ);
  const int row_tiles = (a.group * (qmax < 1 ? 1 : qmax) + R - 1) / R;
  if (row_tiles > 65535 || a.num_seqs > 65535) return cudaErrorInvalidConfiguration;
  if (bf16) {
    return head_dim == 128 ? launch_decode_d<__nv_bfloat16, 128>(a, kmap, vmap, R, row_tiles, pdl, stream)
                           : launch_decode_d<__nv_bfloat16, 64>(a, kmap, vmap, R, row_tiles, pdl, stream);
  }
  return head_dim == 128 ? launch_decode_d<float, 128>(a, kmap, vmap, R, row_tiles, pdl, stream)
                         : launch_decode_d<float, 64>(a, kmap, vmap, R, row_tiles, pdl, stream);
}

cudaError_t launch_combine(const AttnArgs& a, bool bf16, int head_dim, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(a.num_seqs) * kDecodeMaxQ * a.hq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((items + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16) {
    return head_dim == 128 ? cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16, 128>, a)
                           : cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16, 64>, a);
  }
  return head_dim == 128 ? cudaLaunchKernelEx(&cfg, combine_kernel<float, 128>, a)
                         : cudaLaunchKernelEx(&cfg, combine_kernel<float, 64>, a);
}

}  // namespace pkv
