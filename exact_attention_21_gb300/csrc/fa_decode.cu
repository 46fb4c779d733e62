// Split-K/V decoding ("Flash-Decoding").
//
// What it computes ("Attention 算子优化…", section 五; "FlashAttention：从
// Safe Softmax 到分块计算", sections 3 and 10): one decoding step, i.e. for
// every sequence b and query head h the attention of the single new query
// q[b, h] over all cached keys and values of the sequence,
//     O = softmax(scale * K q) V,   LSE = ln sum_j exp(scale * <k_j, q>).
// A decoding step reads the whole K/V cache for a few multiply-adds per byte,
// so it is bound by HBM bandwidth; the arithmetic runs on the CUDA cores and
// the design goal is to keep enough K/V bytes in flight.
//
// Two launches:
//  fa_decode_split_kernel: CTA = (split, K/V head, sequence).  A split is a
//    run of `split_tiles` 128-key tiles of one sequence.  A producer warp
//    streams the split's K and V tiles through a ring of shared-memory stages
//    with TMA; 256 consumer threads keep, for every query head of the GQA
//    group, the running max, running sum and output accumulator of the
//    online-softmax recurrence (section 3 of the safe-softmax page), and
//    finally write the split's normalised output O_s and its LSE_s.
//  fa_decode_combine_kernel: one warp per (sequence, query head) merges the
//    splits with the same rule: LSE = ln sum_s e^{LSE_s} and
//    O = sum_s e^{LSE_s - LSE} O_s.
//
// Consumer thread mappings (256 threads, tiles of 128 keys):
//   scores:  thread t takes key t/2 and half t%2 of the head dimension; the
//            two halves meet with one shuffle.
//   P V:     thread t takes the head-dimension pair 2(t mod d/2), 2(t mod d/2)+1
//            over one 1/(512/d) slice of the tile's keys; the slices are
//            summed once at the end of the split.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "fa_common.cuh"

namespace fa {

constexpr int kDecMaxGroup = 16;   // query heads per K/V head handled by one CTA
constexpr int kDecConsumers = 256;

template <int D>
struct DecLayout {
  static constexpr int kChunkBytes = kTile * 128;            // 128 keys x 64 dims bf16, 128B-swizzled
  static constexpr int kTileBytes = (D / 64) * kChunkBytes;  // one K or V tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = D == 128 ? 3 : 6;
  static constexpr int kOffQ = kStages * kStageBytes;             // f32 [group][D], pre-scaled query
  static constexpr int kOffP = kOffQ + kDecMaxGroup * D * 4;      // f32 [group][128] probabilities
  static constexpr int kOffRed = kOffP + kDecMaxGroup * kTile * 4;  // f32 [8 warps][group]
  static constexpr int kOffML = kOffRed + 8 * kDecMaxGroup * 4;     // f32 m[group], l[group]
  static constexpr int kOffBar = kOffML + 2 * kDecMaxGroup * 4;     // full[kStages], empty[kStages]
  static constexpr int kOffMisc = kOffBar + 2 * kStages * 8;
  static constexpr int kBytes = kOffMisc + 16 + 1024;
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
  static_assert((512 / D) * kDecMaxGroup * D * 4 <= kStageBytes, "slice sums must fit in one stage");
};

// Barrier among the 256 consumer threads only (the producer warp does not take
// part); returns whether `v` was true in every consumer thread.
__device__ __forceinline__ bool consumers_sync_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, 256, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// ---------------------------------------------------------------------------
// Where a sequence's cache lives.  Packed or batched caches: rows seq0 ..
// seq0 + L - 1 of the [T, Hkv, d] cache.  Paged caches ("Attention 算子优化…",
// section 五, PagedAttention): a pool of pages of page_size rows; logical key
// j of sequence b is row  block_table[b][j / page_size] * page_size +
// j % page_size  of the pool, and L = seqlens[b].

// Cache length (and start row, unpaged) of sequence b; false (and a status
// bit) when the offsets or the length are out of range.
__device__ __forceinline__ bool decode_bounds(const DecodeParams& p, int b, long long& seq0, int& L) {
  if (p.block_table == nullptr) return sequence_bounds(p.cu, b, p.N, p.T, seq0, L, p.status);
  const int l = __ldg(p.seqlens + b);
  if (l < 0 || l > p.max_pages * p.page_size) {
    atomicOr(p.status, kStatusBadOffsets);
    return false;
  }
  seq0 = 0;
  L = l;
  return true;
}

// Physical page of logical page lp of sequence b.  Pages past the cache may
// hold anything (their keys are masked), so page 0 is read for them; a table
// entry inside the cache that is out of range sets a status bit and is
// replaced by page 0 as well.
__device__ __forceinline__ int decode_page(const DecodeParams& p, int b, int lp, int L) {
  const bool live = lp * p.page_size < L;
  int phys = live ? __ldg(p.block_table + static_cast<long long>(b) * p.max_pages + lp) : 0;
  if (phys < 0 || phys >= p.num_pages) {
    atomicOr(p.status, kStatusBadOffsets);
    phys = 0;
  }
  return phys;
}

// Cache row of logical key kpos (kpos < L) of sequence b.
__device__ __forceinline__ long long decode_row(const DecodeParams& p, int b, long long seq0, int kpos, int L) {
  if (p.block_table == nullptr) return seq0 + kpos;
  return static_cast<long long>(decode_page(p, b, kpos / p.page_size, L)) * p.page_size + kpos % p.page_size;
}

// TMA loads of the K and V tile of logical keys k0 .. k0 + 127 of sequence b
// (K/V head g), issued by the 32 lanes of the calling warp: CHUNKS boxes of
// 64 (16-bit) or 128 (8-bit) columns per tile, each CHUNK_BYTES apart in
// shared memory; paged caches take one box of page_size rows per page (1
// KB-aligned in shared memory for page_size >= 8, so the 128-byte swizzle
// pattern continues across boxes), lane j copying page j: a tile of small
// pages is many copies, and one warp instruction issues one per lane.
// Returns false for a table entry outside the pool (page 0 is read instead,
// and the status bit is set).
template <int CHUNKS, int CHUNK_BYTES, int COLS>
__device__ __forceinline__ void load_kv_tile(const DecodeParams& p, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                             uint8_t* dst_k, uint8_t* dst_v, uint64_t* bar, int b, int g,
                                             long long seq0, int k0, int L, int lane) {
  if (p.block_table == nullptr) {
    // lane c: K box c; lane CHUNKS + c: V box c
    if (lane < 2 * CHUNKS) {
      const int c = lane % CHUNKS;
      const bool is_v = lane >= CHUNKS;
      tma_load_3d((is_v ? dst_v : dst_k) + c * CHUNK_BYTES, is_v ? tm_v : tm_k, bar, c * COLS, g,
                  static_cast<int>(seq0 + k0));
    }
    return;
  }
  const int ps = p.page_size;
  const int j = lane;  // page of the tile
  if (j < kTile / ps) {
    const int lp = k0 / ps + j;
    int phys = lp * ps < L ? __ldg(p.block_table + static_cast<long long>(b) * p.max_pages + lp) : 0;
    if (phys < 0 || phys >= p.num_pages) {  // see decode_page
      atomicOr(p.status, kStatusBadOffsets);
      phys = 0;
    }
    const int row = phys * ps;
    for (int c = 0; c < CHUNKS; ++c) {
      tma_load_3d(dst_k + c * CHUNK_BYTES + j * ps * 128, tm_k, bar, c * COLS, g, row);
      tma_load_3d(dst_v + c * CHUNK_BYTES + j * ps * 128, tm_v, bar, c * COLS, g, row);
    }
  }
}

template <int D, int G>
__global__ void __launch_bounds__(288, 1)
fa_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const DecodeParams p) {
  using Lay = DecLayout<D>;
  constexpr int NS = Lay::kStages;
  static_assert(G <= kDecMaxGroup, "group too large");

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  long long seq0;
  int L;
  if (!decode_bounds(p, b, seq0, L)) return;
  const int seq_tiles = (L + kTile - 1) / kTile;
  const int t0 = split * p.split_tiles;
  if (t0 >= seq_tiles) return;  // past the end of this sequence's cache: the combine skips it
  const int nt = min(p.split_tiles, seq_tiles - t0);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kOffBar);
  uint64_t* empty = full + NS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kOffMisc);
  auto stage = [&](int st) { return smem + st * Lay::kStageBytes; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kDecConsumers);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  auto give_up = [&]() {
    atomicOr(p.status, kStatusTimeout);
    *abort_flag = 1;
  };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (warp == 8) {
    // ------------------------------------------------------------ producer (one warp)
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    int issued = 0;
    bool ok = true;
    for (int i = 0; i < nt; ++i) {
      const int st = i % NS;
      // lane 0 waits for the stage and posts the byte count before any copy
      if (lane == 0) {
        if (i >= NS) ok = mbar_wait(empty + st, ((i / NS) - 1) & 1, abort_flag);
        if (ok) mbar_arrive_expect_tx(full + st, Lay::kStageBytes);
      }
      if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
      load_kv_tile<D / 64, Lay::kChunkBytes, 64>(p, &tm_k, &tm_v, stage(st), stage(st) + Lay::kTileBytes, full + st,
                                                 b, g, seq0, (t0 + i) * kTile, L, lane);
      ++issued;
    }
    if (lane == 0) {
      if (!ok) give_up();
      // no TMA write may still be in flight when the CTA exits
      int never = 0;
      for (int i = issued > NS ? issued - NS : 0; i < issued; ++i) mbar_wait(full + i % NS, (i / NS) & 1, &never);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int t = threadIdx.x;
  const int group = p.group;
  const int hq0 = g * group;
  float* sQ = reinterpret_cast<float*>(smem + Lay::kOffQ);
  float* sP = reinterpret_cast<float*>(smem + Lay::kOffP);
  float* sRed = reinterpret_cast<float*>(smem + Lay::kOffRed);
  float* sM = reinterpret_cast<float*>(smem + Lay::kOffML);
  float* sL = sM + kDecMaxGroup;

  // the group's queries, scaled by c = scale * log2 e (heads past the group: 0)
  const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(p.q) + (static_cast<long long>(b) * p.Hq + hq0) * D;
  for (int i = t; i < G * D; i += kDecConsumers)
    sQ[i] = (i / D < group) ? __bfloat162float(qb[i]) * p.scale_log2 : 0.f;

  const int key = t >> 1;  // score mapping
  const int dh = t & 1;
  constexpr int kPairs = D / 2;  // P V mapping
  constexpr int kSubs = kDecConsumers / kPairs;
  constexpr int kKeysPerSub = kTile / kSubs;
  const int e0 = 2 * (t % kPairs);
  const int sub = t / kPairs;
  const uint32_t v_off = (e0 / 64) * Lay::kChunkBytes + (e0 % 8) * 2;
  const int v_unit = (e0 % 64) / 8;

  float m[G], lt[G], acc[G][2];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    lt[h] = 0.f;
    acc[h][0] = acc[h][1] = 0.f;
  }
  bool ok = consumers_sync_and(true);  // sQ written
  for (int i = 0; i < nt; ++i) {
    const int st = i % NS;
    // a lane that gave up takes its whole warp along (the shuffles below
    // need every lane), and the vote after the scores takes the rest
    ok = __all_sync(0xffffffffu, mbar_wait(full + st, (i / NS) & 1, abort_flag));
    const uint8_t* sK = stage(st);
    const uint8_t* sV = sK + Lay::kTileBytes;
    float s[G];
#pragma unroll
    for (int h = 0; h < G; ++h) s[h] = 0.f;
    if (ok) {
      // ---- scores s_h = c <q_h, k_key> over this thread's half of the row
#pragma unroll
      for (int u = 0; u < D / 16; ++u) {
        const int unit = dh * (D / 16) + u;  // 16-byte unit of the row
        const uint4 kr =
            *reinterpret_cast<const uint4*>(sK + (unit / 8) * Lay::kChunkBytes + key * 128 + (((unit % 8) ^ (key & 7)) << 4));
        const float kf[8] = {bf16_lo(kr.x), bf16_hi(kr.x), bf16_lo(kr.y), bf16_hi(kr.y),
                             bf16_lo(kr.z), bf16_hi(kr.z), bf16_lo(kr.w), bf16_hi(kr.w)};
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 qa = *reinterpret_cast<const float4*>(sQ + h * D + unit * 8);
          const float4 qc = *reinterpret_cast<const float4*>(sQ + h * D + unit * 8 + 4);
          float x = s[h];
          x = fmaf(kf[0], qa.x, x);
          x = fmaf(kf[1], qa.y, x);
          x = fmaf(kf[2], qa.z, x);
          x = fmaf(kf[3], qa.w, x);
          x = fmaf(kf[4], qc.x, x);
          x = fmaf(kf[5], qc.y, x);
          x = fmaf(kf[6], qc.z, x);
          x = fmaf(kf[7], qc.w, x);
          s[h] = x;
        }
      }
      // keys past the end of the cache (tail tile) take no part
      const bool valid = (t0 + i) * kTile + key < L;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        s[h] += __shfl_xor_sync(0xffffffffu, s[h], 1);
        if (!valid) s[h] = -INFINITY;
        float mx = s[h];
#pragma unroll
        for (int off = 16; off > 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane == 0) sRed[warp * G + h] = mx;
      }
    }
    // every consumer either has its scores or gives up with the others
    if (!(ok = consumers_sync_and(ok))) break;
    // ---- online-softmax update; key 0 of every tile is valid, so the new max is finite
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float tm = sRed[h];
#pragma unroll
      for (int w = 1; w < 8; ++w) tm = fmaxf(tm, sRed[w * G + h]);
      const float mn = fmaxf(m[h], tm);
      const float alpha = ex2_approx(m[h] - mn);  // 0 on the first tile (m = -inf)
      m[h] = mn;
      const float pv = ex2_approx(s[h] - mn);     // 0 for masked keys
      if (dh == 0) {
        sP[h * kTile + key] = pv;
        lt[h] = fmaf(lt[h], alpha, pv);
      }
      acc[h][0] *= alpha;
      acc[h][1] *= alpha;
    }
    consumers_sync();
    // ---- O_h += sum_j p_hj v_j over this thread's key slice and dimension pair
#pragma unroll
    for (int j4 = 0; j4 < kKeysPerSub; j4 += 4) {
      const int kb = sub * kKeysPerSub + j4;
      float pj[G][4];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float4 pp = *reinterpret_cast<const float4*>(sP + h * kTile + kb);
        pj[h][0] = pp.x;
        pj[h][1] = pp.y;
        pj[h][2] = pp.z;
        pj[h][3] = pp.w;
      }
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int kk = kb + jj;
        const uint32_t vv = *reinterpret_cast<const uint32_t*>(sV + v_off + kk * 128 + ((v_unit ^ (kk & 7)) << 4));
        const float v0 = bf16_lo(vv), v1 = bf16_hi(vv);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          acc[h][0] = fmaf(pj[h][jj], v0, acc[h][0]);
          acc[h][1] = fmaf(pj[h][jj], v1, acc[h][1]);
        }
      }
    }
    // this thread is done with the stage (K read above, V read here)
    mbar_arrive(empty + st);
  }
  if (!ok) {
    if (t == 0) give_up();
    return;
  }
  // -------------------------------------------------------------- split result
  consumers_sync();  // every thread is past its last read of the stages
  // l_h: sum of the per-thread partial sums
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float x = lt[h];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    if (lane == 0) sRed[warp * G + h] = x;
  }
  // slice sums of O through the first stage (its last TMA fill was consumed)
  float* sO = reinterpret_cast<float*>(stage(0));
#pragma unroll
  for (int h = 0; h < G; ++h) {
    sO[(sub * G + h) * D + e0] = acc[h][0];
    sO[(sub * G + h) * D + e0 + 1] = acc[h][1];
  }
  consumers_sync();
  if (t < G) {
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) l += sRed[w * G + t];
    sL[t] = l;
  }
  if (t == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) sM[h] = m[h];
  }
  consumers_sync();
  const long long row0 = static_cast<long long>(b) * p.Hq + hq0;
  for (int idx = t; idx < group * D; idx += kDecConsumers) {
    const int h = idx / D, e = idx % D;
    float o = 0.f;
#pragma unroll
    for (int sl = 0; sl < kSubs; ++sl) o += sO[(sl * G + h) * D + e];
    p.o_part[((row0 + h) * p.n_splits + split) * D + e] = o / sL[h];
  }
  if (t < group) {
    // natural-log LSE of the split: (m + log2 l) ln 2, m in log2 units
    p.lse_part[(row0 + t) * p.n_splits + split] = (sM[t] + log2f(sL[t])) * 0.6931471805599453f;
  }
}

// ---------------------------------------------------------------------------
// d = 128: the two products on the tensor cores.  With the query heads of the
// GQA group (padded to 16) as the MMA's N dimension:
//     S^T = K_tile Q^T       M = 128 keys,  N = 16 heads, K = d   (TMEM, f32)
//     O^T += V_tile^T P^T    M = d = 128,   N = 16 heads, K = 128 keys
// so the threads only turn 16 scores per key into probabilities.  The kernel
// is persistent (one CTA per SM over its (split, K/V head, sequence) items).
// Roles:
//   warp 0      TMA producer of the K / V stages.
//   warp 1      TMEM allocator and P V issuer (one thread).
//   warps 2-5,  two softmax warpgroups, half of the heads each: thread = key
//   warps 7-10  row of S^T (TMEM lane) for the probabilities, and = dimension
//               row of O^T for the rescale and the split's output.
//   warp 6      S^T issuer (one thread).
// S^T has three TMEM buffers, so S^T runs up to three tiles ahead of the
// softmax (into the next item too); O^T has two, one per item in flight;
// P^T (K-major: 16 head rows x 128 keys) is double-buffered in shared
// memory.  The running max of a head only moves when a tile's max exceeds it
// by more than a slack (log2 units); any common reference gives the same
// merge, so this is exact and O^T is rarely rescaled.
//
// With the FP8 cache S^T reads the E4M3 K tile as it arrived, in a
// kind::f8f6f4 MMA: each head's query is scaled by s_q = 448 / max|q| and
// written as three E4M3 rows, q1 = e4m3(s_q q), q2 = e4m3(s_q q - q1) and
// q3 = e4m3(s_q q - q1 - q2), which carry s_q q to about 2^-12 relative, so
// S^T (N = 48: 16 columns per term) loses nothing a bf16 query would keep;
// the softmax threads add the three columns of a head and divide by s_q.
// P V reads the E4M3 V tile as it arrived too ("Attention 算子优化…", section
// 六: the cache stays FP8 in HBM, softmax and accumulation in f32): a
// kind::f8f6f4 MMA of V^T (MN-major) with P^T written as three E4M3 terms in
// the same way, so the stage is the only copy of the tile on chip; the terms
// hold a weight w to 2^-12 relative for w >= 4 and to 2^-10 absolute below
// (half E4M3's subnormal step), finer than a bf16 P.  The per-token
// scales fold into the per-key work of the softmax
// threads: s_k multiplies the key's scores, s_v its probabilities before
// they are split into terms (the row sum keeps the unscaled probabilities).
// To keep the terms in E4M3's normal range, s_v is taken relative to 2^E, E
// the largest binary exponent of the scales seen so far (O^T is rescaled
// when E grows), the probabilities are bounded by a slack of 2 instead of 8,
// and the product is scaled by 2^6: the weights stay below 256, and those
// that carry O sit well above E4M3's smallest normal, 2^-6.
constexpr int kDecHeads = 16;               // MMA N: query heads per CTA, padded
constexpr float kDecRescaleSlack = 8.f;
constexpr float kDecRescaleSlackFp8 = 2.f;
constexpr int kDecPScaleLog2 = 6;           // FP8: P^T terms carry p s_v 2^(6 - e), e relative to 2^E

// 2^e as a float for an integer e; 0 below -126.
__device__ __forceinline__ float exp2i(int e) {
  return e < -126 ? 0.f : __uint_as_float(static_cast<uint32_t>(min(e, 127) + 127) << 23);
}

template <bool FP8>
struct DecTcLayout {
  static constexpr int D = 128;
  static constexpr int kChunkBytes = kTile * 128;      // 16-bit tile chunk: 128 keys x 64 dims
  static constexpr int kTileBytes = 2 * kChunkBytes;   // 16-bit 128 x 128 tile
  static constexpr int kTile8Bytes = kTile * 128;      // E4M3 128 x 128 tile (one 128-byte row per key)
  // TMA stages: 16-bit K and V tiles, or E4M3 K and V tiles
  static constexpr int kStageBytes = FP8 ? 2 * kTile8Bytes : 2 * kTileBytes;
  static constexpr int kStages = FP8 ? 6 : 3;
  static constexpr int kHChunkBytes = kDecHeads * 128;  // 16 rows x 128 bytes
  // Q: 16 heads x 128 dims, K-major, bf16; FP8: 48 E4M3 rows (three terms per head) x 128 dims
  static constexpr int kQBytes = (FP8 ? 3 : 2) * kHChunkBytes;
  // P^T: 16 heads x 128 keys, K-major, 16-bit; FP8: kPTerms E4M3 rows per head
  // (two terms run about 6 % faster but hold a weight to 2^-8 only, which a
  // single cached token with a large V row shows at the 1e-2 bar)
  static constexpr int kPTerms = 3;
  static constexpr int kPBytes = (FP8 ? kPTerms : 2) * kHChunkBytes;
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffP = kOffQ + 2 * kQBytes;      // Q: two buffers (this item's, the next one's)
  // P^T: two buffers; then f32 [2 warpgroups][4 warps][16 heads]
  static constexpr int kOffRed = kOffP + 2 * kPBytes;
  static constexpr int kOffInvSq = kOffRed + 2 * 4 * kDecHeads * 4;   // FP8: f32 1 / s_q [2 wg][2 buffers][16 heads]
  static constexpr int kOffRedE = kOffInvSq + 2 * 2 * kDecHeads * 4;  // FP8: int [2 wg][4 warps], scale exponents
  // FP8: per-token scales (s_k, s_v) of the 128 keys of the next kScaleAhead tiles, per warpgroup
  static constexpr int kScaleAhead = 4;
  static constexpr int kOffScale = kOffRedE + 32;
  static constexpr int kOffBar = kOffScale + (FP8 ? 2 * kScaleAhead * kTile * 8 : 0);
  // S^T buffers in TMEM: S^T runs up to three tiles ahead of the softmax
  static constexpr int kSBufs = 3;
  // full[], empty[], q_ready, s_full[3], p_ready[3], pv_done[2], drain, o_free[2]
  static constexpr int kNumBars = 2 * kStages + 12;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // compact item numbering: split-count prefix of up to kPrefixMaxB sequences
  static constexpr int kPrefixMaxB = FP8 ? 192 : 1024;
  static constexpr int kOffPrefix = kOffMisc + 16;
  static constexpr int kBytes = kOffPrefix + (kPrefixMaxB + 1) * 4 + 1024;
  // warp 0 loads, warp 1 issues P V, warps 2-5 and 7-10 run the softmax
  // (two warpgroups, half of the heads each) and warp 6 issues S^T: a single
  // thread issuing both products would start one of these narrow MMAs only
  // every ~100 cycles
  static constexpr int kWarpS = 6;
  static constexpr int kThreads = 32 * 11;
  // S^T buffers of kSCols columns from 0 (FP8: a column per head and term), O^T after them
  static constexpr int kSCols = FP8 ? 3 * kDecHeads : kDecHeads;
  // O^T: a column per head (FP8: per head and term), two buffers
  static constexpr int kOCols = FP8 ? kPTerms * kDecHeads : kDecHeads;
  static constexpr uint32_t kTmemCols = FP8 ? 256 : 128;
  static constexpr uint32_t kColS = 0, kColO = kSBufs * kSCols;
  static_assert(kColO + 2 * kOCols <= kTmemCols, "TMEM budget");
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void sts_u16(uint8_t* p, uint16_t v) { *reinterpret_cast<uint16_t*>(p) = v; }

// Barrier among the 128 threads of a softmax warpgroup (named barrier id);
// returns whether `v` held in all of them.
__device__ __forceinline__ bool softmax_sync_and(bool v, int id) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, 128, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id)
      : "memory");
  return r != 0;
}

// The same; returns whether `v` held in any of them.
__device__ __forceinline__ bool softmax_sync_or(bool v, int id) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, 128, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void softmax_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }

// Two E4M3 codes (low byte first) -> two f16 (low half first), exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xffffu), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// One work item of the persistent kernel: split w / (B Hkv) of K/V head
// w % Hkv of sequence (w / Hkv) % B.  Split-major, so that the items a CTA
// takes (blockIdx.x + j gridDim.x) spread over all split positions: with
// caches of unequal length only the first splits of the short ones exist.
// False for a split past the end of its sequence's cache (the combine skips
// it) and for a sequence with bad offsets or length (a status bit).
struct DecItem {
  long long seq0;
  int split, g, b, L, t0, nt;
};
// Compact numbering (prefix != null): item w is K/V head w % Hkv of the
// (w / Hkv)-th (sequence, split) pair, sequence-major; prefix[b] counts the
// splits of the sequences before b (prefix[B]: all of them), so every item
// exists and consecutive CTAs take consecutive items.
__device__ __forceinline__ bool decode_item(const DecodeParams& p, const int* prefix, long long w, DecItem& it) {
  if (prefix != nullptr) {
    const int j = static_cast<int>(w / p.Hkv);
    it.g = static_cast<int>(w % p.Hkv);
    int lo = 0, hi = p.B;  // prefix[lo] <= j < prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= j) lo = mid; else hi = mid;
    }
    it.b = lo;
    it.split = j - prefix[lo];
    if (!decode_bounds(p, it.b, it.seq0, it.L)) return false;
    const int seq_tiles = (it.L + kTile - 1) / kTile;
    it.t0 = it.split * p.split_tiles;
    if (it.t0 >= seq_tiles) return false;
    it.nt = min(p.split_tiles, seq_tiles - it.t0);
    return true;
  }
  const long long heads = static_cast<long long>(p.B) * p.Hkv;
  it.split = static_cast<int>(w / heads);
  const long long rest = w % heads;
  it.g = static_cast<int>(rest % p.Hkv);
  it.b = static_cast<int>(rest / p.Hkv);
  if (!decode_bounds(p, it.b, it.seq0, it.L)) return false;
  const int seq_tiles = (it.L + kTile - 1) / kTile;
  it.t0 = it.split * p.split_tiles;
  if (it.t0 >= seq_tiles) return false;
  it.nt = min(p.split_tiles, seq_tiles - it.t0);
  return true;
}
// This CTA's first item at or after w (its items are blockIdx.x + j gridDim.x)
// that has work, or n_items.
__device__ __forceinline__ long long next_item(const DecodeParams& p, const int* prefix, long long w, long long n_items,
                                               DecItem& it) {
  for (; w < n_items; w += gridDim.x)
    if (decode_item(p, prefix, w, it)) return w;
  return n_items;
}

// A softmax warpgroup's part in an item's query (thread r: dims 16 (r % 8) ..
// +15 of head r / 8, in qa).  The first warpgroup (write) writes it into a Q
// buffer q, K-major with the 128-byte swizzle (FP8: three E4M3 rows per
// head) and arrives on q_ready; with an FP8 cache each warpgroup puts
// 1 / s_q of the 16 heads into its own inv_sq and meets its other 127
// threads (barrier bar_id).  Out of line: it runs once per item, and inlined
// it would sit in the hot loop's code.
template <bool FP8>
__device__ __noinline__ void dec_store_q(uint8_t* q, float* inv_sq, uint64_t* q_ready, int r, uint4 qa0, uint4 qa1,
                                         bool write, int bar_id) {
  using Lay = DecTcLayout<FP8>;
  const uint4 qa[2] = {qa0, qa1};
  const int h = r / 8, sub = r % 8;
  if (!FP8 && !write) return;
  if constexpr (FP8) {
    // 48 E4M3 rows: the terms of head h in rows h, 16 + h, 32 + h
    const uint32_t wq[8] = {qa[0].x, qa[0].y, qa[0].z, qa[0].w, qa[1].x, qa[1].y, qa[1].z, qa[1].w};
    float v[16];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      v[2 * e] = bf16_lo(wq[e]);
      v[2 * e + 1] = bf16_hi(wq[e]);
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(v[e]));
    // the 8 threads of a head are 8 consecutive lanes
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float sq = amax > 0.f ? 448.f / amax : 1.f;
    uint32_t term[3][4] = {};
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      float2 y = make_float2(v[e] * sq, v[e + 1] * sq);  // remainder still to represent
#pragma unroll
      for (int t = 0; t < 3; ++t) {
        const __nv_fp8x2_storage_t c2 = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
        const __half2_raw hb = __nv_cvt_fp8x2_to_halfraw2(c2, __NV_E4M3);
        y.x -= __half2float(*reinterpret_cast<const __half*>(&hb.x));  // exact in f32
        y.y -= __half2float(*reinterpret_cast<const __half*>(&hb.y));
        term[t][e / 4] |= static_cast<uint32_t>(c2) << (16 * ((e / 2) & 1));
      }
    }
    if (write) {
#pragma unroll
      for (int t = 0; t < 3; ++t) {
        const int row = t * kDecHeads + h;
        *reinterpret_cast<uint4*>(q + row * 128 + ((sub ^ (row & 7)) << 4)) =
            make_uint4(term[t][0], term[t][1], term[t][2], term[t][3]);
      }
    }
    if (sub == 0) inv_sq[h] = 1.f / sq;
  } else {
    // units 2 sub, 2 sub + 1 of the 256-byte row: chunk u / 8, unit u % 8
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int u = 2 * sub + j;
      *reinterpret_cast<uint4*>(q + (u / 8) * Lay::kHChunkBytes + h * 128 + (((u % 8) ^ (h & 7)) << 4)) = qa[j];
    }
  }
  if (write) {
    fence_proxy_async_smem();
    mbar_arrive(q_ready);
  }
  if constexpr (FP8) softmax_sync(bar_id);  // every head's 1 / s_q written
}

// HS: query heads the softmax threads work on (8 when the GQA group has at
// most 8, else 16): the MMA's N is 16 either way, and the rows of P^T and
// columns of O^T past the group are never read.
template <bool FP8, int HS>
__global__ void __launch_bounds__(DecTcLayout<FP8>::kThreads, 1)
fa_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const DecodeParams p) {
  using Lay = DecTcLayout<FP8>;
  constexpr int NS = Lay::kStages;
  constexpr int D = Lay::D;
  constexpr int H = kDecHeads;
  // bf16 cache: bf16 MMAs; E4M3 cache: E4M3 K x the query's E4M3 terms, and
  // E4M3 V^T (MN-major) x the E4M3 terms of P^T
  constexpr uint32_t id_s = FP8 ? idesc_e4m3_f32(kTile, 3 * H) : idesc_bf16_f32(kTile, H, false, false);
  constexpr uint32_t id_o = FP8 ? idesc_e4m3_f32(D, Lay::kPTerms * H, true) : idesc_bf16_f32(D, H, true, false);

  // persistent: the CTA runs its items back to back; the barrier rings and
  // the S^T / P^T / V buffers run on a tile count over all of them (gt), so
  // the loads and S^T of an item overlap the previous item's epilogue
  long long n_items = static_cast<long long>(p.n_splits) * p.Hkv * p.B;

  // the combine kernel, launched as a programmatic dependent, may be scheduled
  // now: it waits for this whole grid before reading the partial results
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Lay::kOffQ;
  float* sRed = reinterpret_cast<float*>(smem + Lay::kOffRed);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = full + NS;
  uint64_t* q_ready = empty + NS;
  uint64_t* s_full = q_ready + 1;
  uint64_t* p_ready = s_full + Lay::kSBufs;
  uint64_t* pv_done = p_ready + Lay::kSBufs;
  uint64_t* drain = pv_done + 2;
  uint64_t* o_free = drain + 1;      // O^T buffer j read by the epilogue of an item
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kOffMisc + 4);
  int* sPre = p.compact ? reinterpret_cast<int*>(smem + Lay::kOffPrefix) : nullptr;
  auto stage = [&](uint32_t st) { return smem + st * Lay::kStageBytes; };
  auto pbuf = [&](uint32_t i) { return smem + Lay::kOffP + (i & 1) * Lay::kPBytes; };
  // the K and V tiles of tile i (E4M3 for an FP8 cache)
  auto ktile = [&](uint32_t i) { return stage(i % NS); };
  auto vtile = [&](uint32_t i) { return stage(i % NS) + (FP8 ? Lay::kTile8Bytes : Lay::kTileBytes); };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, 1);  // P V of the tile completed (after its S^T)
    }
    mbar_init(q_ready, 128);
    for (int i = 0; i < Lay::kSBufs; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_ready + i, 256);  // both softmax warpgroups
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(pv_done + i, 1);
      mbar_init(o_free + i, 256);
    }
    mbar_init(drain, 2);  // both MMA-issuing threads commit
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Lay::kTmemCols);
    tmem_relinquish();
  }
  if (sPre != nullptr && warp == 2) {
    // split counts of the sequences, scanned 32 at a time (exclusive prefix)
    int run = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      int ns = 0;
      long long s0;
      int L;
      if (b < p.B && decode_bounds(p, b, s0, L)) ns = ((L + kTile - 1) / kTile + p.split_tiles - 1) / p.split_tiles;
      int x = ns;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
      }
      if (b < p.B) sPre[b] = run + x - ns;
      run += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) sPre[p.B] = run;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (sPre != nullptr) n_items = static_cast<long long>(sPre[p.B]) * p.Hkv;
  auto give_up = [&]() {
    atomicOr(p.status, kStatusTimeout);
    *abort_flag = 1;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer (one warp)
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    uint32_t gt = 0;  // tiles issued
    bool ok = true;
    DecItem it;
    for (long long w = next_item(p, sPre, blockIdx.x, n_items, it); w < n_items && ok;
         w = next_item(p, sPre, w + gridDim.x, n_items, it)) {
      for (int i = 0; i < it.nt; ++i, ++gt) {
        const uint32_t st = gt % NS;
        // lane 0 waits for the stage and posts the byte count before any copy
        if (lane == 0) {
          if (gt >= NS) ok = mbar_wait(empty + st, ((gt / NS) - 1) & 1, abort_flag);
          if (ok) mbar_arrive_expect_tx(full + st, Lay::kStageBytes);
        }
        if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
        if constexpr (FP8) {
          load_kv_tile<1, Lay::kTile8Bytes, 128>(p, &tm_k, &tm_v, stage(st), stage(st) + Lay::kTile8Bytes, full + st,
                                                  it.b, it.g, it.seq0, (it.t0 + i) * kTile, it.L, lane);
        } else {
          load_kv_tile<2, Lay::kChunkBytes, 64>(p, &tm_k, &tm_v, stage(st), stage(st) + Lay::kTileBytes, full + st,
                                                 it.b, it.g, it.seq0, (it.t0 + i) * kTile, it.L, lane);
        }
      }
    }
    if (lane == 0) {
      if (!ok) give_up();
      // no TMA write may still be in flight when the CTA exits
      int never = 0;
      for (uint32_t j = gt > NS ? gt - NS : 0; j < gt; ++j) mbar_wait(full + j % NS, (j / NS) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ P V issuer
    if (lane == 0) {
      bool ok = true;
      uint32_t gt = 0, kq = 0;  // tiles and items so far
      DecItem it;
      for (long long w = next_item(p, sPre, blockIdx.x, n_items, it); w < n_items && ok;
           w = next_item(p, sPre, w + gridDim.x, n_items, it), ++kq) {
        // O^T buffer kq & 1 was last read by the epilogue of item kq - 2
        if (kq >= 2 && !(ok = mbar_wait(o_free + (kq & 1), ((kq - 2) >> 1) & 1, abort_flag))) break;
        const uint32_t tO = tmem + Lay::kColO + (kq & 1) * Lay::kOCols;
        for (int i = 0; i < it.nt; ++i, ++gt) {
          // P^T of tile gt written, S^T buffer gt % 3 read, O^T rescaled
          if (!(ok = mbar_wait(p_ready + gt % Lay::kSBufs, (gt / Lay::kSBufs) & 1, abort_flag))) break;
          tc_fence_after();
          const uint32_t sVa = smem_u32(vtile(gt)), sPa = smem_u32(pbuf(gt));
          if constexpr (FP8) {
            // V^T: one 128-byte row of dimensions per key, 8-key groups 1 KB
            // apart; P^T: 48 rows of 128 keys; 32 keys per step
#pragma unroll
            for (int kk = 0; kk < kTile / 32; ++kk)
              umma_ss_f8(tO, sdesc_sw128(sVa + kk * 4096, 16, 1024), sdesc_sw128(sPa + kk * 32, 16, 1024), id_o,
                         (i > 0 || kk > 0));
          } else {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              umma_ss(tO, sdesc_sw128(sVa + kk * 2048, Lay::kChunkBytes, 1024),
                      sdesc_sw128(sPa + (kk / 4) * Lay::kHChunkBytes + (kk % 4) * 32, 16, 1024), id_o,
                      (i > 0 || kk > 0));
          }
          // the stage's K was read by S^T of tile gt, complete before the
          // softmax released P^T of tile gt
          umma_commit(empty + gt % NS);
          umma_commit(pv_done + (gt & 1));
        }
      }
      if (!ok) give_up();
      umma_commit(drain);
      int never = 0;
      mbar_wait(drain, 0, &never);
    }
  } else if (warp == Lay::kWarpS) {
    // ------------------------------------------------------------ S^T issuer
    if (lane == 0) {
      bool ok = true;
      uint32_t gt = 0, kq = 0;  // tiles and items so far
      DecItem it;
      for (long long w = next_item(p, sPre, blockIdx.x, n_items, it); w < n_items && ok;
           w = next_item(p, sPre, w + gridDim.x, n_items, it), ++kq) {
        // the item's query, in buffer kq & 1
        if (!(ok = mbar_wait(q_ready, kq & 1, abort_flag))) break;
        const uint32_t sQa = smem_u32(sQ + (kq & 1) * Lay::kQBytes);
        for (int i = 0; i < it.nt; ++i, ++gt) {
          // S^T buffer gt % 3 was read by the softmax of tile gt - 3 once it released P^T
          if (gt >= Lay::kSBufs && !(ok = mbar_wait(p_ready + gt % Lay::kSBufs, ((gt - Lay::kSBufs) / Lay::kSBufs) & 1,
                                                    abort_flag)))
            break;
          if (!(ok = mbar_wait(full + gt % NS, (gt / NS) & 1, abort_flag))) break;
          tc_fence_after();
          const uint32_t sKa = smem_u32(ktile(gt));
          const uint32_t tS = tmem + Lay::kColS + (gt % Lay::kSBufs) * Lay::kSCols;
          if constexpr (FP8) {
            // E4M3 K (one 128-byte row per key) x the 48 E4M3 query rows, 32 elements per step
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk)
              umma_ss_f8(tS, sdesc_sw128(sKa + kk * 32, 16, 1024), sdesc_sw128(sQa + kk * 32, 16, 1024), id_s,
                         kk > 0);
          } else {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              umma_ss(tS, sdesc_sw128(sKa + (kk / 4) * Lay::kChunkBytes + (kk % 4) * 32, 16, 1024),
                      sdesc_sw128(sQa + (kk / 4) * Lay::kHChunkBytes + (kk % 4) * 32, 16, 1024), id_s, kk > 0);
          }
          umma_commit(s_full + gt % Lay::kSBufs);
        }
      }
      if (!ok) give_up();
      umma_commit(drain);
      int never = 0;
      mbar_wait(drain, 0, &never);
    }
  } else if (warp < 6 || warp > Lay::kWarpS) {
    // ------------------------------------------------------------ softmax warpgroups
    // Warps 2-5 and 7-10: two warpgroups over the same keys, each taking half
    // of the heads (HW of them from h0), so that two warps per scheduler
    // share the per-key work.  Each has its own named barrier (1 + wg).
    constexpr int HW = HS / 2;
    const int wg = warp > Lay::kWarpS ? 1 : 0;
    const int h0 = wg * HW;
    const int bar_id = 1 + wg;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // key row of S^T, dimension row of O^T
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32);
    const int group = p.group;
    const float c = p.scale_log2;
    constexpr float kSlack = FP8 ? kDecRescaleSlackFp8 : kDecRescaleSlack;
    float* sRedW = sRed + wg * 4 * kDecHeads;
    int* sRedE = reinterpret_cast<int*>(smem + Lay::kOffRedE) + wg * 4;
    float* sInvSq = reinterpret_cast<float*>(smem + Lay::kOffInvSq) + wg * 2 * kDecHeads;
    // P^T rows of the padded heads (row % 16 >= HS, in both buffers and every
    // 16-row group) are read by the MMA but never written or used: zero them
    // once, before the first P^T is released
    if (wg == 0 && HS < kDecHeads) {
      for (int j = r; j < 2 * Lay::kPBytes / 16; j += 128)
        if ((j / 8) % kDecHeads >= HS) reinterpret_cast<uint4*>(smem + Lay::kOffP)[j] = make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async_smem();
    }
    // this warpgroup's columns of an O^T buffer: kPTerms groups of HW (FP8)
    auto ld_o = [&](uint32_t tO, uint32_t* ov) {
      if constexpr (FP8) {
        static_assert(Lay::kPTerms == 3, "three column groups");
        tmem_ld_cols3<HW>(tmem_addr(tO, lane_base, h0), tmem_addr(tO, lane_base, H + h0),
                          tmem_addr(tO, lane_base, 2 * H + h0), ov);
      } else {
        tmem_ld_cols<HW>(tmem_addr(tO, lane_base, h0), ov);
      }
    };
    auto st_o = [&](uint32_t tO, const uint32_t* ov) {
#pragma unroll
      for (int t = 0; t < (FP8 ? Lay::kPTerms : 1); ++t) tmem_st_cols<HW>(tmem_addr(tO, lane_base, t * H + h0), ov + t * HW);
    };
    // An item's query: thread r holds dims 16 (r % 8) .. +15 of head r / 8
    // (two 16-byte units; 0 past the group), fetched an item ahead.  Pairs of
    // 64-dim K/V heads: softmax warpgroup j serves K/V head 2 g + j of pair g,
    // its slot s (of HW) query head (2 g + j) G + s for s < G (G = group / 2);
    // a query of the first head holds its 64 dims in dims 0..63 and zeros
    // above, one of the second head in 64..127 and zeros below, so each score
    // reads only its own head's key.
    auto pair_qrow = [&](const DecItem& it, int slot) {  // -1: an unused slot
      const int half = slot / HW, s2 = slot % HW, G = group / 2;
      return half < 2 && s2 < G ? static_cast<long long>(it.b) * p.Hq + static_cast<long long>(2 * it.g + half) * G + s2
                                : -1ll;
    };
    auto fetch_q = [&](const DecItem& it, uint4 (&qa)[2]) {
      const int h = r / 8, sub = r % 8;
      const long long qrow =
          p.pair ? pair_qrow(it, h) : (h < group ? static_cast<long long>(it.b) * p.Hq + it.g * group + h : -1ll);
      const bool live = qrow >= 0 && (FP8 || wg == 0) && (!p.pair || (sub >= 4) == (h >= HW));
      if (live) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                                          (p.pair ? qrow * 64 + 16 * (sub & 3) : qrow * D + 16 * sub));
        qa[0] = __ldg(src);
        qa[1] = __ldg(src + 1);
      } else {
        qa[0] = qa[1] = make_uint4(0u, 0u, 0u, 0u);
      }
    };
    auto store_q = [&](int qb, const uint4 (&qa)[2]) {
      dec_store_q<FP8>(sQ + qb * Lay::kQBytes, sInvSq + qb * kDecHeads, q_ready, r, qa[0], qa[1], wg == 0, bar_id);
    };
    // FP8: per-token scales of this thread's key, copied (cp.async) into slot
    // gt % kScaleAhead of this warpgroup's ring, kScaleAhead tiles ahead of
    // their use: in a saturated memory system a load takes several tiles'
    // time.  One copy group per tile, empty or not; bit j of pf: slot j holds
    // copies.
    constexpr int kAhead = Lay::kScaleAhead;
    // index of the per-token scales of key kpos for this warpgroup's K/V head
    auto scale_index = [&](const DecItem& t, int kpos) {
      const long long row = decode_row(p, t.b, t.seq0, kpos, t.L);
      return p.pair ? row * (2 * p.Hkv) + 2 * t.g + wg : row * p.Hkv + t.g;
    };
    float2* sScale = reinterpret_cast<float2*>(smem + Lay::kOffScale) + wg * kAhead * kTile;
    uint32_t pf = 0;
    auto issue_scales = [&](const DecItem& t, int i, uint32_t slot) {
      pf &= ~(1u << slot);
      const int kpos = (t.t0 + i) * kTile + r;
      if (i < t.nt && kpos < t.L) {
        const long long si = scale_index(t, kpos);
        cp_async_4(&sScale[slot * kTile + r].x, p.k_scale + si);
        cp_async_4(&sScale[slot * kTile + r].y, p.v_scale + si);
        pf |= 1u << slot;
      }
      cp_async_commit();
    };
    // A wait that gives up must not leave the other threads at a barrier:
    // results of waits are made warp-uniform (the shuffles and TMEM accesses
    // need whole warps) and the loops end only on a vote of all 128 threads
    // of the warpgroup.
    bool ok = true;
    uint32_t gt = 0, kq = 0;  // tiles and items so far
    DecItem it;
    long long w = next_item(p, sPre, blockIdx.x, n_items, it);
    if (w < n_items) {
      uint4 qa[2];
      fetch_q(it, qa);
      store_q(0, qa);
      if constexpr (FP8) {
#pragma unroll
        for (int j = 0; j < kAhead; ++j) issue_scales(it, j, j);
      }
    }
    while (w < n_items && ok) {
      float inv_sq[HW];  // FP8: 1 / s_q of this warpgroup's heads
#pragma unroll
      for (int hh = 0; hh < HW; ++hh) inv_sq[hh] = FP8 ? sInvSq[(kq & 1) * kDecHeads + h0 + hh] : 1.f;
      // the next item's query: fetched now, stored once this item's first tile
      // is done, so that S^T can run into the next item ahead of the softmax
      DecItem nx;
      const long long w2 = next_item(p, sPre, w + gridDim.x, n_items, nx);
      uint4 qn[2] = {};
      if (w2 < n_items) fetch_q(nx, qn);
      const uint32_t tO = tmem + Lay::kColO + (kq & 1) * Lay::kOCols;
      int E = 0;  // FP8: largest biased exponent of the item's V scales so far
      float m[HW], lt[HW];
#pragma unroll
      for (int h = 0; h < HW; ++h) {
        m[h] = -INFINITY;
        lt[h] = 0.f;
      }
      for (int i = 0; i < it.nt; ++i, ++gt) {
        const int kpos = (it.t0 + i) * kTile + r;
        const bool valid = kpos < it.L;
        float sk = 1.f, sv = 1.f;
        if constexpr (FP8) {
          const uint32_t slot = gt % kAhead;
          cp_async_wait<kAhead - 1>();  // this tile's group
          if (valid) {
            if ((pf >> slot) & 1u) {
              const float2 s2 = sScale[slot * kTile + r];
              sk = s2.x;
              sv = s2.y;
            } else {  // a tile the ring did not reach (items shorter than the ring)
              const long long si = scale_index(it, kpos);
              sk = __ldg(p.k_scale + si);
              sv = __ldg(p.v_scale + si);
            }
          }
          // the slot's next tile, gt + kAhead: of this item or of the next
          const int j = i + kAhead;
          if (j < it.nt) {
            issue_scales(it, j, slot);
          } else if (w2 < n_items) {
            issue_scales(nx, j - it.nt, slot);
          } else {
            pf &= ~(1u << slot);
            cp_async_commit();
          }
        }
        const uint32_t svb = __float_as_uint(sv);
        const int ei = (FP8 && valid) ? static_cast<int>((svb >> 23) & 0xffu) : 0;  // masked keys: none
        const uint32_t sb = gt % Lay::kSBufs;
        bool wt = __all_sync(0xffffffffu, mbar_wait(s_full + sb, (gt / Lay::kSBufs) & 1, abort_flag));
        float x[HW];
        bool over = false;  // a score above its head's reference by more than the slack
        if (wt) {
          tc_fence_after();
          float sc[HW];
          const uint32_t ts = tmem + Lay::kColS + sb * Lay::kSCols;
          if constexpr (FP8) {
            uint32_t svv[3 * HW];
            tmem_ld_cols3<HW>(tmem_addr(ts, lane_base, h0), tmem_addr(ts, lane_base, H + h0),
                              tmem_addr(ts, lane_base, 2 * H + h0), svv);
#pragma unroll
            for (int h = 0; h < HW; ++h)
              sc[h] = (__uint_as_float(svv[h]) + __uint_as_float(svv[HW + h]) + __uint_as_float(svv[2 * HW + h])) *
                      inv_sq[h];
          } else {
            uint32_t svv[HW];
            tmem_ld_cols<HW>(tmem_addr(ts, lane_base, h0), svv);
#pragma unroll
            for (int h = 0; h < HW; ++h) sc[h] = __uint_as_float(svv[h]);
          }
          const float ck = c * sk;
#pragma unroll
          for (int h = 0; h < HW; ++h) {
            x[h] = valid ? sc[h] * ck : -INFINITY;
            over |= x[h] > m[h] + kSlack;  // always for a valid key on the first tile (m = -inf)
          }
          over |= ei > E;
        }
        bool bump = false;
        float beta = 1.f;  // FP8: O^T's factor for a larger E
        float alpha[HW];
#pragma unroll
        for (int h = 0; h < HW; ++h) alpha[h] = 1.f;
        // One vote per tile: in the common case no reference moves and the
        // probabilities are taken against the current m.  Otherwise (the first
        // tile, a score jump, or a wait that gave up) the tile max of every
        // head is reduced over the 128 keys.
        if (softmax_sync_or(over || !wt, bar_id)) {
          if (!(ok = softmax_sync_and(wt, bar_id))) break;
#pragma unroll
          for (int h = 0; h < HW; ++h) {
            float mx = x[h];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            if (lane == 0) sRedW[quad * H + h] = mx;
          }
          if constexpr (FP8) {
            const int em = __reduce_max_sync(0xffffffffu, ei);
            if (lane == 0) sRedE[quad] = em;
          }
          softmax_sync(bar_id);
#pragma unroll
          for (int h = 0; h < HW; ++h) {
            const float tm = fmaxf(fmaxf(sRedW[h], sRedW[H + h]), fmaxf(sRedW[2 * H + h], sRedW[3 * H + h]));
            // the tile's key 0 is valid, so tm is finite
            const bool up = tm > m[h] + kSlack;
            const float mn = up ? tm : m[h];
            alpha[h] = up ? ex2_approx(m[h] - mn) : 1.f;
            bump |= up;
            m[h] = mn;
          }
          if constexpr (FP8) {
            const int te = max(max(sRedE[0], sRedE[1]), max(sRedE[2], sRedE[3]));
            if (te > E) {
              beta = exp2i(E - te);
              bump = true;
              E = te;
            }
          }
          softmax_sync(bar_id);  // sRedW is rewritten by the next reduction
        }
        // P^T buffer gt & 1 was last read by P V of tile gt - 2
        wt = gt < 2 || __all_sync(0xffffffffu, mbar_wait(pv_done + (gt & 1), ((gt - 2) >> 1) & 1, abort_flag));
        if (wt) {
          if constexpr (FP8) {
            // s_v 2^(6 + 126 - E): the scale's exponent moved relative to 2^E
            // (below 64); 0 for a masked key or one 2^126 below the largest
            const int ne = ei + kDecPScaleLog2 + 126 - E;
            const float svs = (ei > 0 && ne > 0) ? __uint_as_float((static_cast<uint32_t>(ne) << 23) | (svb & 0x7fffffu))
                                                 : 0.f;
            // P^T row t * 16 + h, key r: 16-byte unit r / 16 of the row, swizzled
            uint8_t* pb = pbuf(gt) + (r & 15);
#pragma unroll
            for (int h = 0; h < HW; h += 2) {
              const float p0 = ex2_approx(x[h] - m[h]), p1 = ex2_approx(x[h + 1] - m[h + 1]);  // masked keys: 0
              lt[h] = fmaf(lt[h], alpha[h], p0);
              lt[h + 1] = fmaf(lt[h + 1], alpha[h + 1], p1);
              float2 y = make_float2(p0 * svs, p1 * svs);  // below 256: no saturation
#pragma unroll
              for (int t = 0; t < Lay::kPTerms; ++t) {
                const __nv_fp8x2_storage_t c2 = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
                if (t + 1 < Lay::kPTerms) {
                  const __half2_raw hb = __nv_cvt_fp8x2_to_halfraw2(c2, __NV_E4M3);
                  y.x -= __half2float(*reinterpret_cast<const __half*>(&hb.x));  // exact in f32
                  y.y -= __half2float(*reinterpret_cast<const __half*>(&hb.y));
                }
                const int row0 = t * kDecHeads + h0 + h;
                pb[row0 * 128 + ((((r >> 4) ^ (row0 & 7))) << 4)] = static_cast<uint8_t>(c2 & 0xffu);
                pb[(row0 + 1) * 128 + ((((r >> 4) ^ ((row0 + 1) & 7))) << 4)] = static_cast<uint8_t>(c2 >> 8);
              }
            }
          } else {
            uint8_t* pb = pbuf(gt) + (r / 64) * Lay::kHChunkBytes + (r % 8) * 2;
            const int pu = (r % 64) / 8;
#pragma unroll
            for (int h = 0; h < HW; ++h) {
              const float pv = ex2_approx(x[h] - m[h]);  // masked keys: 0
              lt[h] = fmaf(lt[h], alpha[h], pv);
              const __nv_bfloat16 pb16 = __float2bfloat16_rn(pv);
              const int hr = h0 + h;
              sts_u16(pb + hr * 128 + ((pu ^ (hr & 7)) << 4), *reinterpret_cast<const uint16_t*>(&pb16));
            }
          }
        }
        // m is the same in every thread of the warpgroup, so bump is uniform
        if (wt && i > 0 && bump) {
          // O^T may only be touched once P V of tile gt - 1 has completed
          wt = __all_sync(0xffffffffu, mbar_wait(pv_done + ((gt - 1) & 1), ((gt - 1) >> 1) & 1, abort_flag));
          if (wt) {
            tc_fence_after();
            constexpr int NT = FP8 ? Lay::kPTerms : 1;
            uint32_t ov[NT * HW];
            ld_o(tO, ov);
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
              for (int h = 0; h < HW; ++h)
                ov[t * HW + h] = __float_as_uint(__uint_as_float(ov[t * HW + h]) * (alpha[h] * beta));
            st_o(tO, ov);
            tmem_st_wait();
          }
        }
        if (wt) {
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(p_ready + sb);
        }
        // a warp that gave up here stops arriving; the vote of the next tile
        // (or the vote below) ends the loop for the warpgroup
        ok = wt;
        // (every thread, so that the barrier in store_q is met)
        if (i == 0 && w2 < n_items) store_q((kq + 1) & 1, qn);
      }
      if (!(ok = softmax_sync_and(ok, bar_id))) {
        if (lane == 0) give_up();
        break;
      }
      // ---- the split's output for this warpgroup's heads: O^T / l, and the LSE
#pragma unroll
      for (int h = 0; h < HW; ++h) {
        float xs = lt[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) xs += __shfl_xor_sync(0xffffffffu, xs, off);
        if (lane == 0) sRedW[quad * H + h] = xs;
      }
      softmax_sync(bar_id);
      // all four warps take the same way out: the next item has barriers
      ok = softmax_sync_and(
          __all_sync(0xffffffffu, mbar_wait(pv_done + ((gt - 1) & 1), ((gt - 1) >> 1) & 1, abort_flag)), bar_id);
      if (!ok) {
        if (lane == 0) give_up();
        break;
      }
      tc_fence_after();
      constexpr int NT = FP8 ? Lay::kPTerms : 1;
      uint32_t ov[NT * HW];
      ld_o(tO, ov);
      float osum[HW];
      // FP8: the terms' sum times 2^(E - 126 - 6), in two exact steps
      const int e = E - 126 - kDecPScaleLog2, e1 = e / 2;
      const float f1 = FP8 ? exp2i(e1) : 1.f, f2 = FP8 ? exp2i(e - e1) : 1.f;
#pragma unroll
      for (int h = 0; h < HW; ++h) {
        float s = 0.f;
#pragma unroll
        for (int t = 0; t < NT; ++t) s += __uint_as_float(ov[t * HW + h]);
        osum[h] = (s * f1) * f2;
      }
      const long long row0 = static_cast<long long>(it.b) * p.Hq + static_cast<long long>(it.g) * group;
#pragma unroll
      for (int h = 0; h < HW; ++h) {
        const int hh = h0 + h;
        if (p.pair || hh < group) {
          const float l = sRedW[h] + sRedW[H + h] + sRedW[2 * H + h] + sRedW[3 * H + h];
          const float lse = (m[h] + log2f(l)) * 0.6931471805599453f;
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.o);
          if (!p.pair) {
            const long long row = row0 + hh;  // b Hq + h
            if (p.direct) {
              // the only split of the row: the output itself (bf16) and the LSE ([Hq, B])
              o[row * D + r] = __float2bfloat16_rn(osum[h] / l);
              if (r == 0) p.lse[(row % p.Hq) * p.B + row / p.Hq] = lse;
            } else {
              p.o_part[(row * p.n_splits + it.split) * D + r] = osum[h] / l;
              if (r == 0) p.lse_part[row * p.n_splits + it.split] = lse;
            }
          } else if (const long long qr = pair_qrow(it, hh); qr >= 0) {
            // O^T rows of this warpgroup's own K/V head; the other 64 rows mix
            // in the other head's values and are dropped
            if (p.direct) {
              if ((r >= 64) == (wg == 1)) o[qr * 64 + (r & 63)] = __float2bfloat16_rn(osum[h] / l);
              if (r == 0) p.lse[(qr % p.Hq) * p.B + qr / p.Hq] = lse;
            } else {
              if ((r >= 64) == (wg == 1)) p.o_part[(qr * p.n_splits + it.split) * 64 + (r & 63)] = osum[h] / l;
              if (r == 0) p.lse_part[qr * p.n_splits + it.split] = lse;
            }
          }
        }
      }
      // O^T buffer kq & 1 read: P V of item kq + 2 may write it
      tc_fence_before();
      mbar_arrive(o_free + (kq & 1));
      it = nx;
      w = w2;
      ++kq;
    }
    // no copy into shared memory may still be in flight when the CTA exits
    if constexpr (FP8) cp_async_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

// Merges the splits of one (sequence, query head) row per warp.
template <int D>
__global__ void __launch_bounds__(128) fa_decode_combine_kernel(const DecodeParams p) {
  // launched as a programmatic dependent of the split kernel: resident early,
  // it waits here until that grid has finished and its writes are visible (a
  // no-op after an ordinary launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int E = D / 32;  // dimensions per lane
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const long long row = static_cast<long long>(blockIdx.x) * 4 + warp;  // b * Hq + h
  if (row >= static_cast<long long>(p.B) * p.Hq) return;
  const int b = static_cast<int>(row / p.Hq), h = static_cast<int>(row % p.Hq);
  int L = p.N;
  if (p.block_table != nullptr) {
    const int l = __ldg(p.seqlens + b);
    L = (l >= 0 && l <= p.max_pages * p.page_size) ? l : 0;  // bad lengths: reported by the split kernel
  } else if (p.cu != nullptr) {
    const int a = __ldg(p.cu + b), e = __ldg(p.cu + b + 1);
    L = (a >= 0 && e >= a && e <= p.T && e - a <= p.N) ? e - a : 0;  // bad offsets: reported by the split kernel
  }
  const int tiles = (L + kTile - 1) / kTile;
  const int ns = (tiles + p.split_tiles - 1) / p.split_tiles;
  const float* lp = p.lse_part + row * p.n_splits;
  const float* op = p.o_part + row * p.n_splits * D + lane * E;
  // Eight splits at a time: all their loads are issued before any is used
  // (one memory round trip per eight splits, not one per split), then they
  // join a running merge: acc and den are kept relative to the running
  // max mx and rescaled when it grows.
  constexpr int kBatch = 8;
  float mx = -INFINITY, den = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int s0 = 0; s0 < ns; s0 += kBatch) {
    float lv[kBatch], ov[kBatch][E];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int sj = s0 + j;
      lv[j] = -INFINITY;
#pragma unroll
      for (int e = 0; e < E; ++e) ov[j][e] = 0.f;
      if (sj < ns) {
        lv[j] = __ldg(lp + sj);
        const float* src = op + static_cast<long long>(sj) * D;
        if constexpr (E == 4) {
          const float4 v4 = __ldg(reinterpret_cast<const float4*>(src));
          ov[j][0] = v4.x; ov[j][1] = v4.y; ov[j][2] = v4.z; ov[j][3] = v4.w;
        } else {
          const float2 v2 = __ldg(reinterpret_cast<const float2*>(src));
          ov[j][0] = v2.x; ov[j][1] = v2.y;
        }
      }
    }
    float m2 = mx;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) m2 = fmaxf(m2, lv[j]);
    if (m2 == -INFINITY) continue;  // nothing finite yet
    const float sc = expf(mx - m2);  // 0 while mx is still -inf
    den *= sc;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] *= sc;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const float w = expf(lv[j] - m2);  // 0 for the padding entries
      den += w;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(w, ov[j][e], acc[e]);
    }
    mx = m2;
  }
  const float inv = ns > 0 ? 1.f / den : 0.f;
  uint32_t pk[E / 2];
#pragma unroll
  for (int e = 0; e < E / 2; ++e) pk[e] = pack_bf16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.o) + row * D + lane * E;
  if constexpr (E == 4) {
    *reinterpret_cast<uint2*>(o) = make_uint2(pk[0], pk[1]);
  } else {
    *reinterpret_cast<uint32_t*>(o) = pk[0];
  }
  if (lane == 0) p.lse[static_cast<long long>(h) * p.B + b] = ns > 0 ? mx + logf(den) : -INFINITY;
}

template <int D, int G>
int launch_decode_dg(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, cudaStream_t stream) {
  using Lay = DecLayout<D>;
  cudaError_t e =
      cudaFuncSetAttribute(fa_decode_split_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_splits, p.Hkv, p.B);
  note_launch();
  fa_decode_split_kernel<D, G><<<grid, 288, Lay::kBytes, stream>>>(tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long rows = static_cast<long long>(p.B) * p.Hq;
  note_launch();
  fa_decode_combine_kernel<D><<<static_cast<unsigned>((rows + 3) / 4), 128, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
int launch_decode_d(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, cudaStream_t stream) {
  // the kernel is instantiated for power-of-two groups; others round up and
  // leave the extra heads unused
  if (p.group <= 1) return launch_decode_dg<D, 1>(tk, tv, p, stream);
  if (p.group <= 2) return launch_decode_dg<D, 2>(tk, tv, p, stream);
  if (p.group <= 4) return launch_decode_dg<D, 4>(tk, tv, p, stream);
  if (p.group <= 8) return launch_decode_dg<D, 8>(tk, tv, p, stream);
  if (p.group <= 16) return launch_decode_dg<D, 16>(tk, tv, p, stream);
  return -1;
}

template <bool FP8>
int launch_decode_tc(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, cudaStream_t stream) {
  using Lay = DecTcLayout<FP8>;
  if (p.group > kDecHeads) return -1;
  auto kern = p.group <= 8 ? fa_decode_tc_kernel<FP8, 8> : fa_decode_tc_kernel<FP8, kDecHeads>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per multiprocessor (or per item, if fewer)
  const long long items = static_cast<long long>(p.n_splits) * p.Hkv * p.B;
  const unsigned grid = static_cast<unsigned>(std::min<long long>(items, std::max(p.sms, 1)));
  note_launch();
  kern<<<grid, Lay::kThreads, Lay::kBytes, stream>>>(tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.direct) return cudaSuccess;  // the split kernel wrote O and the LSE
  // the combine as a programmatic dependent launch: its CTAs are scheduled
  // while the split kernel runs and start merging as soon as it completes
  const long long rows = static_cast<long long>(p.B) * p.Hq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launch();
  return p.pair ? cudaLaunchKernelEx(&cfg, fa_decode_combine_kernel<64>, p)
                : cudaLaunchKernelEx(&cfg, fa_decode_combine_kernel<128>, p);
}

int launch_decode(int d, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, cudaStream_t stream) {
  if (d == 64 && p.pair) return launch_decode_tc<false>(tk, tv, p, stream);
  if (d == 64) return launch_decode_d<64>(tk, tv, p, stream);
  if (d == 128) return launch_decode_tc<false>(tk, tv, p, stream);
  return -1;
}

int launch_decode_fp8(int d, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                      cudaStream_t stream) {
  if (d == 128 || (d == 64 && p.pair)) return launch_decode_tc<true>(tk, tv, p, stream);
  return -1;
}

// E4M3 quantisation of [rows, D] bf16 rows ("Attention 算子优化…", section 六):
// one warp per row; s = max|x| / 448 in f32 (1 for an all-zero row),
// codes = e4m3(x / s) with round-to-nearest-even and saturation.
template <int D>
__global__ void __launch_bounds__(256) fa_quantize_fp8_kernel(const __nv_bfloat16* x, uint8_t* x8, float* scale,
                                                               long long rows) {
  constexpr int E = D / 32;  // elements per lane
  const long long row = static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  float v[E];
  const __nv_bfloat16* src = x + row * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = __bfloat162float(src[e]);
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint8_t* dst = x8 + row * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const __nv_fp8x2_storage_t two =
        __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(v[e], s), __fdiv_rn(v[e + 1], s)), __NV_SATFINITE, __NV_E4M3);
    *reinterpret_cast<__nv_fp8x2_storage_t*>(dst + e) = two;
  }
  if (lane == 0) scale[row] = s;
}

int launch_quantize_fp8(int d, const void* x, void* x8, float* scale, long long rows, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
  if (d == 64) {
    note_launch();
    fa_quantize_fp8_kernel<64><<<blocks, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x),
                                                           static_cast<uint8_t*>(x8), scale, rows);
  } else if (d == 128) {
    note_launch();
    fa_quantize_fp8_kernel<128><<<blocks, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x),
                                                            static_cast<uint8_t*>(x8), scale, rows);
  } else {
    return -1;
  }
  return cudaGetLastError();
}

}  // namespace fa
