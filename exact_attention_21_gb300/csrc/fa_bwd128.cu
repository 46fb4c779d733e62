// Backward kernel for head dimension 128.
//
// The same computation as the d = 64 kernel ("企业官网建设流程全解析", section
// 2.3; "Attention 算子优化…", section 四): for every visible (key tile j,
// query tile i) pair of a (sequence, K/V head), with c = scale * log2 e,
//     S^T  = K_j Q_i^T                 P^T = exp2(S^T * c - LSE * log2 e)
//     dP^T = V_j dO_i^T                dS^T = P^T * (dP^T - D)
//     dV_j += P^T dO_i                 dK_j += dS^T Q_i
//     dQ_i += dS K_j   (f32 bulk reduce-add into a global accumulator).
//
// At d = 128 the four 128 x 128 f32 tiles S^T, dP^T, dV and dK fill the 512
// TMEM columns of an SM, so the score tile is single-buffered and dQ_i lands
// in the dP^T region once the score warpgroups have read dP^T.  Shared memory
// (226 KB) holds K_j and V_j, the dS^T tile, one dO tile, two Q stages and a
// 32 KB dQ staging tile.  That leaves no room to round the dynamic shared
// memory base up to the 1 KB alignment of the 128-byte swizzle, so the kernel
// requires the base to be aligned (it is, with no static shared memory) and
// otherwise sets a status bit and does nothing.
// The score warpgroups work in two phases so the tensor core is not idle
// while they run: phase 1 turns S^T into P^T (TMEM, bf16) as soon as S^T is
// ready, which lets dV += P^T dO start; phase 2 waits for dP^T, re-reads P^T
// and writes dS^T to shared memory, which releases dK and dQ.
//
// One CTA per (key tile, K/V head, sequence); it walks the query heads of the
// group and their query tiles ("steps").  Warp roles:
//   warp 0       producer: K_j, V_j once; per step Q_i (two stages, with the
//                LSE / D values of the tile) and dO_i (one stage), by TMA.
//   warp 1       TMEM allocator and MMA issuer (one thread).  Per step:
//                S^T; dP^T (after dO_i and the read-out of the previous dQ);
//                dV (after phase 1); dK, dQ (after phase 2).
//   warps 2..9   two score warpgroups: thread = key row (TMEM lane); the
//                first takes query columns 0..63, the second 64..127; dV / dK
//                epilogue.
//   warps 10..13 dQ warpgroup: dQ tile TMEM -> registers -> swizzled shared
//                memory -> TMA bulk reduce-add (f32), in two batches of 64
//                columns; the TMEM region is released once the second batch
//                is in registers.
// TMEM: S^T / P^T [0, 128) (P^T of queries 0..63 over columns 0..31, of
// queries 64..127 over 64..95), dP^T / dQ [128, 256), dV [256, 384),
// dK [384, 512).
#include <cuda_bf16.h>

#include "fa_common.cuh"

namespace fa {

struct Bwd128Layout {
  static constexpr int D = 128;
  static constexpr int kChunkBytes = kTile * 128;     // 128 rows x 64 bf16: one 128-byte swizzle column
  static constexpr int kTileBytes = 2 * kChunkBytes;  // 128 x 128 bf16
  static constexpr int kQStages = 2;
  static constexpr int kStatBytes = 2 * kTile * 4;    // -LSE log2 e [128], -D [128]
  static constexpr int kDQBoxBytes = kTile * 32 * 4;  // 128 queries x 32 f32: one TMA reduce box
  static constexpr int kDQBytes = 2 * kDQBoxBytes;    // staging for 64 dQ columns
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffDS = kOffV + kTileBytes;
  static constexpr int kOffDO = kOffDS + kTileBytes;
  static constexpr int kOffQ = kOffDO + kTileBytes;
  static constexpr int kOffDQ = kOffQ + kQStages * kTileBytes;
  static constexpr int kOffStats = kOffDQ + kDQBytes;
  static constexpr int kOffBar = kOffStats + kQStages * kStatBytes;
  // kv_full, q_full[2], q_empty[2], do_full, do_empty, s_full, dp_full, p_ready,
  // ds_ready, dq_full, dq_free, dq_staged, dq_stage_free, epi, drain
  static constexpr int kNumBars = 1 + 2 * kQStages + 14;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

// DQ = false compiles the dQ product and the dQ warpgroup out (the
// deterministic backward computes dQ in a separate kernel).
template <bool DQ>
__global__ void __launch_bounds__(448, 1)
fa_bwd128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                 const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using Lay = Bwd128Layout;
  constexpr int D = Lay::D;
  constexpr int NQ = Lay::kQStages;

  const int g = blockIdx.x;  // K/V head
  const int kt = blockIdx.y;
  const int s = blockIdx.z;
  long long seq0;
  int L;
  if (!sequence_bounds(p.cu, s, p.N, p.T, seq0, L, p.status)) return;
  const int k0 = kt * kTile;
  if (k0 >= L) return;
  const bool causal = p.causal != 0;
  const int nqt = (L + kTile - 1) / kTile;
  const int i0 = first_q_tile_for(kt, causal);
  const int per_head = nqt - i0;
  const int nsteps = p.group * per_head;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusSmemAlign);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sK = smem + Lay::kOffK;
  uint8_t* sV = smem + Lay::kOffV;
  uint8_t* sDS = smem + Lay::kOffDS;
  uint8_t* sDO = smem + Lay::kOffDO;
  uint8_t* sDQ = smem + Lay::kOffDQ;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBar);
  uint64_t* kv_full = bars;
  uint64_t* q_full = kv_full + 1;
  uint64_t* q_empty = q_full + NQ;
  uint64_t* do_full = q_empty + NQ;
  uint64_t* do_empty = do_full + 1;
  uint64_t* s_full = do_empty + 1;
  uint64_t* dp_full = s_full + 1;
  uint64_t* p_ready = dp_full + 1;
  uint64_t* ds_ready = p_ready + 1;
  uint64_t* dq_full = ds_ready + 1;
  uint64_t* dq_free = dq_full + 1;
  uint64_t* dq_staged = dq_free + 1;
  uint64_t* dq_stage_free = dq_staged + 1;
  uint64_t* epi = dq_stage_free + 1;
  uint64_t* drain = epi + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kOffMisc + 4);

  auto stage_q = [&](int st) { return smem + Lay::kOffQ + st * Lay::kTileBytes; };
  auto stage_stats = [&](int st) { return reinterpret_cast<float*>(smem + Lay::kOffStats + st * Lay::kStatBytes); };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < NQ; ++i) { mbar_init(q_full + i, 32); mbar_init(q_empty + i, 1); }
    mbar_init(do_full, 1);
    mbar_init(do_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_ready, 256);
    mbar_init(ds_ready, 256);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 128);
    mbar_init(dq_staged, 128);
    mbar_init(dq_stage_free, 1);
    mbar_init(epi, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Lay::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto give_up = [&]() {
    atomicOr(p.status, kStatusTimeout);
    *abort_flag = 1;
  };
  // step n -> (query head, query tile)
  auto step_head = [&](int n) { return g * p.group + n / per_head; };
  auto step_qtile = [&](int n) { return i0 + n % per_head; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_dq);
      mbar_arrive_expect_tx(kv_full, 2 * Lay::kTileBytes);
      for (int c = 0; c < 2; ++c) {
        tma_load_3d(sK + c * Lay::kChunkBytes, &tm_k, kv_full, c * 64, g, static_cast<int>(seq0 + k0));
        tma_load_3d(sV + c * Lay::kChunkBytes, &tm_v, kv_full, c * 64, g, static_cast<int>(seq0 + k0));
      }
    }
    int q_uses[NQ] = {};
    int do_uses = 0;
    bool ok = true;
    for (int n = 0; n < nsteps; ++n) {
      const int st = n % NQ;
      const int h = step_head(n), q0 = step_qtile(n) * kTile;
      const int row = static_cast<int>(seq0 + q0);
      // Q_n and its statistics: the stage was last read by dK of step n - 2
      if (n >= NQ && !(ok = mbar_wait(q_empty + st, ((n / NQ) - 1) & 1, abort_flag))) break;
      if (lane == 0) {
        mbar_expect_tx(q_full + st, Lay::kTileBytes);
        for (int c = 0; c < 2; ++c)
          tma_load_3d(stage_q(st) + c * Lay::kChunkBytes, &tm_q, q_full + st, c * 64, h, row);
      }
      float* stats = stage_stats(st);
      const long long lrow = static_cast<long long>(h) * p.T + seq0 + q0;
      float lv[kTile / 32], dv[kTile / 32];
#pragma unroll
      for (int t = 0; t < kTile / 32; ++t) {
        const int idx = lane + 32 * t;
        const bool valid = q0 + idx < L;
        lv[t] = valid ? __ldg(p.lse + lrow + idx) : INFINITY;
        dv[t] = valid ? __ldg(p.rowdot + lrow + idx) : 0.f;
      }
#pragma unroll
      for (int t = 0; t < kTile / 32; ++t) {
        // stored negated: -LSE * log2 e and -D (queries past the end: P = 0)
        stats[lane + 32 * t] = -lv[t] * kLog2e;
        stats[kTile + lane + 32 * t] = -dv[t];
      }
      mbar_arrive(q_full + st);
      ++q_uses[st];
      // dO_n: the single buffer was last read by dV of step n - 1
      if (n >= 1 && !(ok = mbar_wait(do_empty, (n - 1) & 1, abort_flag))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(do_full, Lay::kTileBytes);
        for (int c = 0; c < 2; ++c) tma_load_3d(sDO + c * Lay::kChunkBytes, &tm_do, do_full, c * 64, h, row);
      }
      ++do_uses;
    }
    if (!ok && lane == 0) give_up();
    if (lane == 0) {
      // no TMA write may still be in flight when the CTA exits
      int never = 0;
      mbar_wait(kv_full, 0, &never);
      for (int i = 0; i < NQ; ++i)
        if (q_uses[i]) mbar_wait(q_full + i, (q_uses[i] - 1) & 1, &never);
      if (do_uses) mbar_wait(do_full, (do_uses - 1) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_kk = idesc_bf16_f32(kTile, kTile, false, false);  // K-major x K-major
      constexpr uint32_t id_tmn = idesc_bf16_f32(kTile, D, false, true);      // (TMEM or K-major) A x MN-major B
      constexpr uint32_t id_mnmn = idesc_bf16_f32(kTile, D, true, true);      // MN-major A x MN-major B
      const uint32_t sKa = smem_u32(sK), sVa = smem_u32(sV), sDSa = smem_u32(sDS), sDOa = smem_u32(sDO);
      bool ok = mbar_wait(kv_full, 0, abort_flag);
      int issued = 0;  // steps whose S^T this thread issued
      for (int n = 0; n < nsteps && ok; ++n) {
        const int st = n % NQ;
        const uint32_t sQa = smem_u32(stage_q(st));
        // S^T = K Q^T.  The S region was last read by dV and by phase 2 of
        // step n - 1, both before ds_ready of that step.
        if (!(ok = mbar_wait(q_full + st, (n / NQ) & 1, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * Lay::kChunkBytes + (kk % 4) * 32;
          umma_ss(tmem + Lay::kColS, sdesc_sw128(sKa + off, 16, 1024), sdesc_sw128(sQa + off, 16, 1024), id_kk,
                  kk > 0);
        }
        umma_commit(s_full);
        ++issued;
        // dP^T = V dO^T into the region the previous dQ has been read out of
        if (!(ok = mbar_wait(do_full, n & 1, abort_flag))) break;
        if (DQ && n >= 1 && !(ok = mbar_wait(dq_free, (n - 1) & 1, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * Lay::kChunkBytes + (kk % 4) * 32;
          umma_ss(tmem + Lay::kColDP, sdesc_sw128(sVa + off, 16, 1024), sdesc_sw128(sDOa + off, 16, 1024), id_kk,
                  kk > 0);
        }
        umma_commit(dp_full);
        // dV += P^T dO  (A: P^T in TMEM; B: dO rows = queries = K, MN-major)
        if (!(ok = mbar_wait(p_ready, n & 1, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ts(tmem + Lay::kColDV, tmem + Lay::kColS + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8),
                  sdesc_sw128(sDOa + kk * 2048, Lay::kChunkBytes, 1024), id_tmn, (n > 0 || kk > 0));
        umma_commit(do_empty);
        // dK += dS^T Q  (A: dS^T, rows = keys, K-major; B: Q rows = K, MN-major)
        if (!(ok = mbar_wait(ds_ready, n & 1, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ss(tmem + Lay::kColDK, sdesc_sw128(sDSa + (kk / 4) * Lay::kChunkBytes + (kk % 4) * 32, 16, 1024),
                  sdesc_sw128(sQa + kk * 2048, Lay::kChunkBytes, 1024), id_tmn, (n > 0 || kk > 0));
        umma_commit(q_empty + st);
        if constexpr (DQ) {
          // dQ_n = dS K into the dP^T region, which phase 2 has finished reading
          // (A: the dS^T tile read query-major, MN-major; B: K, MN-major)
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_ss(tmem + Lay::kColDP, sdesc_sw128(sDSa + kk * 2048, Lay::kChunkBytes, 1024),
                    sdesc_sw128(sKa + kk * 2048, Lay::kChunkBytes, 1024), id_mnmn, kk > 0);
          umma_commit(dq_full);
        }
      }
      if (p.tile_count != nullptr && issued > 0)
        atomicAdd(p.tile_count + s, static_cast<unsigned long long>(issued));
      if (ok) umma_commit(epi);
      if (!ok) give_up();
      umma_commit(drain);
      int never = 0;
      mbar_wait(drain, 0, &never);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ score warpgroups
    const int half = (warp - 2) / 4;  // query columns [64 * half, 64 * half + 64)
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // key row within the tile
    const int kpos = k0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32);
    const float c = p.scale_log2;
    const float2 c2 = make_float2(c, c);
    const bool key_ok = kpos < L;
    bool ok = true;
    for (int n = 0; n < nsteps; ++n) {
      const int st = n % NQ;
      if (!(ok = mbar_wait(s_full, n & 1, abort_flag))) break;
      if (!(ok = mbar_wait(q_full + st, (n / NQ) & 1, abort_flag))) break;
      tc_fence_after();
      const float2* nlse2 = reinterpret_cast<const float2*>(stage_stats(st)) + half * 32;
      const float2* ndot2 = nlse2 + kTile / 2;
      const int q0 = step_qtile(n) * kTile;
      // Keys past the sequence end and keys after the query (diagonal tile,
      // causal) get P = 0: query columns below zero_below are zeroed.
      // Queries past the end carry -LSE = -inf, so their P is 0 already.
      const int zero_below = !key_ok ? kTile : ((causal && q0 == k0) ? r : 0);
      // ---- phase 1: P^T = exp2(S^T c - LSE log2 e), bf16, over S^T columns
      // this thread has already read
#pragma unroll
      for (int cl = 0; cl < 2; ++cl) {
        const int col0 = half * 64 + cl * 32;
        uint32_t sv[32];
        tmem_ld_x32(tmem_addr(tmem + Lay::kColS, lane_base, col0), sv);
        uint32_t pk[16];
        const bool mask_chunk = zero_below > col0;
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float2 x =
              fma2(make_float2(__uint_as_float(sv[2 * t]), __uint_as_float(sv[2 * t + 1])), c2, nlse2[cl * 16 + t]);
          float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          if (mask_chunk) {
            if (col0 + 2 * t < zero_below) pv.x = 0.f;
            if (col0 + 2 * t + 1 < zero_below) pv.y = 0.f;
          }
          pk[t] = pack_bf16x2(pv.x, pv.y);
        }
        tmem_st_x16(tmem_addr(tmem + Lay::kColS, lane_base, half * 64 + cl * 16), pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_ready);
      // ---- phase 2: dS^T = P^T (dP^T - D), from the bf16 P^T just written
      if (!(ok = mbar_wait(dp_full, n & 1, abort_flag))) break;
      tc_fence_after();
      uint8_t* ds_row = sDS + half * Lay::kChunkBytes + r * 128;
#pragma unroll
      for (int cl = 0; cl < 2; ++cl) {
        const int col0 = half * 64 + cl * 32;
        uint32_t pp[16], dpv[32];
        tmem_ld_x16_x32_pair(tmem_addr(tmem + Lay::kColS, lane_base, half * 64 + cl * 16), pp,
                             tmem_addr(tmem + Lay::kColDP, lane_base, col0), dpv);
        uint32_t dsk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          __nv_bfloat162 pb = *reinterpret_cast<const __nv_bfloat162*>(&pp[t]);
          const float2 pv = __bfloat1622float2(pb);
          const float2 dd = mul2(
              pv, add2(make_float2(__uint_as_float(dpv[2 * t]), __uint_as_float(dpv[2 * t + 1])), ndot2[cl * 16 + t]));
          dsk[t] = pack_bf16x2(dd.x, dd.y);
        }
        // dS^T row r into the 128B-swizzled tile (query-contiguous rows).
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          const int u = cl * 4 + u4;
          *reinterpret_cast<uint4*>(ds_row + ((u ^ (r & 7)) << 4)) =
              make_uint4(dsk[4 * u4], dsk[4 * u4 + 1], dsk[4 * u4 + 2], dsk[4 * u4 + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(ds_ready);
    }
    if (ok) ok = mbar_wait(epi, 0, abort_flag);
    if (!ok) {
      give_up();
    } else {
      tc_fence_after();
      // first warpgroup stores dV, second stores dK (scaled)
      const bool row_ok = kpos < L;
      const long long tok = seq0 + kpos;
      const uint32_t col = half == 0 ? Lay::kColDV : Lay::kColDK;
      const float mul = half == 0 ? 1.f : p.scale;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(half == 0 ? p.dv : p.dk) + (tok * p.Hkv + g) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        tmem_ld_x32(tmem_addr(tmem, lane_base, col + cc * 32), v);
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
          pk[t] = pack_bf16x2(__uint_as_float(v[2 * t]) * mul, __uint_as_float(v[2 * t + 1]) * mul);
        if (row_ok) {
          uint4* o4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
          for (int t = 0; t < 4; ++t) o4[t] = make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
        }
      }
    }
  } else if (DQ) {
    // ------------------------------------------------------------ dQ warpgroup
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // query row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32);
    const bool issuer = (warp == 10 && lane == 0);
    bool ok = true;
    for (int n = 0; n < nsteps && ok; ++n) {
      if (!(ok = mbar_wait(dq_full, n & 1, abort_flag))) break;
      tc_fence_after();
      const int h = step_head(n), q0 = step_qtile(n) * kTile;
      uint32_t v[64];
      tmem_ld_x64(tmem_addr(tmem + Lay::kColDP, lane_base, 0), v);
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int use = 2 * n + b;  // staging-tile use counter
        // the previous batch's reduces have finished reading the staging tile
        if (use > 0 && !(ok = mbar_wait(dq_stage_free, (use - 1) & 1, abort_flag))) break;
        // two f32 boxes of 32 columns x 128 rows, 128-byte swizzle
#pragma unroll
        for (int box = 0; box < 2; ++box) {
          uint8_t* row = sDQ + box * Lay::kDQBoxBytes + r * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(row + ((u ^ (r & 7)) << 4)) = make_uint4(
                v[32 * box + 4 * u], v[32 * box + 4 * u + 1], v[32 * box + 4 * u + 2], v[32 * box + 4 * u + 3]);
        }
        fence_proxy_async_smem();
        if (b == 0) {
          // second batch into registers; then the dP^T / dQ region is free
          tmem_ld_x64(tmem_addr(tmem + Lay::kColDP, lane_base, 64), v);
          tc_fence_before();
          mbar_arrive(dq_free);
        }
        mbar_arrive(dq_staged);
        if (issuer) {
          if (!(ok = mbar_wait(dq_staged, use & 1, abort_flag))) break;
          // Rows past the sequence end hold exact zeros (P = 0 there), so the
          // whole tile can be added; rows past T are clipped by the TMA unit.
          for (int box = 0; box < 2; ++box)
            tma_reduce_add_3d(&tm_dq, sDQ + box * Lay::kDQBoxBytes, 64 * b + 32 * box, h,
                              static_cast<int>(seq0 + q0));
          bulk_commit_group();
          bulk_wait_group_read0();
          mbar_arrive(dq_stage_free);
        }
      }
    }
    if (issuer) bulk_wait_group0();
    if (!ok) give_up();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

int launch_bwd128_main(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& tdq, const BwdParams& p, bool dq, cudaStream_t stream) {
  using Lay = Bwd128Layout;
  auto kern = dq ? fa_bwd128_kernel<true> : fa_bwd128_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(p.Hkv, p.n_kvtiles, p.B);
  note_launch();
  kern<<<grid, 448, Lay::kBytes, stream>>>(tq, tk, tv, tdo, tdq, p);
  return cudaGetLastError();
}

}  // namespace fa
