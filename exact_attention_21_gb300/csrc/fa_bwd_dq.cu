// dQ of the deterministic backward.
//
// What it computes ("企业官网建设流程全解析", section 2.3; "Attention 算子优化…",
// section 四 on recomputation): for query tile i of a (sequence, query head),
// over the visible key tiles j in ascending order,
//     S  = Q_i K_j^T                 P  = exp2(S c - LSE log2 e)
//     dP = dO_i V_j^T                dS = P * (dP - D)
//     dQ_i += dS K_j
// and finally dQ_i = scale * dQ_i in bf16.  Every row of dQ is accumulated in
// TMEM by one CTA in a fixed order, so the result does not depend on the
// order in which CTAs run (the fast backward sums dQ across key-tile CTAs with
// bulk reduce-adds instead).  S and dP are recomputed here: 3 of the 5
// products of a tile pair, on top of the dK/dV kernel's 4.
//
// One CTA per (query tile, query head, sequence), heaviest causal tiles
// first.  Warp roles:
//   warp 0     producer: Q_i and dO_i once, K_j and V_j through a ring (TMA).
//   warp 1     TMEM allocator and MMA issuer (one thread).
//   warps 2-5  score warpgroup: thread = query row (TMEM lane): P and dS from
//              S and dP, dS written back to TMEM as bf16 over S columns it has
//              already read; the dQ epilogue.
// TMEM: S / dS [0, 128), dP [128, 256), dQ [256, 256 + d).
#include <cuda_bf16.h>

#include "fa_common.cuh"

namespace fa {

template <int D>
struct BwdDqLayout {
  static constexpr int kChunkBytes = kTile * 128;  // 128 rows x 64 bf16, 128-byte swizzle
  static constexpr int kTileBytes = (D / 64) * kChunkBytes;
  static constexpr int kStages = D == 64 ? 4 : 2;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K_j, V_j
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kOffQ + kTileBytes;
  static constexpr int kOffRing = kOffDO + kTileBytes;
  static constexpr int kOffBar = kOffRing + kStages * kStageBytes;
  // qdo_full, full[], empty[], sdp_full, ds_ready, dq_done, drain
  static constexpr int kNumBars = 5 + 2 * kStages;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256;
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(192, 1)
fa_bwd_dq_det_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdParams p) {
  using Lay = BwdDqLayout<D>;
  constexpr int NS = Lay::kStages;

  const int qt = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);  // heaviest first
  const int h = blockIdx.y;
  const int s = blockIdx.z;
  long long seq0;
  int L;
  if (!sequence_bounds(p.cu, s, p.N, p.T, seq0, L, p.status)) return;
  const int q0 = qt * kTile;
  if (q0 >= L) return;
  const bool causal = p.causal != 0;
  const int nkv = kv_tiles_for(qt, L, causal);
  const int g = h / p.group;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Lay::kOffQ;
  uint8_t* sDO = smem + Lay::kOffDO;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBar);
  uint64_t* qdo_full = bars;
  uint64_t* full = qdo_full + 1;
  uint64_t* empty = full + NS;
  uint64_t* sdp_full = empty + NS;
  uint64_t* ds_ready = sdp_full + 1;
  uint64_t* dq_done = ds_ready + 1;
  uint64_t* drain = dq_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kOffMisc + 4);
  auto stage_k = [&](int st) { return smem + Lay::kOffRing + st * Lay::kStageBytes; };
  auto stage_v = [&](int st) { return stage_k(st) + Lay::kTileBytes; };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(qdo_full, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, 1);
    }
    mbar_init(sdp_full, 1);
    mbar_init(ds_ready, 128);
    mbar_init(dq_done, 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      const int qrow = static_cast<int>(seq0 + q0);
      mbar_arrive_expect_tx(qdo_full, 2 * Lay::kTileBytes);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(sQ + c * Lay::kChunkBytes, &tm_q, qdo_full, c * 64, h, qrow);
        tma_load_3d(sDO + c * Lay::kChunkBytes, &tm_do, qdo_full, c * 64, h, qrow);
      }
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < nkv; ++j) {
        const int st = j % NS;
        if (j >= NS && !(ok = mbar_wait(empty + st, ((j / NS) - 1) & 1, abort_flag))) break;
        mbar_arrive_expect_tx(full + st, Lay::kStageBytes);
        const int krow = static_cast<int>(seq0 + static_cast<long long>(j) * kTile);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(stage_k(st) + c * Lay::kChunkBytes, &tm_k, full + st, c * 64, g, krow);
          tma_load_3d(stage_v(st) + c * Lay::kChunkBytes, &tm_v, full + st, c * 64, g, krow);
        }
        ++issued;
      }
      if (!ok) give_up();
      // no TMA write may still be in flight when the CTA exits
      int never = 0;
      mbar_wait(qdo_full, 0, &never);
      for (int j = issued > NS ? issued - NS : 0; j < issued; ++j) mbar_wait(full + j % NS, (j / NS) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(kTile, kTile, false, false);  // Q, K: K-major
      constexpr uint32_t id_dq = idesc_bf16_f32(kTile, D, false, true);      // dS (TMEM) x K (MN-major)
      const uint32_t sQa = smem_u32(sQ), sDOa = smem_u32(sDO);
      bool ok = mbar_wait(qdo_full, 0, abort_flag);
      for (int j = 0; j < nkv && ok; ++j) {
        const int st = j % NS;
        // S and dP of tile j overwrite what the score warpgroup of tile j - 1
        // read before ds_ready, and dS of tile j - 1, which dQ (issued
        // before, in order) reads first
        if (!(ok = mbar_wait(full + st, (j / NS) & 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t sKa = smem_u32(stage_k(st)), sVa = smem_u32(stage_v(st));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * Lay::kChunkBytes + (kk % 4) * 32;
          umma_ss(tmem + Lay::kColS, sdesc_sw128(sQa + off, 16, 1024), sdesc_sw128(sKa + off, 16, 1024), id_s,
                  kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * Lay::kChunkBytes + (kk % 4) * 32;
          umma_ss(tmem + Lay::kColDP, sdesc_sw128(sDOa + off, 16, 1024), sdesc_sw128(sVa + off, 16, 1024), id_s,
                  kk > 0);
        }
        umma_commit(sdp_full);
        if (!(ok = mbar_wait(ds_ready, j & 1, abort_flag))) break;
        tc_fence_after();
        // dQ += dS K_j  (A: bf16 dS over S columns 0..63; B: K_j rows = keys = K, MN-major)
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ts(tmem + Lay::kColDQ, tmem + Lay::kColS + kk * 8, sdesc_sw128(sKa + kk * 2048, Lay::kChunkBytes, 1024),
                  id_dq, (j > 0 || kk > 0));
        umma_commit(empty + st);
      }
      if (ok) umma_commit(dq_done);
      if (!ok) give_up();
      umma_commit(drain);
      int never = 0;
      mbar_wait(drain, 0, &never);
    }
  } else {
    // ------------------------------------------------------------ score warpgroup
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // query row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32);
    const int qpos = q0 + r;
    const bool row_ok = qpos < L;
    const long long srow = static_cast<long long>(h) * p.T + seq0 + qpos;
    // -LSE log2 e and -D of this row; rows past the end get P = 0
    const float nl = row_ok ? -__ldg(p.lse + srow) * kLog2e : -INFINITY;
    const float nd = row_ok ? -__ldg(p.rowdot + srow) : 0.f;
    const float c = p.scale_log2;
    const float2 c2 = make_float2(c, c), nl2 = make_float2(nl, nl), nd2 = make_float2(nd, nd);
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      if (!(ok = mbar_wait(sdp_full, j & 1, abort_flag))) break;
      tc_fence_after();
      // key columns at or past lim are masked: past the sequence end, and
      // after the query on the diagonal tile
      const int k0 = j * kTile;
      int lim = min(kTile, L - k0);
      if (causal) lim = min(lim, qpos - k0 + 1);
#pragma unroll
      for (int cl = 0; cl < 4; ++cl) {
        uint32_t sv[32], dpv[32];
        tmem_ld_x32_pair(tmem_addr(tmem + Lay::kColS, lane_base, cl * 32), sv,
                         tmem_addr(tmem + Lay::kColDP, lane_base, cl * 32), dpv);
        uint32_t dsk[16];
        const bool mask_chunk = lim < (cl + 1) * 32;
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float2 x = fma2(make_float2(__uint_as_float(sv[2 * t]), __uint_as_float(sv[2 * t + 1])), c2, nl2);
          float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          if (mask_chunk) {
            if (cl * 32 + 2 * t >= lim) pv.x = 0.f;
            if (cl * 32 + 2 * t + 1 >= lim) pv.y = 0.f;
          }
          const float2 dd =
              mul2(pv, add2(make_float2(__uint_as_float(dpv[2 * t]), __uint_as_float(dpv[2 * t + 1])), nd2));
          dsk[t] = pack_bf16x2(dd.x, dd.y);
        }
        // dS over S columns this thread has already read (cl * 16 < (cl + 1) * 32)
        tmem_st_x16(tmem_addr(tmem + Lay::kColS, lane_base, cl * 16), dsk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(ds_ready);
    }
    if (ok) ok = mbar_wait(dq_done, 0, abort_flag);
    if (!ok) {
      give_up();
    } else {
      tc_fence_after();
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.dq) + ((seq0 + qpos) * p.Hq + h) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        tmem_ld_x32(tmem_addr(tmem + Lay::kColDQ, lane_base, cc * 32), v);
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
          pk[t] = pack_bf16x2(__uint_as_float(v[2 * t]) * p.scale, __uint_as_float(v[2 * t + 1]) * p.scale);
        if (row_ok) {
          uint4* o4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
          for (int t = 0; t < 4; ++t) o4[t] = make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

template <int D>
int launch_bwd_dq_det_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                        const BwdParams& p, cudaStream_t stream) {
  using Lay = BwdDqLayout<D>;
  cudaError_t e =
      cudaFuncSetAttribute(fa_bwd_dq_det_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_kvtiles, p.Hq, p.B);  // query tiles: the same count as key tiles
  note_launch();
  fa_bwd_dq_det_kernel<D><<<grid, 192, Lay::kBytes, stream>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

int launch_bwd_dq_det(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream) {
  if (d == 64) return launch_bwd_dq_det_d<64>(tq, tk, tv, tdo, p, stream);
  if (d == 128) return launch_bwd_dq_det_d<128>(tq, tk, tv, tdo, p, stream);
  return -1;
}

}  // namespace fa
