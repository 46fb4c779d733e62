// Forward kernel: tiled exact attention with the online-softmax recurrence.
//
// What it computes ("FlashAttention：从 Safe Softmax 到分块计算", sections 3.2
// and 7; "企业官网建设流程全解析", section 2.1): for a 128-row query tile Q_i
// and each visible 128-row key tile j,
//     S     = Q_i K_j^T                      (tcgen05, f32 in TMEM)
//     m_new = max(m, rowmax(S) * c)          (c = scale * log2 e)
//     P     = exp2(S * c - m_new)            (bf16, written back to TMEM)
//     l     = exp2(m - m_new) * l + rowsum(P)
//     O     = exp2(m - m_new) * O + P V_j    (tcgen05, f32 in TMEM)
// and at the end O / l (bf16) and LSE = (m + log2 l) * ln 2.  Base 2 with
// log2 e folded into c is the same function as the pages' base-e form.
//
// The reference max m is moved only when a row's max grows by more than
// kRescaleSlack (in log2 units); otherwise P is taken against the older,
// smaller reference (values up to 2^kRescaleSlack) and O, l need no rescale.
// The merge rule holds for any common reference, so the result is the same
// exact attention; this only skips O rescales that would multiply by nearly 1.
//
// One CTA owns two consecutive 128-row query tiles of one (query head,
// sequence).  Warp roles:
//   warp 0      TMA producer: both Q tiles once, then K_j and V_j through rings.
//   warp 1      TMEM allocator and MMA issuer (one thread).
//   warps 2..5  softmax of query tile 0; warps 6..9 softmax of query tile 1.
//               Thread t of a warpgroup owns query row 32 * (warp % 4) + lane,
//               i.e. that TMEM lane, so row max and row sum stay in-thread;
//               each warpgroup also rescales its O and writes its output.
// MMA order: S0_0, S1_0, then per key tile j: PV0_j, S0_{j+1}, PV1_j, S1_{j+1}.
// While one warpgroup turns S_t into P_t, the tensor core works on the other
// tile, so the exponentials overlap the matrix products.
//
// TMEM (512 columns): S0 [0, 128), S1 [128, 256) (each with its bf16 P over
// its first 64 columns once read), O0 [256, 256 + d), O1 [256 + d, 256 + 2d).
#include <cuda_bf16.h>

#include "fa_common.cuh"

namespace fa {

template <int D>
struct FwdLayout {
  static constexpr int kChunkBytes = kTile * 128;          // 128 rows x 64 bf16 (one SW128 box)
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kChunks * kChunkBytes;  // one 128 x D bf16 tile
  static constexpr int kStagesK = D == 128 ? 2 : 4;
  static constexpr int kStagesV = D == 128 ? 2 : 3;
  static constexpr int kOffQ = 0;  // two query tiles
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kStagesK * kTileBytes;
  static constexpr int kOffBar = kOffV + kStagesV * kTileBytes;
  // q_full, k_full[], k_empty[], v_full[], v_empty[], s_full[2], p_full[2], o_final[2], drain
  static constexpr int kNumBars = 1 + 2 * kStagesK + 2 * kStagesV + 2 + 2 + 2 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColO = 256;
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleSlack = 8.f;  // P values stay below 2^8 between rescales

template <int D>
__global__ void __launch_bounds__(320, 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using Lay = FwdLayout<D>;
  constexpr int NK = Lay::kStagesK, NV = Lay::kStagesV;

  const int h = blockIdx.x;
  const int pair = p.n_qtiles - 1 - static_cast<int>(blockIdx.y);  // longest rows first
  const int s = blockIdx.z;
  long long seq0;
  int L;
  if (!sequence_bounds(p.cu, s, p.N, p.T, seq0, L, p.status)) return;
  const int q0 = pair * 2 * kTile;
  if (q0 >= L) return;  // uniform across the CTA
  const bool causal = p.causal != 0;
  // key tiles seen by each query tile (0 when the tile starts past the end)
  const int nkv0 = kv_tiles_for(2 * pair, L, causal);
  const int nkv1 = q0 + kTile < L ? kv_tiles_for(2 * pair + 1, L, causal) : 0;
  const int nkv = nkv0 > nkv1 ? nkv0 : nkv1;
  const int kvh = h / p.group;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Lay::kOffQ;
  uint8_t* sK = smem + Lay::kOffK;
  uint8_t* sV = smem + Lay::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  uint64_t* s_full = v_empty + NV;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_final = p_full + 2;
  uint64_t* drain = o_final + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kOffMisc + 4);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NK; ++i) { mbar_init(k_full + i, 1); mbar_init(k_empty + i, 1); }
    for (int i = 0; i < NV; ++i) { mbar_init(v_full + i, 1); mbar_init(v_empty + i, 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(s_full + i, 1); mbar_init(p_full + i, 128); mbar_init(o_final + i, 1); }
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(q_full, 2 * Lay::kTileBytes);
      for (int t = 0; t < 2; ++t)
        for (int c = 0; c < Lay::kChunks; ++c)
          tma_load_3d(sQ + t * Lay::kTileBytes + c * Lay::kChunkBytes, &tm_q, q_full, c * 64, h,
                      static_cast<int>(seq0 + q0 + t * kTile));
      int k_uses[NK] = {}, v_uses[NV] = {};
      bool ok = true;
      for (int j = 0; j < nkv && ok; ++j) {
        const int row_k = static_cast<int>(seq0 + j * kTile);
        const int ks = j % NK, vs = j % NV;
        if (j >= NK && !(ok = mbar_wait(k_empty + ks, ((j / NK) - 1) & 1, abort_flag))) break;
        mbar_arrive_expect_tx(k_full + ks, Lay::kTileBytes);
        for (int c = 0; c < Lay::kChunks; ++c)
          tma_load_3d(sK + ks * Lay::kTileBytes + c * Lay::kChunkBytes, &tm_k, k_full + ks, c * 64, kvh, row_k);
        ++k_uses[ks];
        if (j >= NV && !(ok = mbar_wait(v_empty + vs, ((j / NV) - 1) & 1, abort_flag))) break;
        mbar_arrive_expect_tx(v_full + vs, Lay::kTileBytes);
        for (int c = 0; c < Lay::kChunks; ++c)
          tma_load_3d(sV + vs * Lay::kTileBytes + c * Lay::kChunkBytes, &tm_v, v_full + vs, c * 64, kvh, row_k);
        ++v_uses[vs];
      }
      if (!ok) give_up();
      // Every copy this thread issued has landed before the CTA may exit.
      int never = 0;
      mbar_wait(q_full, 0, &never);
      for (int i = 0; i < NK; ++i)
        if (k_uses[i]) mbar_wait(k_full + i, (k_uses[i] - 1) & 1, &never);
      for (int i = 0; i < NV; ++i)
        if (v_uses[i]) mbar_wait(v_full + i, (v_uses[i] - 1) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kTile, kTile, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kTile, D, false, true);
      const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
      const int nkv_t[2] = {nkv0, nkv1};
      auto issue_s = [&](int t, int j) {  // S_t = Q_t K_j^T into S region t
        const uint32_t kbase = sKa + (j % NK) * Lay::kTileBytes, qbase = sQa + t * Lay::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * Lay::kChunkBytes + (kk % 4) * 32;
          umma_ss(tmem + Lay::kColS + t * kTile, sdesc_sw128(qbase + off, 16, 1024),
                  sdesc_sw128(kbase + off, 16, 1024), idesc_s, kk > 0);
        }
        umma_commit(s_full + t);
      };
      bool ok = mbar_wait(q_full, 0, abort_flag) && mbar_wait(k_full, 0, abort_flag);
      tc_fence_after();
      if (ok) {
        for (int t = 0; t < 2; ++t)
          if (nkv_t[t] > 0) issue_s(t, 0);
        umma_commit(k_empty);
      }
      for (int j = 0; j < nkv && ok; ++j) {
        const int vs = j % NV;
        bool v_ready = false, k_ready = false;
        for (int t = 0; t < 2 && ok; ++t) {
          if (j >= nkv_t[t]) continue;
          if (!(ok = mbar_wait(p_full + t, j & 1, abort_flag))) break;
          if (!v_ready && !(ok = v_ready = mbar_wait(v_full + vs, (j / NV) & 1, abort_flag))) break;
          tc_fence_after();
          const uint32_t a_tm = tmem + Lay::kColS + t * kTile;  // P_t, bf16 pairs
          const uint32_t vbase = sVa + vs * Lay::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_ts(tmem + Lay::kColO + t * D, a_tm + kk * 8, sdesc_sw128(vbase + kk * 2048, Lay::kChunkBytes, 1024),
                    idesc_o, (j > 0 || kk > 0));
          if (j + 1 < nkv_t[t]) {
            // S_t of the next key tile overwrites P_t after the product above has read it
            if (!k_ready && !(ok = k_ready = mbar_wait(k_full + (j + 1) % NK, ((j + 1) / NK) & 1, abort_flag))) break;
            tc_fence_after();
            issue_s(t, j + 1);
          } else {
            umma_commit(o_final + t);
          }
        }
        if (!ok) break;
        umma_commit(v_empty + vs);
        if (k_ready) umma_commit(k_empty + (j + 1) % NK);
      }
      if (!ok) give_up();
      // Drain: every MMA issued above completes before TMEM is released.
      umma_commit(drain);
      int never = 0;
      mbar_wait(drain, 0, &never);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 2) / 4;  // query tile of this warpgroup
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int qt = 2 * pair + t;
    const int qpos = qt * kTile + r;
    const int my_nkv = t == 0 ? nkv0 : nkv1;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32);
    const uint32_t tS = tmem + Lay::kColS + t * kTile, tO = tmem + Lay::kColO + t * D;
    const float c = p.scale_log2;
    const float2 c2 = make_float2(c, c);
    float m = -INFINITY, l = 0.f;  // reference max (log2 units) and row sum against it
    bool ok = true;
    for (int j = 0; j < my_nkv; ++j) {
      if (!(ok = mbar_wait(s_full + t, j & 1, abort_flag))) break;
      tc_fence_after();
      uint32_t sr[kTile];
      tmem_ld_x128(tmem_addr(tS, lane_base, 0), sr);
      float* x = reinterpret_cast<float*>(sr);
      const int k0 = j * kTile;
      const bool need_mask = (causal && j == qt) || (k0 + kTile > L);
      if (need_mask) {
        const int lim = causal ? min(qpos + 1, L) : L;  // visible keys: [0, lim)
#pragma unroll
        for (int i = 0; i < kTile; ++i)
          if (k0 + i >= lim) x[i] = -INFINITY;
      }
      float mx0 = fmaxf(x[0], x[1]), mx1 = fmaxf(x[2], x[3]);
#pragma unroll
      for (int i = 4; i < kTile; i += 4) {
        mx0 = max3(mx0, x[i], x[i + 1]);
        mx1 = max3(mx1, x[i + 2], x[i + 3]);
      }
      const float mt = fmaxf(mx0, mx1) * c;
      // move the reference only when the row max grows past the slack
      const bool bump = mt > m + kRescaleSlack;
      const float m_new = bump ? mt : m;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = bump ? ex2_approx(m - m_use) : 1.f;
      const float2 nm = make_float2(-m_use, -m_use);
      float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float2 e = fma2(make_float2(x[cc * 32 + 2 * u], x[cc * 32 + 2 * u + 1]), c2, nm);
          const float2 pv = make_float2(ex2_approx(e.x), ex2_approx(e.y));
          sum2 = add2(sum2, pv);
          pk[u] = pack_bf16x2(pv.x, pv.y);
        }
        tmem_st_x16(tmem_addr(tS, lane_base, cc * 16), pk);
      }
      l = l * alpha + (sum2.x + sum2.y);
      m = m_new;
      // O was last written by P V of the previous key tile, which completed
      // before S of this tile (same issuing thread, committed after it).
      if (j > 0 && __any_sync(0xffffffffu, bump)) {
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t ov[32];
          const uint32_t ta = tmem_addr(tO, lane_base, cc * 32);
          tmem_ld_x32(ta, ov);
#pragma unroll
          for (int u = 0; u < 32; ++u) ov[u] = __float_as_uint(__uint_as_float(ov[u]) * alpha);
          tmem_st_x32(ta, ov);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_full + t);
    }
    if (ok && my_nkv > 0) ok = mbar_wait(o_final + t, 0, abort_flag);
    if (!ok) {
      give_up();
    } else if (my_nkv > 0) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool row_ok = qpos < L;
      const long long tok = seq0 + qpos;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) + (tok * p.Hq + h) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t ov[32];
        tmem_ld_x32(tmem_addr(tO, lane_base, cc * 32), ov);
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          pk[u] = pack_bf16x2(__uint_as_float(ov[2 * u]) * inv_l, __uint_as_float(ov[2 * u + 1]) * inv_l);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u) dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      if (row_ok) p.lse[static_cast<long long>(h) * p.T + tok] = l > 0.f ? (m + lg2_approx(l)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

// Host-side launch for one head dimension; returns a cudaError_t value.
template <int D>
int launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                 cudaStream_t stream) {
  using Lay = FwdLayout<D>;
  cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
  if (e != cudaSuccess) return e;
  FwdParams q = p;
  q.n_qtiles = (p.n_qtiles + 1) / 2;  // the grid walks pairs of query tiles
  dim3 grid(q.Hq, q.n_qtiles, q.B);
  fa_fwd_kernel<D><<<grid, 320, Lay::kBytes, stream>>>(tq, tk, tv, q);
  return cudaGetLastError();
}

int launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
               cudaStream_t stream) {
  return d == 64 ? launch_fwd_d<64>(tq, tk, tv, p, stream) : launch_fwd_d<128>(tq, tk, tv, p, stream);
}

}  // namespace fa
