// Forward kernel: tiled exact attention with the online-softmax recurrence.
//
// What it computes ("FlashAttention：从 Safe Softmax 到分块计算", sections 3.2
// and 7; "企业官网建设流程全解析", section 2.1): for one 128-row query tile Q_i
// and each visible 128-row key tile j,
//     S     = Q_i K_j^T                      (tcgen05, f32 in TMEM)
//     m_new = max(m_old, rowmax(S) * c)      (c = scale * log2 e)
//     P     = exp2(S * c - m_new)            (bf16, written back to TMEM)
//     l     = exp2(m_old - m_new) * l + rowsum(P)
//     O     = exp2(m_old - m_new) * O + P V_j   (tcgen05, f32 in TMEM)
// and at the end O / l (bf16) and LSE = (m + log2 l) * ln 2.  Working in base
// 2 with log2 e folded into c is the same function as the pages' base-e form.
//
// One CTA owns one (query tile, query head, sequence).  Warp roles:
//   warp 0      TMA producer: Q once, then K_j and V_j through two rings.
//   warp 1      TMEM allocator and MMA issuer (one thread).
//   warps 2..5  softmax, O rescale and epilogue: thread t of this warpgroup
//               owns query row 32 * (warp % 4) + lane, i.e. that TMEM lane.
// The issue order S_0, S_1, PV_0, S_2, PV_1, ... lets the tensor core compute
// the next score tile while the softmax warps work on the current one.
//
// TMEM columns (512 allocated): S double buffer [0, 256), O [256, 256 + d),
// P double buffer (bf16 pairs) [384, 512).
#include <cuda_bf16.h>

#include "fa_common.cuh"

namespace fa {

template <int D>
struct FwdLayout {
  static constexpr int kChunkBytes = kTile * 128;          // 128 rows x 64 bf16 (one SW128 box)
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kChunks * kChunkBytes;  // one 128 x D bf16 tile
  static constexpr int kStagesK = D == 128 ? 3 : 4;
  static constexpr int kStagesV = D == 128 ? 2 : 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kStagesK * kTileBytes;
  static constexpr int kOffBar = kOffV + kStagesV * kTileBytes;
  // barriers: q_full, k_full[], k_empty[], v_full[], v_empty[], s_full[2], p_full[2], o_done, drain
  static constexpr int kNumBars = 1 + 2 * kStagesK + 2 * kStagesV + 2 + 2 + 1 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
};

constexpr float kLn2 = 0.6931471805599453f;

template <int D>
__global__ void __launch_bounds__(192, 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using Lay = FwdLayout<D>;
  constexpr int NK = Lay::kStagesK, NV = Lay::kStagesV;

  const int h = blockIdx.x;
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.y);  // longest rows first
  const int s = blockIdx.z;
  long long seq0;
  int L;
  if (!sequence_bounds(p.cu, s, p.N, p.T, seq0, L, p.status)) return;
  const int q0 = qt * kTile;
  if (q0 >= L) return;  // uniform across the CTA
  const bool causal = p.causal != 0;
  const int nkv = kv_tiles_for(qt, L, causal);
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
  uint64_t* o_done = p_full + 2;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kOffMisc + 4);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NK; ++i) { mbar_init(k_full + i, 1); mbar_init(k_empty + i, 1); }
    for (int i = 0; i < NV; ++i) { mbar_init(v_full + i, 1); mbar_init(v_empty + i, 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(s_full + i, 1); mbar_init(p_full + i, 128); }
    mbar_init(o_done, 1);
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
      const int row_q = static_cast<int>(seq0 + q0);
      mbar_arrive_expect_tx(q_full, Lay::kTileBytes);
      for (int c = 0; c < Lay::kChunks; ++c)
        tma_load_3d(sQ + c * Lay::kChunkBytes, &tm_q, q_full, c * 64, h, row_q);
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
      bool ok = mbar_wait(q_full, 0, abort_flag);
      tc_fence_after();
      auto issue_s = [&](int j) -> bool {
        const int ks = j % NK;
        if (!mbar_wait(k_full + ks, (j / NK) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t d_tm = tmem + Lay::kColS + (j & 1) * kTile;
        const uint32_t kbase = sKa + ks * Lay::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * Lay::kChunkBytes + (kk % 4) * 32;
          umma_ss(d_tm, sdesc_sw128(sQa + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024), idesc_s, kk > 0);
        }
        umma_commit(k_empty + ks);
        umma_commit(s_full + (j & 1));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < nkv && ok; ++j) {
        if (j + 1 < nkv && !(ok = issue_s(j + 1))) break;
        if (!(ok = mbar_wait(p_full + (j & 1), (j >> 1) & 1, abort_flag))) break;
        const int vs = j % NV;
        if (!(ok = mbar_wait(v_full + vs, (j / NV) & 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t a_tm = tmem + Lay::kColP + (j & 1) * 64;
        const uint32_t vbase = sVa + vs * Lay::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ts(tmem + Lay::kColO, a_tm + kk * 8, sdesc_sw128(vbase + kk * 2048, Lay::kChunkBytes, 1024),
                  idesc_o, (j > 0 || kk > 0));
        umma_commit(v_empty + vs);
        umma_commit(o_done);
      }
      if (!ok) give_up();
      // Drain: every MMA issued above completes before TMEM is released.
      umma_commit(drain);
      int never = 0;
      mbar_wait(drain, 0, &never);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int qpos = q0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32);
    const float c = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      if (!(ok = mbar_wait(s_full + (j & 1), (j >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      uint32_t sr[kTile];
      tmem_ld_x128(tmem_addr(tmem, lane_base, Lay::kColS + (j & 1) * kTile), sr);
      float* x = reinterpret_cast<float*>(sr);
      const int k0 = j * kTile;
      const bool need_mask = (causal && j == qt) || (k0 + kTile > L);
      if (need_mask) {
        const int lim = causal ? min(qpos + 1, L) : L;  // visible keys: [0, lim)
#pragma unroll
        for (int i = 0; i < kTile; ++i)
          if (k0 + i >= lim) x[i] = -INFINITY;
      }
      float mx = x[0];
#pragma unroll
      for (int i = 1; i < kTile; ++i) mx = fmaxf(mx, x[i]);
      const float m_new = fmaxf(m, mx * c);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(m - m_use);
      float sum = 0.f;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float p0 = ex2_approx(fmaf(x[cc * 32 + 2 * t], c, -m_use));
          const float p1 = ex2_approx(fmaf(x[cc * 32 + 2 * t + 1], c, -m_use));
          sum += p0 + p1;
          pk[t] = pack_bf16x2(p0, p1);
        }
        tmem_st_x16(tmem_addr(tmem, lane_base, Lay::kColP + (j & 1) * 64 + cc * 16), pk);
      }
      l = l * alpha + sum;
      m = m_new;
      tmem_st_wait();
      if (j > 0) {
        // O may only be rescaled once the previous P V product has landed.
        if (!(ok = mbar_wait(o_done, (j - 1) & 1, abort_flag))) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t ov[32];
            const uint32_t ta = tmem_addr(tmem, lane_base, Lay::kColO + cc * 32);
            tmem_ld_x32(ta, ov);
#pragma unroll
            for (int t = 0; t < 32; ++t) ov[t] = __float_as_uint(__uint_as_float(ov[t]) * alpha);
            tmem_st_x32(ta, ov);
          }
          tmem_st_wait();
        }
      }
      tc_fence_before();
      mbar_arrive(p_full + (j & 1));
    }
    if (ok) ok = mbar_wait(o_done, (nkv - 1) & 1, abort_flag);
    if (!ok) {
      give_up();
    } else {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool row_ok = qpos < L;
      const long long tok = seq0 + qpos;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) + (tok * p.Hq + h) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t ov[32];
        tmem_ld_x32(tmem_addr(tmem, lane_base, Lay::kColO + cc * 32), ov);
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
          pk[t] = pack_bf16x2(__uint_as_float(ov[2 * t]) * inv_l, __uint_as_float(ov[2 * t + 1]) * inv_l);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int t = 0; t < 4; ++t) dst[t] = make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
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
  dim3 grid(p.Hq, p.n_qtiles, p.B);
  fa_fwd_kernel<D><<<grid, 192, Lay::kBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

int launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
               cudaStream_t stream) {
  return d == 64 ? launch_fwd_d<64>(tq, tk, tv, p, stream) : launch_fwd_d<128>(tq, tk, tv, p, stream);
}

}  // namespace fa
