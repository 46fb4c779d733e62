// Backward kernels: recompute-based attention gradient.
//
// What it computes ("企业官网建设流程全解析", section 2.3; "Attention 算子优化…",
// section 四 on recomputation; "FlashAttention：从 Safe Softmax 到分块计算",
// section 8 on the saved LSE): with D_q = rowsum(dO_q * O_q) (equal to
// rowsum(dP * P) for that query row), for every visible (key tile j, query
// tile i) pair of a (sequence, K/V head):
//     S^T  = K_j Q_i^T                 P^T = exp2(S^T * c - LSE * log2 e)
//     dP^T = V_j dO_i^T                dS^T = P^T * (dP^T - D)
//     dV_j += P^T dO_i                 dK_j += dS^T Q_i
//     dQ_i += dS K_j   (f32 bulk reduce-adds into a global accumulator)
// and finally dK *= scale, dQ = scale * dQ_acc.  P is recomputed already
// normalised from the LSE, so no running max is needed.
//
// Three launches: fa_bwd_rowdot_kernel (D and zeroing of the dQ accumulator),
// the gradient kernel (the five tcgen05 products per tile pair: fa_bwd_kernel
// below for d = 64, fa_bwd128_kernel in fa_bwd128.cu for d = 128),
// fa_bwd_dq_kernel (dQ accumulator -> bf16).
//
// fa_bwd_kernel: persistent, one CTA per SM walking work units (key tile j,
// K/V head, sequence), heaviest first; per unit it walks the query heads of
// the group and their query tiles ("steps"), so dK and dV of the group
// accumulate in TMEM with no atomics.  Steps are counted across units, so
// the rings and the step-parity barriers run on from one unit to the next
// and the next unit's first products start while the last one drains.
// Warp roles:
//   warp 0       producer: per step Q_i, dO_i (TMA) and the LSE / D values of
//                the tile (plain loads) into a 3-stage ring.
//   warp 1       TMEM allocator; MMA issuer A (one thread): dV and dQ.
//   warp 14      MMA issuer B (one thread): dP^T and dK.
//   warp 15      MMA issuer C (one thread): K_j, V_j of each unit (TMA, once
//                every product of the previous unit that reads them is done)
//                and S^T.
//   warps 2..9   two score warpgroups: thread = key row (TMEM lane); the
//                first takes query columns 0..63, the second 64..127; P^T to
//                TMEM (bf16), dS^T to TMEM and (for dQ) shared memory; the
//                unit's dV / dK epilogue (a whole key tile staged in shared
//                memory and written by two TMA bulk stores).
//   warps 10..13 dQ warpgroup: dQ tile TMEM -> swizzled shared memory (the
//                step's dS^T buffer, free once the dQ product has read it) ->
//                two TMA bulk reduce-adds (f32) into the global accumulator.
// MMA issue order: once the score warpgroups finish step n, dV += P^T_n dO_n
// (A) and dK += dS^T_n Q_n (B) run side by side, both taking queries 64..127
// first, then dQ_n = dS_n K (A, once dK_n has read those queries, whose
// columns dQ_n overwrites); S^T_{n+2} (C) follows as soon as the dQ of step n
// has been read out and dV_n, dK_n are done, and dP^T_{n+2} (B) as soon as
// the score warpgroups of step n+1 have read their dP^T.  The scores of the
// next step are thus computed while the score warpgroups still work on the
// current one.
// TMEM (d = 64, 512 columns): two step regions of 128 columns (S^T f32; each
// 16-column chunk of S^T, once read, takes the bf16 P^T of its 16 queries in
// its first 8 columns and their bf16 dS^T in the last 8, so dV and dK both
// take their A operand from TMEM; dQ f32 over columns 64..127, written by an
// MMA issued after the dV and dK products that read them),
// dP^T [256, 384), dV [384, 448), dK [448, 512).  dS^T also goes to shared
// memory (three buffers) as the MN-major A operand of dQ (rows = queries).
#include <cuda_bf16.h>

#include "fa_common.cuh"

namespace fa {

template <int D>
struct BwdLayout {
  static constexpr int kChunkBytes = kTile * 128;
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kStages = 3;
  static constexpr int kStageBytes = 2 * kTileBytes;  // Q_i, dO_i
  static constexpr int kDSBytes = 2 * kChunkBytes;    // 128 keys x 128 queries bf16
  static constexpr int kDSBufs = 3;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  // dS^T of step n in buffer n % 3, which then stages the f32 dQ tile of the
  // step (32 KB as well) for its bulk reduce-adds
  static constexpr int kOffDS = kOffV + kTileBytes;
  static constexpr int kOffRing = kOffDS + kDSBufs * kDSBytes;
  // -LSE log2 e and -D of the step's 128 queries, f32, in slot n % 2: the
  // score warpgroups read them during step n only.  Interleaved by query
  // pair, {-LSE q, -LSE q+1, -D q, -D q+1}, so one 16-byte load serves a pair.
  static constexpr int kOffStats = kOffRing + kStages * kStageBytes;
  static constexpr int kStatBytes = 2 * kTile * 4;
  static constexpr int kOffBar = kOffStats + 2 * kStatBytes;
  // kv_full, qdo_full[], qdo_empty[], sdp_full[2], ps_ready[2], dp_free, dq_full[2], dq_free[2],
  // dq_staged, ds_free[3], epi, drain, dk_hi[2], kv_free, acc_free, epi_staged, epi_read
  static constexpr int kNumBars = 1 + 2 * kStages + 22;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // no room to round the dynamic shared memory base up to the 1 KB alignment
  // of the 128-byte swizzle: the kernel requires an aligned base (it is, with
  // no static shared memory) and otherwise sets a status bit and does nothing
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColStep = 0;      // + 128 * (n & 1)
  static constexpr uint32_t kColDQ = 64;       // within a step region
  static constexpr uint32_t kColDP = 256, kColDV = 384, kColDK = 384 + D;
  static_assert(D == 64, "TMEM plan is for d = 64");
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

constexpr int kWarpIssuerB = 14, kWarpIssuerC = 15;
constexpr int kBwdThreads = 32 * (kWarpIssuerC + 1);

// DQ = false compiles the dQ product and the dQ warpgroup out (the
// deterministic backward computes dQ in a separate kernel).
template <int D, bool DQ>
__global__ void __launch_bounds__(kBwdThreads, 1)
fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
              const __grid_constant__ CUtensorMap tm_dv, const BwdParams p) {
  using Lay = BwdLayout<D>;
  constexpr int NS = Lay::kStages;
  const bool causal = p.causal != 0;

  // Persistent: work units (128-key tile, K/V head, sequence), key tile
  // outermost so the causal work goes heaviest first; CTA i takes the units
  // i, 2G-1-i, 2G+i, ... (G = grid size).  Every role walks the same units
  // and counts steps globally, so the step-indexed barriers and buffers run
  // on across units; units past the end of their sequence are skipped by
  // every role alike.
  const int n_units = p.n_kvtiles * p.B * p.Hkv;
  const int G = static_cast<int>(gridDim.x);
  auto unit_of = [&](int k) {
    return k * G + ((k & 1) ? G - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x));
  };
  struct Unit {
    long long seq0;
    int L, g, k0, i0, per_head, nsteps, sq;
  };
  auto unit_at = [&](int u, Unit& w) -> bool {
    w.g = u % p.Hkv;
    const int rest = u / p.Hkv;
    const int kt = rest / p.B;
    w.sq = rest % p.B;
    if (!sequence_bounds(p.cu, w.sq, p.N, p.T, w.seq0, w.L, p.status)) return false;
    w.k0 = kt * kTile;
    if (w.k0 >= w.L) return false;
    w.i0 = first_q_tile_for(kt, causal);
    w.per_head = (w.L + kTile - 1) / kTile - w.i0;
    w.nsteps = p.group * w.per_head;
    return true;
  };
  // local step nl of unit w -> (query head, query tile)
  auto step_head = [&](const Unit& w, int nl) { return w.g * p.group + nl / w.per_head; };
  auto step_qtile = [&](const Unit& w, int nl) { return w.i0 + nl % w.per_head; };

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusSmemAlign);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sK = smem + Lay::kOffK;
  uint8_t* sV = smem + Lay::kOffV;
  uint8_t* sDS = smem + Lay::kOffDS;
  uint8_t* ring = smem + Lay::kOffRing;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBar);
  uint64_t* kv_full = bars;
  uint64_t* qdo_full = kv_full + 1;
  uint64_t* qdo_empty = qdo_full + NS;
  uint64_t* sdp_full = qdo_empty + NS;  // sdp_full[n & 1]
  uint64_t* ps_ready = sdp_full + 2;
  uint64_t* dp_free = ps_ready + 2;  // ps_ready[n & 1]: one per step parity
  uint64_t* dq_full = dp_free + 1;  // dq_full[n & 1]
  uint64_t* dq_free = dq_full + 2;  // dq_free[n & 1]
  uint64_t* dq_staged = dq_free + 2;
  uint64_t* ds_free = dq_staged + 1;  // ds_free[n % 3]
  uint64_t* epi = ds_free + Lay::kDSBufs;
  uint64_t* drain = epi + 1;
  uint64_t* dk_hi = drain + 1;  // dk_hi[n & 1]: dK_n has read queries 64..127
  uint64_t* kv_free = dk_hi + 2;   // the unit's K / V tiles have been read by every product
  uint64_t* acc_free = kv_free + 1;  // the unit's dV / dK have been read out of TMEM
  uint64_t* epi_staged = acc_free + 1;  // a whole tile's dV / dK staged in shared memory
  uint64_t* epi_read = epi_staged + 1;  // and read by its bulk stores
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kOffMisc + 4);

  auto stage_q = [&](int st) { return ring + st * Lay::kStageBytes; };
  auto stage_do = [&](int st) { return ring + st * Lay::kStageBytes + Lay::kTileBytes; };
  auto step_stats = [&](int n) { return reinterpret_cast<float*>(smem + Lay::kOffStats + (n & 1) * Lay::kStatBytes); };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    // the MMA issuers: S^T and dP^T commit on sdp_full (one barrier per step
    // parity: S^T_{m+1} has no reason to wait for dP^T_m), dV and dK on
    // qdo_empty and epi, all three on drain
    for (int i = 0; i < NS; ++i) { mbar_init(qdo_full + i, 32); mbar_init(qdo_empty + i, 2); }
    mbar_init(sdp_full, 2);
    mbar_init(sdp_full + 1, 2);
    mbar_init(ps_ready, 256);
    mbar_init(ps_ready + 1, 256);
    mbar_init(dp_free, 256);
    mbar_init(dq_full, 1);
    mbar_init(dq_full + 1, 1);
    mbar_init(dq_free, 128);
    mbar_init(dq_free + 1, 128);
    mbar_init(dq_staged, 128);
    for (int i = 0; i < Lay::kDSBufs; ++i) mbar_init(ds_free + i, 1);
    mbar_init(epi, 2);
    mbar_init(drain, 3);
    mbar_init(dk_hi, 1);
    mbar_init(dk_hi + 1, 1);
    mbar_init(kv_free, 3);   // the three MMA threads, once per unit
    mbar_init(acc_free, 256);
    mbar_init(epi_staged, 256);
    mbar_init(epi_read, 1);
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
  auto region = [&](int n) { return tmem + Lay::kColStep + static_cast<uint32_t>(n & 1) * 128; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Q_i, dO_i (TMA) and the LSE / D values of every step; K_j, V_j are
    // loaded by thread C, the first to need them.
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_dq);
      tma_prefetch_desc(&tm_dk);
      tma_prefetch_desc(&tm_dv);
    }
    int uses[NS] = {};
    bool ok = true;
    int n = 0;  // steps so far
    for (int k = 0, un = unit_of(0); un < n_units && ok; un = unit_of(++k)) {
      Unit w;
      if (!unit_at(un, w)) continue;
      for (int nl = 0; nl < w.nsteps; ++nl, ++n) {
        const int st = n % NS;
        if (n >= NS &&
            !(ok = __all_sync(0xffffffffu, mbar_wait(qdo_empty + st, ((n / NS) - 1) & 1, abort_flag))))
          break;
        const int h = step_head(w, nl), q0 = step_qtile(w, nl) * kTile;
        if (lane == 0) {
          mbar_expect_tx(qdo_full + st, 2 * Lay::kTileBytes);
          const int row = static_cast<int>(w.seq0 + q0);
          for (int c = 0; c < Lay::kChunks; ++c) {
            tma_load_3d(stage_q(st) + c * Lay::kChunkBytes, &tm_q, qdo_full + st, c * 64, h, row);
            tma_load_3d(stage_do(st) + c * Lay::kChunkBytes, &tm_do, qdo_full + st, c * 64, h, row);
          }
        }
        const long long lrow = static_cast<long long>(h) * p.T + w.seq0 + q0;
        float lv[kTile / 32], dv[kTile / 32];
#pragma unroll
        for (int t = 0; t < kTile / 32; ++t) {
          const int idx = lane + 32 * t;
          const bool valid = q0 + idx < w.L;
          lv[t] = valid ? __ldg(p.lse + lrow + idx) : INFINITY;
          dv[t] = valid ? __ldg(p.rowdot + lrow + idx) : 0.f;
        }
        // the stats slot of this step parity: the score warpgroups are done
        // with step n - 2 (on a failed wait the stage still completes, so the
        // drain below covers the loads already issued)
        if (n >= 2)
          ok = __all_sync(0xffffffffu, mbar_wait(ps_ready + (n & 1), ((n - 2) >> 1) & 1, abort_flag));
        if (ok) {
          float* stats = step_stats(n);
#pragma unroll
          for (int t = 0; t < kTile / 32; ++t) {
            // stored negated: -LSE * log2 e and -D (queries past the end: P = 0)
            const int qq = lane + 32 * t;
            stats[(qq >> 1) * 4 + (qq & 1)] = -lv[t] * kLog2e;
            stats[(qq >> 1) * 4 + 2 + (qq & 1)] = -dv[t];
          }
        }
        mbar_arrive(qdo_full + st);
        ++uses[st];
        if (!ok) break;
      }
    }
    if (!ok && lane == 0) give_up();
    if (lane == 0) {
      int never = 0;
      for (int i = 0; i < NS; ++i)
        if (uses[i]) mbar_wait(qdo_full + i, (uses[i] - 1) & 1, &never);
    }
  } else if (warp == 1 || warp == kWarpIssuerB || warp == kWarpIssuerC) {
    // ------------------------------------------------------------ MMA issuers
    // Three issuing threads, each with its own order of waits, so that no
    // product queues behind a wait that belongs to another (one thread also
    // starts an N = 64 product only about every 55 cycles, half the tensor
    // core's rate for that shape).  A (warp 1): dV, dQ.  B: dK, dP^T.  C: S^T.
    if (lane == 0) {
      const int role = warp == 1 ? 0 : (warp == kWarpIssuerB ? 1 : 2);
      constexpr uint32_t id_sdp = idesc_bf16_f32(kTile, kTile, false, false);  // K-major x K-major
      constexpr uint32_t id_dvk = idesc_bf16_f32(kTile, D, false, true);       // TMEM A x MN-major B
      constexpr uint32_t id_dq = idesc_bf16_f32(kTile, D, true, true);         // MN-major A x MN-major B
      const uint32_t sKa = smem_u32(sK), sVa = smem_u32(sV), sDSa = smem_u32(sDS);
      // S^T_m (C) or dP^T_m (B) = K or V times the Q or dO tile of step m
      auto issue_score = [&](int m) {
        const int st = m % NS;
        const bool s_t = role == 2;
        const uint32_t xa = s_t ? sKa : sVa;
        const uint32_t ya = smem_u32(s_t ? stage_q(st) : stage_do(st));
        const uint32_t dst = s_t ? region(m) : tmem + Lay::kColDP;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * Lay::kChunkBytes + (kk % 4) * 32;
          umma_ss(dst, sdesc_sw128(xa + off, 16, 1024), sdesc_sw128(ya + off, 16, 1024), id_sdp, kk > 0);
        }
        umma_commit(sdp_full + (m & 1));
      };
      // S^T_m needs the Q stage of step m and the step region of m-2: its dQ
      // read out and its dV and dK products done.  dP^T_m needs the
      // dO stage and the dP^T region, which the score warpgroups of step m-1
      // release (dp_free) once their dP^T loads are done.
      auto issue_next = [&](int m) -> bool {
        if (!mbar_wait(qdo_full + m % NS, (m / NS) & 1, abort_flag)) return false;
        if (role == 2 && m >= 2) {
          const int r = m - 2;
          if (DQ && !mbar_wait(dq_free + (r & 1), (r >> 1) & 1, abort_flag)) return false;
          // dV and dK of step m-2 are done with the region too (thread B's dK
          // has no order with respect to thread A's dQ, so dq_free alone does
          // not cover it)
          if (!mbar_wait(qdo_empty + r % NS, (r / NS) & 1, abort_flag)) return false;
        }
        if (role == 1 && m >= 1 && !mbar_wait(dp_free, (m - 1) & 1, abort_flag)) return false;
        tc_fence_after();
        issue_score(m);
        return true;
      };
      bool ok = true;
      int n0 = 0, uc = 0, kv_loads = 0;  // steps and units so far, K / V loads issued (C)
      for (int k = 0, un = unit_of(0); un < n_units && ok; un = unit_of(++k)) {
        Unit w;
        if (!unit_at(un, w)) continue;
        if (role == 2) {
          // K_j, V_j of this unit, once every product of the previous unit
          // that reads them is done
          if (uc >= 1 && !(ok = mbar_wait(kv_free, (uc - 1) & 1, abort_flag))) break;
          mbar_arrive_expect_tx(kv_full, 2 * Lay::kTileBytes);
          for (int c = 0; c < Lay::kChunks; ++c) {
            tma_load_3d(sK + c * Lay::kChunkBytes, &tm_k, kv_full, c * 64, w.g, static_cast<int>(w.seq0 + w.k0));
            tma_load_3d(sV + c * Lay::kChunkBytes, &tm_v, kv_full, c * 64, w.g, static_cast<int>(w.seq0 + w.k0));
          }
          ++kv_loads;
          // and the next unit's K_j, V_j into L2, so that their load at the
          // unit boundary does not wait for DRAM
          for (int k2 = k + 1, un2 = unit_of(k2); un2 < n_units; un2 = unit_of(++k2)) {
            Unit w2;
            if (!unit_at(un2, w2)) continue;
            for (int c = 0; c < Lay::kChunks; ++c) {
              tma_prefetch_l2_3d(&tm_k, c * 64, w2.g, static_cast<int>(w2.seq0 + w2.k0));
              tma_prefetch_l2_3d(&tm_v, c * 64, w2.g, static_cast<int>(w2.seq0 + w2.k0));
            }
            break;
          }
        }
        if ((role != 0 || DQ) && !(ok = mbar_wait(kv_full, uc & 1, abort_flag))) break;
        tc_fence_after();
        if (role == 2) {
          int issued = 0;
          for (int nl = 0; nl < w.nsteps && ok; ++nl) {
            ok = issue_next(n0 + nl);
            issued += ok ? 1 : 0;
          }
          // tile pairs whose S^T this thread issued for the unit
          if (p.tile_count != nullptr && issued > 0)
            atomicAdd(p.tile_count + w.sq, static_cast<unsigned long long>(issued));
        } else {
          if (ok && role == 1) ok = issue_next(n0);
          if (ok && role == 1 && w.nsteps > 1) ok = issue_next(n0 + 1);
          for (int nl = 0; nl < w.nsteps && ok; ++nl) {
            const int n = n0 + nl;
            const int st = n % NS;
            // Score warpgroups may finish step n + 1 before this thread looks at
            // step n, so each step parity has its own barrier: step n + 2 cannot
            // start before its S^T and dP^T are issued.
            if (!(ok = mbar_wait(ps_ready + (n & 1), (n >> 1) & 1, abort_flag))) break;
            // dV and dK of the previous unit have been read out before this
            // unit's first products overwrite them
            if (nl == 0 && uc >= 1 && !(ok = mbar_wait(acc_free, (uc - 1) & 1, abort_flag))) break;
            tc_fence_after();
            // dV += P^T dO (A) or dK += dS^T Q (B)  (A operand: P^T or dS^T in
            // TMEM, queries 16 kk .. 16 kk + 15 at the columns the score
            // warpgroups chose; B operand: dO or Q, rows = queries = K, MN-major)
            const uint32_t ya = smem_u32(role == 0 ? stage_do(st) : stage_q(st));
            const uint32_t acc = tmem + (role == 0 ? Lay::kColDV : Lay::kColDK);
            const uint32_t a0 = region(n) + (role == 0 ? 0 : 8);
            // queries 64..127 first: their columns are where dQ_n goes
#pragma unroll
            for (int j = 0; j < kTile / 16; ++j) {
              const int kk = (j + 4) % 8;
              umma_ts(acc, a0 + 16 * kk, sdesc_sw128(ya + kk * 2048, Lay::kChunkBytes, 1024), id_dvk,
                      (nl > 0 || j > 0));
              if (role == 1 && j == 3) umma_commit(dk_hi + (n & 1));  // dK has read queries 64..127
            }
            umma_commit(qdo_empty + st);
            if (role == 0 && DQ) {
              // dQ_n = dS K into columns 64..127 of the step region of n, once
              // dV_n (above, this thread) and the first half of dK_n (thread B)
              // have read the P^T / dS^T there; its dQ_{n-2} was read before
              // S^T_n was issued  (A: the dS^T tile read query-major, MN-major;
              // B: K, MN-major)
              if (!(ok = mbar_wait(dk_hi + (n & 1), (n >> 1) & 1, abort_flag))) break;
              tc_fence_after();
              const uint32_t dsb = sDSa + (n % Lay::kDSBufs) * Lay::kDSBytes;
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                umma_ss(region(n) + Lay::kColDQ, sdesc_sw128(dsb + kk * 2048, Lay::kChunkBytes, 1024),
                        sdesc_sw128(sKa + kk * 2048, Lay::kChunkBytes, 1024), id_dq, kk > 0);
              umma_commit(dq_full + (n & 1));
            }
            if (role == 1 && nl + 2 < w.nsteps && !(ok = issue_next(n + 2))) break;
          }
          if (ok) umma_commit(epi);  // this unit's dV / dK are complete
        }
        if (ok) umma_commit(kv_free);  // this thread's products of the unit are done with K, V
        n0 += w.nsteps;
        ++uc;
      }
      if (role == 2 && kv_loads > 0) {
        // no K / V copy may still be in flight when the CTA exits
        int never = 0;
        mbar_wait(kv_full, (kv_loads - 1) & 1, &never);
      }
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
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32);
    const float c = p.scale_log2;
    const float2 c2 = make_float2(c, c);
    bool ok = true;
    int n = 0, uc = 0, ue = 0;  // steps, units and whole-tile stores so far
    bool pending = false;       // the last whole-tile stores may still be reading their staging
    // Wait until the stores of the last whole tile have read their staging
    // (the thread that issued them waits for its bulk group, then lets the
    // others go on).
    auto staging_read = [&]() -> bool {
      if (!pending) return true;
      pending = false;
      if (warp == 2 && lane == 0) {
        bulk_wait_group_read0();
        mbar_arrive(epi_read);
      }
      return __all_sync(0xffffffffu, mbar_wait(epi_read, (ue - 1) & 1, abort_flag));
    };
    for (int k = 0, un = unit_of(0); un < n_units && ok; un = unit_of(++k)) {
    Unit w;
    if (!unit_at(un, w)) continue;
    const int k0 = w.k0, L = w.L;
    const long long seq0 = w.seq0;
    const int kpos = k0 + r;
    const bool key_ok = kpos < L;
    for (int nl = 0; nl < w.nsteps; ++nl, ++n) {
      const int st = n % NS;
      if (!(ok = mbar_wait(sdp_full + (n & 1), (n >> 1) & 1, abort_flag))) break;
      if (!(ok = mbar_wait(qdo_full + st, (n / NS) & 1, abort_flag))) break;
      tc_fence_after();
      const int q0 = step_qtile(w, nl) * kTile;
      const float4* nst4 = reinterpret_cast<const float4*>(step_stats(n)) + half * 32;
      // Keys past the sequence end and keys after the query (diagonal tile,
      // causal) get P = 0: query columns below zero_below are zeroed.
      // Queries past the end carry -LSE = -inf, so their P is 0 already.
      const int zero_below = !key_ok ? kTile : ((causal && q0 == k0) ? r : 0);
      uint8_t* ds_row = sDS + (n % Lay::kDSBufs) * Lay::kDSBytes + half * Lay::kChunkBytes + r * 128;
      const uint32_t reg = region(n);
      // S^T and dP^T of chunk cl + 1 load while chunk cl is computed
      uint32_t sv[2][16], dpv[2][16];
      tmem_ld_x16_pair(tmem_addr(reg, lane_base, half * 64), sv[0], tmem_addr(tmem, lane_base, Lay::kColDP + half * 64),
                       dpv[0]);
#pragma unroll
      for (int cl = 0; cl < 4; ++cl) {
        const int col0 = half * 64 + cl * 16;  // first query column of this chunk
        const int cb = cl & 1;
        if (cl < 3)
          tmem_ld_x16_pair_nowait(tmem_addr(reg, lane_base, col0 + 16), sv[cb ^ 1],
                                  tmem_addr(tmem, lane_base, Lay::kColDP + col0 + 16), dpv[cb ^ 1]);
        if (cl == 3) {
          // dP^T fully read: the next step's dP^T may overwrite it
          tc_fence_before();
          mbar_arrive(dp_free);
        }
        uint32_t pk[8], dsk[8];
        const bool mask_chunk = zero_below > col0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const float4 s4 = nst4[cl * 8 + t];
          const float2 nl2 = make_float2(s4.x, s4.y), nd = make_float2(s4.z, s4.w);
          const float2 x =
              fma2(make_float2(__uint_as_float(sv[cb][2 * t]), __uint_as_float(sv[cb][2 * t + 1])), c2, nl2);
          float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          if (mask_chunk) {
            if (col0 + 2 * t < zero_below) pv.x = 0.f;
            if (col0 + 2 * t + 1 < zero_below) pv.y = 0.f;
          }
          const float2 dd =
              mul2(pv, add2(make_float2(__uint_as_float(dpv[cb][2 * t]), __uint_as_float(dpv[cb][2 * t + 1])), nd));
          pk[t] = pack_bf16x2(pv.x, pv.y);
          dsk[t] = pack_bf16x2(dd.x, dd.y);
        }
        // P^T and dS^T (bf16) overwrite the 16 S^T columns this chunk has
        // just read: P^T in the first 8, dS^T in the last 8.
        tmem_st_x8(tmem_addr(reg, lane_base, col0), pk);
        tmem_st_x8(tmem_addr(reg, lane_base, col0 + 8), dsk);
        // The dS^T buffer of this step (n % 3) is free once the bulk reduces
        // of dQ_{n-3}, staged there, have read it (one vote per warp, so the
        // warp stays together for the TMEM loads that follow).
        if (DQ && cl == 0 && n >= Lay::kDSBufs)
          ok = __all_sync(0xffffffffu, mbar_wait(ds_free + n % Lay::kDSBufs, (n / Lay::kDSBufs - 1) & 1, abort_flag));
        if (DQ && cl == 0 && ok) ok = staging_read();
        // dS^T row r into the 128B-swizzled tile (query-contiguous rows; the
        // 16-byte unit u holds queries 8 u .. 8 u + 7 of this 64-query half).
#pragma unroll
        for (int u2 = 0; u2 < 2 && DQ && ok; ++u2) {
          const int uu = cl * 2 + u2;
          *reinterpret_cast<uint4*>(ds_row + ((uu ^ (r & 7)) << 4)) =
              make_uint4(dsk[4 * u2], dsk[4 * u2 + 1], dsk[4 * u2 + 2], dsk[4 * u2 + 3]);
        }
        if (cl < 3) tmem_ld_wait_x16_pair(sv[cb ^ 1], dpv[cb ^ 1]);
      }
      if (!ok) break;
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(ps_ready + (n & 1));
    }
    if (ok) ok = mbar_wait(epi, uc & 1, abort_flag);
    if (!ok) break;
    // first warpgroup stores dV, second dK (scaled)
    const uint32_t col = half == 0 ? Lay::kColDV : Lay::kColDK;
    const float mul = half == 0 ? 1.f : p.scale;
    if (k0 + kTile <= L) {
      // A whole tile: staged as a 128B-swizzled 128 x 64 bf16 box per
      // warpgroup in the dS^T buffer of the next step (free once the reduces
      // it staged have read it), then written by two bulk tensor stores, so
      // that the rows go out as whole 128-byte lines.
      if (DQ && n >= Lay::kDSBufs)
        ok = __all_sync(0xffffffffu, mbar_wait(ds_free + n % Lay::kDSBufs, (n / Lay::kDSBufs - 1) & 1, abort_flag));
      if (ok) ok = staging_read();
      if (!ok) break;
      uint8_t* stage = sDS + (n % Lay::kDSBufs) * Lay::kDSBytes;
      uint8_t* row = stage + half * Lay::kChunkBytes + r * 128;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        tmem_ld_x32(tmem_addr(tmem, lane_base, col + cc * 32), v);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(v[8 * t + 2 * e]) * mul, __uint_as_float(v[8 * t + 2 * e + 1]) * mul);
          const int u = cc * 4 + t;
          *reinterpret_cast<uint4*>(row + ((u ^ (r & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      // dV and dK are read out of TMEM: the next unit may restart them
      tc_fence_before();
      mbar_arrive(acc_free);
      fence_proxy_async_smem();
      mbar_arrive(epi_staged);
      if (warp == 2 && lane == 0 && (ok = mbar_wait(epi_staged, ue & 1, abort_flag))) {
        const int row0 = static_cast<int>(seq0 + k0);
        tma_store_3d(&tm_dv, stage, 0, w.g, row0);
        tma_store_3d(&tm_dk, stage + Lay::kChunkBytes, 0, w.g, row0);
        bulk_commit_group();
      }
      // the stores run on while the next unit starts; the buffer takes
      // dS^T (or the next tile's staging) only once they have read it
      ++ue;
      pending = true;
    } else {
      // the sequence's last, ragged tile: row by row, rows past the end skipped
      tc_fence_after();
      const bool row_ok = kpos < L;
      const long long tok = seq0 + kpos;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(half == 0 ? p.dv : p.dk) + (tok * p.Hkv + w.g) * D;
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
      // dV and dK are in registers and stored: the next unit may restart them
      tc_fence_before();
      mbar_arrive(acc_free);
    }
    ++uc;
    }
    // no bulk store may still be writing when the CTA exits
    if (warp == 2 && lane == 0) bulk_wait_group0();
    if (!ok) give_up();
  } else if (DQ) {
    // ------------------------------------------------------------ dQ warpgroup
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // query row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32);
    const bool issuer = (warp == 10 && lane == 0);
    bool ok = true;
    int n = 0;  // steps so far
    for (int k = 0, un = unit_of(0); un < n_units && ok; un = unit_of(++k)) {
    Unit w;
    if (!unit_at(un, w)) continue;
    for (int nl = 0; nl < w.nsteps && ok; ++nl, ++n) {
      if (!(ok = mbar_wait(dq_full + (n & 1), (n >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      uint32_t v[D];
      tmem_ld_x64(tmem_addr(region(n), lane_base, Lay::kColDQ), v);
      tc_fence_before();
      mbar_arrive(dq_free + (n & 1));
      const int h = step_head(w, nl), q0 = step_qtile(w, nl) * kTile;
      // Stage dQ_n in the dS^T buffer of step n, which the dQ product has
      // finished reading: two f32 boxes of 32 columns x 128 rows, 128-byte
      // swizzle, added to the accumulator by two bulk reduces in flight at once.
      uint8_t* buf = sDS + (n % Lay::kDSBufs) * Lay::kDSBytes;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint8_t* row = buf + cc * kTile * 128 + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(row + ((u ^ (r & 7)) << 4)) =
              make_uint4(v[32 * cc + 4 * u], v[32 * cc + 4 * u + 1], v[32 * cc + 4 * u + 2], v[32 * cc + 4 * u + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(dq_staged);
      if (issuer) {
        if (!(ok = mbar_wait(dq_staged, n & 1, abort_flag))) break;
        // Rows past the sequence end hold exact zeros (P = 0 there), so the
        // whole tile can be added; rows past T are clipped by the TMA unit.
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc)
          tma_reduce_add_3d(&tm_dq, buf + cc * kTile * 128, cc * 32, h, static_cast<int>(w.seq0 + q0));
        bulk_commit_group();
        // The buffer of step n - 1 goes back to the score warpgroups (dS^T of
        // step n + 2) once its reduces have read it; those of step n stay in
        // flight meanwhile.
        bulk_wait_group_read1();
        if (n >= 1) mbar_arrive(ds_free + (n - 1) % Lay::kDSBufs);
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

// D[h, t] = sum_d dO[t, h, d] * O[t, h, d] (f32) and dQ_acc = 0.  Eight
// threads per (token, head) row, 16 bytes each per pass.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_rowdot_kernel(const BwdParams p) {
  constexpr int kPerRow = 8;
  const long long rows = p.T * p.Hq;
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / kPerRow;
  const int sub = threadIdx.x % kPerRow;
  float acc = 0.f;
  if (row < rows) {
    const uint4* o4 = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.o) + row * D);
    const uint4* d4 = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.dout) + row * D);
    float4* z = reinterpret_cast<float4*>(p.dq_acc + row * D);
#pragma unroll
    for (int i = sub; i < D / 8; i += kPerRow) {
      const uint4 a = __ldg(o4 + i), b = __ldg(d4 + i);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa2 = __bfloat1622float2(a2[e]), fb2 = __bfloat1622float2(b2[e]);
        acc = fmaf(fa2.x, fb2.x, acc);
        acc = fmaf(fa2.y, fb2.y, acc);
      }
      z[2 * i] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[2 * i + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int off = kPerRow / 2; off > 0; off /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && sub == 0) {
    const long long t = row / p.Hq;
    const int h = static_cast<int>(row % p.Hq);
    p.rowdot[static_cast<long long>(h) * p.T + t] = acc;
  }
}

// dQ = bf16(scale * dQ_acc), eight elements per thread.
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const BwdParams p, long long n8) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4* src = reinterpret_cast<const float4*>(p.dq_acc) + 2 * i;
  const float4 a = src[0], b = src[1];
  const float s = p.scale;
  uint4 out = make_uint4(pack_bf16x2(a.x * s, a.y * s), pack_bf16x2(a.z * s, a.w * s), pack_bf16x2(b.x * s, b.y * s),
                         pack_bf16x2(b.z * s, b.w * s));
  reinterpret_cast<uint4*>(p.dq)[i] = out;
}

int launch_bwd128_main(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& tdq, const BwdParams& p, bool dq, cudaStream_t stream);
int launch_bwd_dq_det(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream);

// deterministic: dK and dV by the gradient kernel without its dQ part, dQ
// by fa_bwd_dq_det_kernel (one CTA per query tile, key tiles in a fixed
// order), so no sum depends on the order in which CTAs run.
template <int D>
int launch_bwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                 const CUtensorMap& tdq, const CUtensorMap& tdk, const CUtensorMap& tdv, const BwdParams& p,
                 bool deterministic, cudaStream_t stream) {
  const long long rows = p.T * p.Hq;
  const long long pre_blocks = (rows * 8 + 255) / 256;
  note_launch();
  fa_bwd_rowdot_kernel<D><<<static_cast<unsigned>(pre_blocks), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if constexpr (D == 64) {
    using Lay = BwdLayout<D>;
    auto kern = deterministic ? fa_bwd_kernel<D, false> : fa_bwd_kernel<D, true>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
    if (e != cudaSuccess) return e;
    // persistent: one CTA per SM, or one per unit when there are fewer
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long units = static_cast<long long>(p.n_kvtiles) * p.B * p.Hkv;
    const int grid = static_cast<int>(units < sms ? units : sms);
    note_launch();
    kern<<<grid, kBwdThreads, Lay::kBytes, stream>>>(tq, tk, tv, tdo, tdq, tdk, tdv, p);
    e = cudaGetLastError();
  } else {
    e = static_cast<cudaError_t>(launch_bwd128_main(tq, tk, tv, tdo, tdq, p, !deterministic, stream));
  }
  if (e != cudaSuccess) return e;
  if (deterministic) return launch_bwd_dq_det(D, tq, tk, tv, tdo, p, stream);
  const long long n8 = rows * D / 8;
  note_launch();
  fa_bwd_dq_kernel<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, stream>>>(p, n8);
  return cudaGetLastError();
}

int launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
               const CUtensorMap& tdq, const CUtensorMap& tdk, const CUtensorMap& tdv, const BwdParams& p,
               bool deterministic, cudaStream_t stream) {
  if (d == 64) return launch_bwd_d<64>(tq, tk, tv, tdo, tdq, tdk, tdv, p, deterministic, stream);
  if (d == 128) return launch_bwd_d<128>(tq, tk, tv, tdo, tdq, tdk, tdv, p, deterministic, stream);
  return -1;
}

}  // namespace fa
