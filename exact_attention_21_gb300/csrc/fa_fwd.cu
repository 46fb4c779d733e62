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
// After a unit's first tile, P is taken against the current reference
// before any row max: the tile is kept when its row sum stays within
// 2^kRescaleSlack (so every p does), which is exactly when the max test
// would have kept the reference; otherwise the tile is redone with the row
// max.  Same P, same result, without the max in the common case.  With the
// key columns split between the two softmax warpgroups (d = 64) each keeps
// its own reference and decides per warp; with one shared reference per row
// (d = 128) the 256 softmax threads take one decision per tile through the
// exchange barrier the row max would have used.
//
// The kernel is persistent: one CTA per SM walks work units (128-row query
// tile, query head, sequence) in heavy-first order, keeping its TMEM,
// barriers and K/V ring across units so each unit's loads overlap the previous
// unit's tail.  The products are issued from two threads and the score tile
// is triple-buffered: S of the next key tiles is computed while the softmax
// works on the current one and P V of the previous one runs, and an S never
// queues behind a P V that is still waiting for its softmax.  Warp roles:
//   warp 0       TMA producer for Q (per unit) and K_j (lane 0), and at
//                d = 64 also for V_j (lane 1);
//   warp 3       TMA producer for V_j (d = 128); at d = 64 the second P V
//                issuer.  K and V are loaded by separate threads, so a K load
//                never waits behind a V ring slot that P V has not released.
//   warp 1       TMEM allocator and S issuer: S_j = Q K_j^T into buffer j % 3.
//   warp 2       P V issuer: O += P_j V_j (P_j read from TMEM); at d = 64
//                keys 0..63 only, keys 64..127 by warp 3 (paged: warp 12,
//                since the paged producers take whole warps).
//   warps 4..7   softmax, key columns 0..63 of each score tile;
//   warps 8..11  softmax, key columns 64..127.
//                Thread t of each softmax warpgroup owns query row
//                32 * (warp % 4) + lane (that TMEM lane).  The two
//                warpgroups exchange their partial row maxima through shared
//                memory once per key tile, so both use the same reference;
//                each keeps its own partial row sum, rescales its half of O
//                and writes its half of the output.
//
// TMEM (512 columns): S buffers [0, 128), [128, 256), [256, 384) (bf16 P over
// the first 64 columns of a buffer once read: keys 0..63 in columns 0..31,
// keys 64..127 in columns 32..63), O [384, 384 + d).
#include <cuda_bf16.h>

#include <array>
#include <map>
#include <mutex>
#include <vector>

#include "fa_common.cuh"

namespace fa {

template <int D>
struct FwdLayout {
  static constexpr int kChunkBytes = kTile * 128;          // 128 rows x 64 bf16 (one SW128 box)
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kChunks * kChunkBytes;  // one 128 x D bf16 tile
  // d = 128: one Q buffer (the next unit's Q loads under the current unit's
  // tail) so that K gets three stages; d = 64 has room for two.
  static constexpr int kQBufs = D == 128 ? 1 : 2;
  static constexpr int kStagesK = D == 128 ? 3 : 4;
  static constexpr int kStagesV = D == 128 ? 2 : 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBufs * kTileBytes;
  static constexpr int kOffV = kOffK + kStagesK * kTileBytes;
  static constexpr int kOffX = kOffV + kStagesV * kTileBytes;  // row-max exchange [2 parity][2 halves][128]
  static constexpr int kOffL = kOffX + 2 * 2 * kTile * 4;      // final row-sum exchange [2 parity][2 halves][128]
  // d = 64: two 128 x 64 bf16 tiles (128-byte swizzle) in which a unit's
  // output is staged for one TMA store; d = 128 has no room and stores rows
  static constexpr int kStageBufs = D == 64 ? 2 : 0;
  static constexpr int kOffStage = kOffL + 2 * 2 * kTile * 4;
  static constexpr int kOffBar = kOffStage + kStageBufs * kTileBytes;
  static constexpr int kSBufs = 3;
  // d = 64: the two softmax warpgroups keep separate statistics for their key
  // halves and P V accumulates each half in its own O (TMEM has room for two
  // 64-column accumulators next to the three score buffers); the halves are
  // merged once per unit.  d = 128: one O, statistics exchanged per key tile.
  static constexpr bool kSplit = D == 64;
  // paged d = 64: warp 12 is the second P V issuer (the paged producers
  // need whole warps); otherwise 12 warps (d = 64: the K and V producers
  // share warp 0 and warp 3 issues the second P V), so that one scheduler
  // holds three warps and a thread may use 168 registers
  static constexpr int threads(bool paged) { return kSplit && paged ? 416 : 384; }
  // q_full[2], q_empty[2], k_full[], k_empty[], v_full[], v_empty[], s_full[3], s_free[3],
  // p_full[2][3], pv_done[2][2], xchg, o_final, o_free, drain
  static constexpr int kNumBars = 4 + 2 * kStagesK + 2 * kStagesV + 4 * kSBufs + 4 + 5;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // misc: TMEM slot, abort flag (d = 128: and three per-phase "some row left
  // the rescale bound" flags)
  static constexpr int kBytes = kOffMisc + (kSplit ? 16 : 32) + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColO = 384, kColO1 = 448;  // kColO1: second half's O (d = 64)
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleSlack = 8.f;  // P values stay below 2^8 between rescales
constexpr float kFastLimit = 256.f;   // 2^kRescaleSlack

// PAGED: K and V are read through a page table (prefill over a paged cache),
// the keys of a sequence may outnumber its queries (a cached earlier part),
// and the causal mask is aligned at the newest token.
template <int D, bool PAGED>
__global__ void __launch_bounds__(FwdLayout<D>::threads(PAGED), 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  using Lay = FwdLayout<D>;
  constexpr int NK = Lay::kStagesK, NV = Lay::kStagesV;

  const bool causal = p.causal != 0;
  // Work units: (sequence, query head) pairs are taken in groups of kGroup
  // (chosen by the host)
  // (consecutive heads, so query heads sharing a K/V head stay together); within
  // a group the query tiles go heavy-first (last tile down), so the K/V being
  // read at any time is one group's and stays in L2.  CTA i takes the units i,
  // 2G-1-i, 2G+i, ... of that order (G = gridDim.x), which balances the causal
  // work to within a few per cent.  Units past the end of their sequence are
  // skipped by every role alike.
  const int kGroup = p.group_pairs;
  const int n_pairs = p.Hq * p.B;
  const int n_units = n_pairs * p.n_qtiles;
  const int G = static_cast<int>(gridDim.x);
  auto unit_of = [&](int k) { return k * G + ((k & 1) ? G - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x)); };
  struct Unit {
    long long seq0;
    int L, h, qt, q0, nkv, kvh, sq;
    int Lk, off;  // keys of the sequence; query i sits at key position off + i
  };
  auto unit_at = [&](int u, Unit& w) -> bool {
    // (the divisions by launch constants go through precomputed reciprocals)
    const int gi = fast_div(u, p.div_group_units);  // only the last group can be short
    const int gp = min(kGroup, n_pairs - gi * kGroup);
    const int r = u - gi * kGroup * p.n_qtiles;
    const int rq = gp == kGroup ? fast_div(r, p.div_group_pairs) : r / gp;
    const int pair = gi * kGroup + (r - rq * gp);
    w.qt = p.n_qtiles - 1 - rq;
    const int sq = fast_div(pair, p.div_hq);
    w.h = pair - sq * p.Hq;
    w.sq = sq;
    if (!sequence_bounds(p.cu, sq, p.N, p.T, w.seq0, w.L, p.status)) return false;
    w.q0 = w.qt * kTile;
    if (w.q0 >= w.L) return false;
    if constexpr (PAGED) {
      const int lk = __ldg(p.seqlens_k + sq);
      if (lk < 0 || lk > p.max_pages * p.page_size) {
        atomicOr(p.status, kStatusBadOffsets);
        return false;
      }
      w.Lk = lk;
      w.off = lk - w.L;
      const int n_kt = (lk + kTile - 1) / kTile;
      // causal: the tile's last query row sees keys up to off + that row
      const int last = w.off + min(w.q0 + kTile - 1, w.L - 1);
      w.nkv = !causal ? n_kt : (last < 0 ? 0 : min(n_kt, last / kTile + 1));
    } else {
      w.Lk = w.L;
      w.off = 0;
      w.nkv = kv_tiles_for(w.qt, w.L, causal);
    }
    w.kvh = fast_div(w.h, p.div_qgroup);
    return true;
  };

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Lay::kOffQ;
  uint8_t* sK = smem + Lay::kOffK;
  uint8_t* sV = smem + Lay::kOffV;
  float* xmax = reinterpret_cast<float*>(smem + Lay::kOffX);
  float* xsum = reinterpret_cast<float*>(smem + Lay::kOffL);
  uint8_t* sStage = smem + Lay::kOffStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* q_empty = q_full + 2;
  uint64_t* k_full = q_empty + 2;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  constexpr int NB = Lay::kSBufs;
  constexpr bool kMergedProducers = Lay::kSplit && !PAGED;
  uint64_t* s_full = v_empty + NV;
  uint64_t* s_free = s_full + NB;
  uint64_t* p_full = s_free + NB;   // [half (split) or 0][buffer]
  uint64_t* pv_done = p_full + 2 * NB;  // [half (split) or 0][key-tile parity]
  uint64_t* xchg = pv_done + 4;
  uint64_t* o_final = xchg + 1;
  uint64_t* o_free = o_final + 1;
  uint64_t* drain = o_free + 1;
  uint64_t* stage_full = drain + 1;  // every softmax thread has written its rows of a staged tile
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kOffMisc + 4);
  int* any_out = reinterpret_cast<int*>(smem + Lay::kOffMisc + 8);  // [3]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) { mbar_init(q_full + i, 1); mbar_init(q_empty + i, 1); }
    for (int i = 0; i < NK; ++i) { mbar_init(k_full + i, 1); mbar_init(k_empty + i, 1); }
    // split: both P V issuers release score buffers and V stages and finish O
    constexpr uint32_t npv = Lay::kSplit ? 2 : 1;
    for (int i = 0; i < NV; ++i) { mbar_init(v_full + i, 1); mbar_init(v_empty + i, npv); }
    for (int i = 0; i < NB; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(s_free + i, npv);
      mbar_init(p_full + i, Lay::kSplit ? 128 : 256);
      mbar_init(p_full + NB + i, 128);
    }
    for (int i = 0; i < 4; ++i) mbar_init(pv_done + i, 1);
    mbar_init(xchg, 256);
    mbar_init(o_final, npv);
    mbar_init(o_free, 256);
    mbar_init(drain, npv + 1);
    mbar_init(stage_full, 256);
    *abort_flag = 0;
    if constexpr (!Lay::kSplit) any_out[0] = any_out[1] = any_out[2] = 0;
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

  if (PAGED && (warp == 0 || warp == 3)) {
    // ------------------------------------------------------------ TMA producers, paged K/V
    // The whole warp walks the units: lane 0 waits for ring slots and posts
    // byte counts, then lane j copies page j of the key tile (one box of
    // page_size rows per 64-column chunk, 1 KB-aligned in the slot for
    // page_size >= 8, so the 128-byte swizzle pattern runs on across boxes).
    const bool is_k = warp == 0;  // warp 0: Q and K; warp 3: V
    if (lane == 0) {
      if (is_k) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
      } else {
        tma_prefetch_desc(&tm_v);
      }
    }
    const int ps = p.page_size, pages_per_tile = kTile / ps;
    int k_uses[NK] = {}, v_uses[NV] = {}, q_uses[2] = {};
    int jg = 0, uc = 0;  // key tiles and units so far
    bool ok = true;
    for (int k = 0, u = unit_of(0); u < n_units && ok; u = unit_of(++k)) {
      Unit w;
      if (!unit_at(u, w)) continue;
      if (is_k) {
        const int qb = uc % Lay::kQBufs, qn = uc / Lay::kQBufs;
        if (lane == 0) {
          if (qn >= 1) ok = mbar_wait(q_empty + qb, (qn - 1) & 1, abort_flag);
          if (ok) {
            mbar_arrive_expect_tx(q_full + qb, Lay::kTileBytes);
            for (int c = 0; c < Lay::kChunks; ++c)
              tma_load_3d(sQ + qb * Lay::kTileBytes + c * Lay::kChunkBytes, &tm_q, q_full + qb, c * 64, w.h,
                          static_cast<int>(w.seq0 + w.q0));
          }
        }
        if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
        ++q_uses[qb];
      }
      ++uc;
      for (int j = 0; j < w.nkv; ++j, ++jg) {
        const int slot = is_k ? jg % NK : jg % NV;
        uint64_t* full = is_k ? k_full + slot : v_full + slot;
        if (lane == 0) {
          const int nst = is_k ? NK : NV;
          if (jg >= nst) ok = mbar_wait((is_k ? k_empty : v_empty) + slot, ((jg / nst) - 1) & 1, abort_flag);
          if (ok) mbar_arrive_expect_tx(full, Lay::kTileBytes);
        }
        if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
        if (lane < pages_per_tile) {
          // pages past the cache hold keys that are masked: page 0 is read
          const int lp = j * pages_per_tile + lane;
          int phys = 0;
          if (lp * ps < w.Lk) {
            phys = __ldg(p.block_table + static_cast<long long>(w.sq) * p.max_pages + lp);
            if (phys < 0 || phys >= p.num_pages) {
              atomicOr(p.status, kStatusBadOffsets);
              phys = 0;
            }
          }
          uint8_t* dst = (is_k ? sK : sV) + slot * Lay::kTileBytes + lane * ps * 128;
          for (int c = 0; c < Lay::kChunks; ++c)
            tma_load_3d(dst + c * Lay::kChunkBytes, is_k ? &tm_k : &tm_v, full, c * 64, w.kvh, phys * ps);
        }
        if (is_k) ++k_uses[slot]; else ++v_uses[slot];
      }
    }
    if (lane == 0) {
      if (!ok) give_up();
      // Every copy this warp issued has landed before the CTA may exit.
      int never = 0;
      for (int i = 0; i < Lay::kQBufs; ++i)
        if (q_uses[i]) mbar_wait(q_full + i, (q_uses[i] - 1) & 1, &never);
      for (int i = 0; i < NK; ++i)
        if (k_uses[i]) mbar_wait(k_full + i, (k_uses[i] - 1) & 1, &never);
      for (int i = 0; i < NV; ++i)
        if (v_uses[i]) mbar_wait(v_full + i, (v_uses[i] - 1) & 1, &never);
    }
  } else if (warp == 0 || (warp == 3 && !kMergedProducers)) {
    // ------------------------------------------------------------ TMA producers
    if (kMergedProducers ? lane < 2 : lane == 0) {
      // Q and K: warp 0 (lane 0); V: warp 3, or lane 1 of warp 0
      const bool is_k = kMergedProducers ? lane == 0 : warp == 0;
      if (is_k) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
      } else {
        tma_prefetch_desc(&tm_v);
      }
      int k_uses[NK] = {}, v_uses[NV] = {}, q_uses[2] = {};
      int jg = 0, uc = 0;  // key tiles and units so far
      bool ok = true;
      for (int k = 0, u = unit_of(0); u < n_units && ok; u = unit_of(++k)) {
        Unit w;
        if (!unit_at(u, w)) continue;
        if (is_k) {
          const int qb = uc % Lay::kQBufs, qn = uc / Lay::kQBufs;
          if (qn >= 1 && !(ok = mbar_wait(q_empty + qb, (qn - 1) & 1, abort_flag))) break;
          mbar_arrive_expect_tx(q_full + qb, Lay::kTileBytes);
          for (int c = 0; c < Lay::kChunks; ++c)
            tma_load_3d(sQ + qb * Lay::kTileBytes + c * Lay::kChunkBytes, &tm_q, q_full + qb, c * 64, w.h,
                        static_cast<int>(w.seq0 + w.q0));
          ++q_uses[qb];
        }
        ++uc;
        for (int j = 0; j < w.nkv; ++j, ++jg) {
          const int row_k = static_cast<int>(w.seq0 + j * kTile);
          if (is_k) {
            const int ks = jg % NK;
            if (jg >= NK && !(ok = mbar_wait(k_empty + ks, ((jg / NK) - 1) & 1, abort_flag))) break;
            mbar_arrive_expect_tx(k_full + ks, Lay::kTileBytes);
            for (int c = 0; c < Lay::kChunks; ++c)
              tma_load_3d(sK + ks * Lay::kTileBytes + c * Lay::kChunkBytes, &tm_k, k_full + ks, c * 64, w.kvh,
                          row_k);
            ++k_uses[ks];
          } else {
            const int vs = jg % NV;
            if (jg >= NV && !(ok = mbar_wait(v_empty + vs, ((jg / NV) - 1) & 1, abort_flag))) break;
            mbar_arrive_expect_tx(v_full + vs, Lay::kTileBytes);
            for (int c = 0; c < Lay::kChunks; ++c)
              tma_load_3d(sV + vs * Lay::kTileBytes + c * Lay::kChunkBytes, &tm_v, v_full + vs, c * 64, w.kvh,
                          row_k);
            ++v_uses[vs];
          }
        }
      }
      if (!ok) give_up();
      // Every copy this thread issued has landed before the CTA may exit.
      int never = 0;
      for (int i = 0; i < Lay::kQBufs; ++i)
        if (q_uses[i]) mbar_wait(q_full + i, (q_uses[i] - 1) & 1, &never);
      for (int i = 0; i < NK; ++i)
        if (k_uses[i]) mbar_wait(k_full + i, (k_uses[i] - 1) & 1, &never);
      for (int i = 0; i < NV; ++i)
        if (v_uses[i]) mbar_wait(v_full + i, (v_uses[i] - 1) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kTile, kTile, false, false);
      // Descriptors are built once; a K step only moves the start address.
      const uint64_t q_desc = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t k_desc = sdesc_sw128(smem_u32(sK), 16, 1024);
      int g = 0, uc = 0;  // score tiles and units so far
      bool ok = true;
      for (int k = 0, u = unit_of(0); u < n_units && ok; u = unit_of(++k)) {
        Unit w;
        if (!unit_at(u, w)) continue;
        const int qb = uc % Lay::kQBufs;
        if (!(ok = mbar_wait(q_full + qb, (uc / Lay::kQBufs) & 1, abort_flag))) break;
        ++uc;
        const uint64_t qd = q_desc + static_cast<uint64_t>((qb * Lay::kTileBytes) >> 4);
        int j = 0;
        for (; j < w.nkv; ++j, ++g) {
          const int b = g % NB, ks = g % NK;
          if (!(ok = mbar_wait(k_full + ks, (g / NK) & 1, abort_flag))) break;
          // buffer b still holds the P of score tile g-NB until P V has read it
          if (g >= NB && !(ok = mbar_wait(s_free + b, ((g / NB) - 1) & 1, abort_flag))) break;
          tc_fence_after();
          const uint64_t kd = k_desc + static_cast<uint64_t>((ks * Lay::kTileBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = static_cast<uint64_t>(((kk / 4) * Lay::kChunkBytes + (kk % 4) * 32) >> 4);
            umma_ss(tmem + Lay::kColS + b * kTile, qd + off, kd + off, idesc_s, kk > 0);
          }
          umma_commit(s_full + b);
          umma_commit(k_empty + ks);
        }
        // tile pairs whose S this thread issued for the unit
        if (p.tile_count != nullptr && j > 0) atomicAdd(p.tile_count + w.sq, static_cast<unsigned long long>(j));
        if (ok) umma_commit(q_empty + qb);
      }
      if (!ok) give_up();
      umma_commit(drain);
      int never = 0;
      mbar_wait(drain, 0, &never);
    }
  } else if (warp == 2 || (Lay::kSplit && warp == (kMergedProducers ? 3 : 12))) {
    // ------------------------------------------------------------ P V issuer(s)
    // split: warp 2 accumulates keys 0..63 of every tile into O, warp 3
    // (paged: 12) keys 64..127 into O1 (two threads also keep two N = 64
    // products in flight)
    if (lane == 0) {
      const int hv = warp == 2 ? 0 : 1;
      constexpr uint32_t idesc_o = idesc_bf16_f32(kTile, D, false, true);
      const uint64_t v_desc = sdesc_sw128(smem_u32(sV), Lay::kChunkBytes, 1024);
      int g = 0, uc = 0;  // score tiles and units so far
      bool ok = true;
      for (int k = 0, u = unit_of(0); u < n_units && ok; u = unit_of(++k)) {
        Unit w;
        if (!unit_at(u, w)) continue;
        // O of the previous unit must have been read out before P V restarts it
        if (uc >= 1 && !(ok = mbar_wait(o_free, (uc - 1) & 1, abort_flag))) break;
        ++uc;
        for (int j = 0; j < w.nkv; ++j, ++g) {
          const int b = g % NB, vs = g % NV;
          if (!(ok = mbar_wait(p_full + hv * NB + b, (g / NB) & 1, abort_flag))) break;
          if (!(ok = mbar_wait(v_full + vs, (g / NV) & 1, abort_flag))) break;
          tc_fence_after();
          const uint64_t vd = v_desc + static_cast<uint64_t>((vs * Lay::kTileBytes) >> 4);
          const uint32_t a_tm = tmem + Lay::kColS + b * kTile;  // P, bf16 pairs
          if constexpr (Lay::kSplit) {
            // P of keys 64 hv .. 64 hv + 63 sits in columns 64 hv .. 64 hv + 31
#pragma unroll
            for (int kk = 0; kk < kTile / 32; ++kk)
              umma_ts(tmem + (hv ? Lay::kColO1 : Lay::kColO), a_tm + 64 * hv + kk * 8,
                      vd + static_cast<uint64_t>(((4 * hv + kk) * 2048) >> 4), idesc_o, (j > 0 || kk > 0));
          } else {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              umma_ts(tmem + Lay::kColO, a_tm + (kk / 4) * 64 + (kk % 4) * 8,
                      vd + static_cast<uint64_t>((kk * 2048) >> 4), idesc_o, (j > 0 || kk > 0));
          }
          umma_commit(s_free + b);
          umma_commit(v_empty + vs);
          umma_commit(pv_done + 2 * hv + (g & 1));
        }
        if (ok) umma_commit(o_final);
      }
      if (!ok) give_up();
      umma_commit(drain);
      int never = 0;
      mbar_wait(drain, 0, &never);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax
    const int half = (warp - 4) / 4;  // key columns [64 * half, 64 * half + 64)
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32);
    const float c = p.scale_log2;
    const float2 c2 = make_float2(c, c);
    int g = 0, uc = 0, xp = 0;  // score tiles, units and exchange phases so far
    int fp = 0;                 // tiles that took P against the kept reference first (d = 128)
    int nst = 0;  // units whose output went through a staging tile
    const bool store_issuer = warp == 4 && lane == 0;
    bool ok = true;
    int k = 0, u = unit_of(0);
    Unit w;
    for (; u < n_units; u = unit_of(++k))
      if (unit_at(u, w)) break;
    while (u < n_units && ok) {
      const int qpos = w.q0 + r;
      float m = -INFINITY, l = 0.f;  // reference max (log2 units) and this half's row sum against it
      for (int j = 0; j < w.nkv; ++j, ++g) {
        const int b = g % NB;
        const uint32_t tS = tmem + Lay::kColS + b * kTile;
        if (!(ok = mbar_wait(s_full + b, (g / NB) & 1, abort_flag))) break;
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld_x64(tmem_addr(tS, lane_base, half * 64), sr);
        float* x = reinterpret_cast<float*>(sr);
        const int k0 = j * kTile + half * 64;
        // visible keys of this row: [0, lim)
        const bool need_mask = PAGED ? ((causal && k0 + 63 > w.off + w.q0) || (k0 + 64 > w.Lk))
                                     : ((causal && j == w.qt) || (k0 + 64 > w.L));
        if (need_mask) {
          const int lim = PAGED ? (causal ? min(w.off + qpos + 1, w.Lk) : w.Lk) : (causal ? min(qpos + 1, w.L) : w.L);
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (k0 + i >= lim) x[i] = -INFINITY;
        }
        // Split halves, after a unit's first tile: P against the current
        // reference first, without the row max.  The tile is kept when its row
        // sum stays within 2^slack (then every p does, the bound the lazy
        // rescale keeps); otherwise (also a NaN sum: no reference yet) the
        // warp redoes the tile below with the row max, overwriting P.
        if (j > 0) {
          const float2 nm0 = make_float2(-m, -m);
          float2 fs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                           make_float2(0.f, 0.f)};
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t pk[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              const float2 e = fma2(make_float2(x[cc * 32 + 2 * t], x[cc * 32 + 2 * t + 1]), c2, nm0);
              const float2 pv = make_float2(ex2_approx(e.x), ex2_approx(e.y));
              fs2[t & 3] = add2(fs2[t & 3], pv);
              pk[t] = pack_bf16x2(pv.x, pv.y);
            }
            tmem_st_x16(tmem_addr(tS, lane_base, 64 * half + cc * 16), pk);
          }
          const float2 f01 = add2(fs2[0], fs2[1]), f23 = add2(fs2[2], fs2[3]);
          const float fsum = (f01.x + f01.y) + (f23.x + f23.y);
          bool keep;
          if constexpr (Lay::kSplit) {
            keep = !__any_sync(0xffffffffu, !(fsum <= kFastLimit));
          } else {
            // both halves share the row's reference: one decision for all 256
            // threads, through the exchange barrier (flag slot fp % 3; the
            // slot of two phases on is cleared once every thread has read it)
            if (!(fsum <= kFastLimit)) atomicOr(any_out + fp % 3, 1);
            mbar_arrive(xchg);
            if (!(ok = mbar_wait(xchg, xp & 1, abort_flag))) break;
            ++xp;
            keep = *reinterpret_cast<volatile int*>(any_out + fp % 3) == 0;
            if (half == 0 && r == 0) any_out[(fp + 2) % 3] = 0;
            ++fp;
          }
          if (keep) {
            l += fsum;
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(p_full + (Lay::kSplit ? half * NB : 0) + b);
            continue;
          }
          tmem_st_wait();  // the redo below stores P to the same columns
        }
        float mx[4] = {fmaxf(x[0], x[1]), fmaxf(x[2], x[3]), fmaxf(x[4], x[5]), fmaxf(x[6], x[7])};
#pragma unroll
        for (int i = 8; i < 64; i += 8) {
#pragma unroll
          for (int t = 0; t < 4; ++t) mx[t] = max3(mx[t], x[i + 2 * t], x[i + 2 * t + 1]);
        }
        float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        if constexpr (!Lay::kSplit) {
          // exchange the partial row max with the other half (double-buffered by phase)
          float* xm = xmax + ((xp & 1) * 2) * kTile;
          xm[half * kTile + r] = mt;
          mbar_arrive(xchg);
          if (!(ok = mbar_wait(xchg, xp & 1, abort_flag))) break;
          ++xp;
          mt = fmaxf(xm[r], xm[kTile + r]);
        }
        mt *= c;
        // move the reference only when the row max grows past the slack
        const bool bump = mt > m + kRescaleSlack;
        const float m_new = bump ? mt : m;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = bump ? ex2_approx(m - m_use) : 1.f;
        const float2 nm = make_float2(-m_use, -m_use);
        float2 sum2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const float2 e = fma2(make_float2(x[cc * 32 + 2 * t], x[cc * 32 + 2 * t + 1]), c2, nm);
            const float2 pv = make_float2(ex2_approx(e.x), ex2_approx(e.y));
            sum2[t & 3] = add2(sum2[t & 3], pv);
            pk[t] = pack_bf16x2(pv.x, pv.y);
          }
          // P for keys [64 half + 32 cc, +32) goes to columns [64 half + 16 cc,
          // +16): columns this thread has read itself (the P V issuer takes
          // keys 16 kk .. 16 kk + 15 from column 64 (kk / 4) + 8 (kk % 4)).
          tmem_st_x16(tmem_addr(tS, lane_base, 64 * half + cc * 16), pk);
        }
        const float2 s01 = add2(sum2[0], sum2[1]), s23 = add2(sum2[2], sum2[3]);
        l = l * alpha + ((s01.x + s01.y) + (s23.x + s23.y));
        m = m_new;
        if (j > 0 && __any_sync(0xffffffffu, bump)) {
          // O may only be rescaled once P V of the previous key tile has landed
          // (P V of tile g-NB is done, so the barrier of tile g-1's parity is at
          // most one phase behind: its parity identifies the phase)
          const int ph = Lay::kSplit ? half : 0;
          if (!(ok = mbar_wait(pv_done + 2 * ph + ((g - 1) & 1), ((g - 1) >> 1) & 1, abort_flag))) break;
          tc_fence_after();
          // this half's columns of O, or, split, all of this half's O
#pragma unroll
          for (int cc = 0; cc < (Lay::kSplit ? D / 32 : D / 64); ++cc) {
            uint32_t ov[32];
            const uint32_t ta = Lay::kSplit
                                    ? tmem_addr(tmem + (half ? Lay::kColO1 : Lay::kColO), lane_base, cc * 32)
                                    : tmem_addr(tmem + Lay::kColO, lane_base, half * (D / 2) + cc * 32);
            tmem_ld_x32(ta, ov);
#pragma unroll
            for (int t = 0; t < 32; ++t) ov[t] = __float_as_uint(__uint_as_float(ov[t]) * alpha);
            tmem_st_x32(ta, ov);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full + (Lay::kSplit ? half * NB : 0) + b);
      }
      if (!ok) break;
      // ---- epilogue of this unit.  The next unit is looked up first, while
      // the last P V of this one completes.
      Unit wn;
      int kn = k + 1, un = unit_of(kn);
      for (; un < n_units; un = unit_of(++kn))
        if (unit_at(un, wn)) break;
      // d = 64, whole tile (no row of another sequence in it): the output
      // goes through a staging tile and one TMA store.  Staging buffer
      // nst % 2 was last stored two staged units ago; the issuing thread
      // checks that store has read it before the exchange below, which every
      // softmax thread passes before writing.
      const bool staged = Lay::kStageBufs > 0 && w.q0 + kTile <= w.L && w.seq0 + w.q0 + kTile <= p.T;
      if (staged && store_issuer && nst >= 2) bulk_wait_group_read1();
      if (!(ok = mbar_wait(o_final, uc & 1, abort_flag))) break;
      const int sb = nst & 1;
      ++uc;
      // combine the two halves' row sums (split: and reference maxima)
      xsum[(xp & 1) * kTile * 2 + half * kTile + r] = l;
      if constexpr (Lay::kSplit) xmax[(xp & 1) * kTile * 2 + half * kTile + r] = m;
      mbar_arrive(xchg);
      if (!(ok = mbar_wait(xchg, xp & 1, abort_flag))) break;
      const float l0 = xsum[(xp & 1) * kTile * 2 + r], l1 = xsum[(xp & 1) * kTile * 2 + kTile + r];
      float lt, a0 = 1.f, a1 = 1.f;
      if constexpr (Lay::kSplit) {
        // O = (2^(m0 - m) O0 + 2^(m1 - m) O1) / (2^(m0 - m) l0 + 2^(m1 - m) l1)
        const float m0 = xmax[(xp & 1) * kTile * 2 + r], m1 = xmax[(xp & 1) * kTile * 2 + kTile + r];
        const float mm = fmaxf(m0, m1);
        a0 = mm == -INFINITY ? 0.f : ex2_approx(m0 - mm);
        a1 = mm == -INFINITY ? 0.f : ex2_approx(m1 - mm);
        lt = a0 * l0 + a1 * l1;
        m = mm;
      } else {
        lt = l0 + l1;
      }
      ++xp;
      tc_fence_after();
      uint32_t ov[D / 2];
      if constexpr (Lay::kSplit) {
        // this thread writes output columns [D/2 half, D/2 half + D/2) of its row
        uint32_t ov1[D / 2];
        tmem_ld_x32(tmem_addr(tmem + Lay::kColO, lane_base, half * (D / 2)), ov);
        tmem_ld_x32(tmem_addr(tmem + Lay::kColO1, lane_base, half * (D / 2)), ov1);
#pragma unroll
        for (int t = 0; t < D / 2; ++t)
          ov[t] = __float_as_uint(__uint_as_float(ov[t]) * a0 + __uint_as_float(ov1[t]) * a1);
      } else {
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc)
          tmem_ld_x32(tmem_addr(tmem + Lay::kColO, lane_base, half * (D / 2) + cc * 32), ov + 32 * cc);
      }
      if constexpr (PAGED) {
        // a row with no visible key (more queries than keys under the mask)
        // has nothing accumulated in O: its output is 0
        if (!(lt > 0.f)) {
#pragma unroll
          for (int t = 0; t < D / 2; ++t) ov[t] = 0u;
        }
      }
      // O is in registers: the next unit's P V may start overwriting it
      tc_fence_before();
      mbar_arrive(o_free);
      const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
      const bool row_ok = qpos < w.L;
      const long long tok = w.seq0 + qpos;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) + (tok * p.Hq + w.h) * D + half * (D / 2);
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
          pk[t] = pack_bf16x2(__uint_as_float(ov[32 * cc + 2 * t]) * inv_l, __uint_as_float(ov[32 * cc + 2 * t + 1]) * inv_l);
        if (Lay::kStageBufs > 0 && staged) {
          // row r of the 128-byte-swizzled tile: this half's four 16-byte units
          uint8_t* srow = sStage + sb * Lay::kTileBytes + r * 128;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int unit16 = half * 4 + t;
            *reinterpret_cast<uint4*>(srow + ((unit16 ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
          }
        } else if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int t = 0; t < 4; ++t) dst[t] = make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
        }
      }
      if (Lay::kStageBufs > 0 && staged) {
        fence_proxy_async_smem();
        mbar_arrive(stage_full);
        if (store_issuer) {
          if (!(ok = mbar_wait(stage_full, nst & 1, abort_flag))) break;
          tma_store_3d(&tm_o, sStage + sb * Lay::kTileBytes, 0, w.h, static_cast<int>(w.seq0 + w.q0));
          bulk_commit_group();
        }
        ++nst;
      }
      if (row_ok && half == 0)
        p.lse[static_cast<long long>(w.h) * p.T + tok] = lt > 0.f ? (m + lg2_approx(lt)) * kLn2 : -INFINITY;
      w = wn;
      k = kn;
      u = un;
    }
    // every staged output tile has been written before the CTA exits
    if (store_issuer) bulk_wait_group0();
    if (!ok) give_up();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

// Scheduling group size (in (sequence, head) pairs) for the persistent grid.
// Batched inputs: simulate the kernel's snake assignment of the grouped,
// heavy-first unit order for a few group sizes and keep the one with the
// smallest busiest-CTA load (ties: the smaller group, for L2 locality), among
// groups whose K/V fits in 48 MB.  Packed inputs (lengths on the device): 16.
static int simulate_group_pairs(const FwdParams& p, int G, int d);

static int choose_group_pairs(const FwdParams& p, int G, int d) {
  const int n_pairs = p.Hq * p.B;
  if (p.cu != nullptr || G > 1024 || static_cast<long long>(n_pairs) * p.n_qtiles > (1 << 22))
    return n_pairs < 16 ? n_pairs : 16;
  // one simulation per shape, cached
  static std::mutex mu;
  static std::map<std::array<int, 8>, int> cache;
  const std::array<int, 8> key = {p.Hq, p.B, p.N, p.n_qtiles, p.causal, p.group, G, d};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  const int gs = simulate_group_pairs(p, G, d);
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = gs;
  return gs;
}

static int simulate_group_pairs(const FwdParams& p, int G, int d) {
  const int n_pairs = p.Hq * p.B;
  const int nq = p.n_qtiles;
  const int L = p.N;
  const long long kv_bytes_per_pair = 2ll * L * d * 2 / p.group;  // K and V, shared by the query group
  const int cands[] = {8, 16, 24, 32, 48, 64, 96, 128, 1 << 30};
  int best = n_pairs;
  double best_load = 1e300;
  std::vector<double> load(G);
  for (int gs0 : cands) {
    const int gs = gs0 < n_pairs ? gs0 : n_pairs;
    if (gs * kv_bytes_per_pair > (48ll << 20) && gs != cands[0]) continue;
    for (int i = 0; i < G; ++i) load[i] = 0.0;
    const int n_units = n_pairs * nq;
    for (int u = 0; u < n_units; ++u) {
      const int gi = u / (gs * nq), gp = (gs < n_pairs - gi * gs) ? gs : n_pairs - gi * gs;
      const int r = u - gi * gs * nq;
      const int qt = nq - 1 - r / gp;
      const int k = u / G, i = u % G;
      const int cta = (k & 1) ? G - 1 - i : i;
      load[cta] += (p.causal ? (qt + 1 < nq ? qt + 1 : nq) : nq) + 0.3;  // + per-unit overhead
    }
    double mx = 0.0;
    for (int i = 0; i < G; ++i) mx = load[i] > mx ? load[i] : mx;
    if (mx < best_load * 0.995) {
      best_load = mx;
      best = gs;
    }
    if (gs == n_pairs) break;
  }
  return best;
}

// Host-side launch for one head dimension; returns a cudaError_t value.
template <int D, bool PAGED>
int launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                 const FwdParams& p, cudaStream_t stream) {
  using Lay = FwdLayout<D>;
  cudaError_t e =
      cudaFuncSetAttribute(fa_fwd_kernel<D, PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long units = static_cast<long long>(p.Hq) * p.n_qtiles * p.B;
  const int grid = static_cast<int>(units < sms ? units : sms);  // one CTA per SM, persistent
  FwdParams q = p;
  q.group_pairs = choose_group_pairs(p, grid, D);
  q.div_group_units = make_fast_div(q.group_pairs * q.n_qtiles);
  q.div_group_pairs = make_fast_div(q.group_pairs);
  q.div_hq = make_fast_div(q.Hq);
  q.div_qgroup = make_fast_div(q.group);
  note_launch();
  fa_fwd_kernel<D, PAGED><<<grid, Lay::threads(PAGED), Lay::kBytes, stream>>>(tq, tk, tv, to, q);
  return cudaGetLastError();
}

int launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
               const FwdParams& p, cudaStream_t stream) {
  if (p.block_table != nullptr)
    return d == 64 ? launch_fwd_d<64, true>(tq, tk, tv, to, p, stream)
                   : launch_fwd_d<128, true>(tq, tk, tv, to, p, stream);
  return d == 64 ? launch_fwd_d<64, false>(tq, tk, tv, to, p, stream)
                 : launch_fwd_d<128, false>(tq, tk, tv, to, p, stream);
}

}  // namespace fa
