// Definitions shared by the attention kernels and the host launcher.
#pragma once

#include <atomic>
#include <cstdint>

#include "ptx.cuh"

namespace fa {

// Kernels this library has launched in the process: every launch site counts
// itself just before it launches (read by fa_launch_count).
inline std::atomic<unsigned long long>& launch_counter() {
  static std::atomic<unsigned long long> count{0};
  return count;
}
inline void note_launch() { launch_counter().fetch_add(1, std::memory_order_relaxed); }

// Query and key tiles are 128 x 128: 128 is the M of one tcgen05 MMA and the
// number of TMEM lanes, so each query row owns one TMEM lane.
constexpr int kTile = 128;

constexpr float kLog2e = 1.4426950408889634f;

// Bits of the device status word.
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusBadOffsets = 2u;
constexpr unsigned kStatusSmemAlign = 4u;  // dynamic shared memory not 1 KB aligned

// Key tiles visible from query tile i of a sequence of length L: all of them
// without a mask, else tiles 0..i (tiles right of the diagonal hold only
// masked scores and are skipped).
__host__ __device__ __forceinline__ int kv_tiles_for(int i, int L, bool causal) {
  const int n = (L + kTile - 1) / kTile;
  return causal ? (i + 1 < n ? i + 1 : n) : n;
}

// First query tile that sees key tile j.
__host__ __device__ __forceinline__ int first_q_tile_for(int j, bool causal) {
  return causal ? j : 0;
}

// Start token and length of sequence s; false (and a status bit) when packed
// offsets are out of range.
__device__ __forceinline__ bool sequence_bounds(const int* cu, int s, int N, long long T,
                                                long long& start, int& len, unsigned* status) {
  if (cu == nullptr) {
    start = static_cast<long long>(s) * N;
    len = N;
    return true;
  }
  const int a = __ldg(cu + s), b = __ldg(cu + s + 1);
  if (a < 0 || b < a || b > T || b - a > N) {
    atomicOr(status, kStatusBadOffsets);
    return false;
  }
  start = a;
  len = b - a;
  return true;
}

// n / d for 0 <= n < 2^31 and a divisor d fixed per launch: (n m) >> s with
// l = ceil(log2 d), s = 31 + l and m = ceil(2^s / d) < 2^32 (division by
// invariant integers using multiplication, Granlund and Montgomery), one
// wide multiply and a shift instead of the division's instruction sequence.
struct FastDiv {
  uint32_t m;
  int s;
};
inline FastDiv make_fast_div(int d) {
  int l = 0;
  while ((1 << l) < d) ++l;
  const uint64_t m = ((1ull << (31 + l)) + static_cast<uint64_t>(d) - 1) / static_cast<uint64_t>(d);
  return FastDiv{static_cast<uint32_t>(m), 31 + l};
}
__device__ __forceinline__ int fast_div(int n, FastDiv f) {
  return static_cast<int>((static_cast<uint64_t>(static_cast<uint32_t>(n)) * f.m) >> f.s);
}

struct FwdParams {
  void* o;            // bf16 [T, Hq, d]
  float* lse;         // f32 [Hq, T]
  const int* cu;      // device int32 [B + 1] or null
  unsigned* status;   // device status word
  long long T;
  int B, Hq, Hkv, N, group, causal, n_qtiles;
  int group_pairs;    // (sequence, head) pairs per scheduling group
  // the divisors of the forward's work-unit lookup: units per scheduling
  // group (group_pairs x query tiles), group_pairs, Hq, the GQA group
  FastDiv div_group_units, div_group_pairs, div_hq, div_qgroup;
  float scale_log2;   // scale * log2(e)
  // null, or device [B]: the S-issuing thread adds the (query tile, key tile)
  // pairs whose S it computed, per sequence (summed over query heads)
  unsigned long long* tile_count;
  // paged K/V (prefill over a paged cache): sequence b's keys are the first
  // seqlens_k[b] logical tokens of its pages, logical page j being physical
  // page block_table[b * max_pages + j] of the pool; null for contiguous K/V
  const int* block_table;
  const int* seqlens_k;
  int page_size, max_pages, num_pages;
};

struct BwdParams {
  const void* o;      // bf16 [T, Hq, d]
  const void* dout;   // bf16 [T, Hq, d]
  const float* lse;   // f32 [Hq, T]
  float* rowdot;      // f32 [Hq, T]: D = rowsum(dO * O)
  float* dq_acc;      // f32 [T, Hq, d]
  void* dq;           // bf16 [T, Hq, d]
  void* dk;           // bf16 [T, Hkv, d]
  void* dv;           // bf16 [T, Hkv, d]
  const int* cu;
  unsigned* status;
  long long T;
  int B, Hq, Hkv, N, group, causal, n_kvtiles;
  float scale, scale_log2;
  // null, or device [B]: the S^T-issuing thread adds the (key tile, query
  // tile) pairs whose S^T it computed, per sequence (summed over query heads)
  unsigned long long* tile_count;
};

struct DecodeParams {
  const void* q;      // bf16 [B, Hq, d]: the new token's query per sequence
  void* o;            // bf16 [B, Hq, d]
  float* lse;         // f32 [Hq, B]
  float* o_part;      // f32 [B, Hq, n_splits, d]: normalised output of each split
  float* lse_part;    // f32 [B, Hq, n_splits]
  const int* cu;      // device int32 [B + 1] offsets into the K/V cache, or null
  const float* k_scale;  // E4M3 cache only: f32 [T, Hkv] per-token scales
  const float* v_scale;
  const int* block_table;  // paged cache only: device int32 [B, max_pages], else null
  const int* seqlens;      // paged cache only: device int32 [B]
  int page_size, max_pages, num_pages;
  unsigned* status;
  long long T;        // cached tokens in all
  int B, Hq, Hkv, N, group;
  int n_splits;       // splits per (sequence, K/V head) in the grid
  int split_tiles;    // 128-key tiles per split
  int sms;            // multiprocessors: CTAs of the persistent decode kernel
  float scale_log2;   // scale * log2(e)
  // 1: head dimension 64 run by the 128-row tensor-core kernel on pairs of
  // adjacent K/V heads (Hkv and group above are then per pair: Hkv / 2 pairs,
  // 2 x the GQA group of query heads per pair); 0 otherwise
  int pair;
  // 1: the (split, K/V head, sequence) items are numbered compactly through a
  // prefix of each sequence's split count, built in shared memory at kernel
  // start (packed caches of unequal length); 0: split-major over n_splits
  int compact;
  // 1: one split per (sequence, K/V head) and every sequence non-empty
  // (batched caches): the split kernel writes O and the LSE itself and no
  // combine runs; 0: partial results for the combine
  int direct;
};

}  // namespace fa
