/*
 * fa.h — C ABI of the exact-attention library (libfa.so, sm_103a / GB300).
 *
 * The library computes exact scaled-dot-product attention
 *     O = softmax(scale * Q K^T) V
 * tile by tile with the online-softmax recurrence, so that the N x N score and
 * probability matrices never reach device memory, and its gradient by
 * recomputing each tile from the saved per-row LogSumExp.  Sources:
 *   - "FlashAttention：从 Safe Softmax 到分块计算": section 1 (formula and
 *     shapes), section 3.2 (merge rule of the running max m, sum l and
 *     unnormalised output), section 5.2 (causal mask s_ij = -inf for j > i),
 *     section 7 (tiled forward), section 8 (per-row LogSumExp kept for the
 *     backward pass).
 *   - "企业官网建设流程全解析" (FlashAttention data-flow notes), section 2.1
 *     (forward loop, P = exp(S - m_new)), section 2.3 (backward:
 *     dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(dP * P))).
 *   - "Attention 算子优化…", section 四 (causal tile skipping, recompute in
 *     the backward pass), section 五 (GQA: consecutive groups of query heads
 *     share one K/V head), section 二 (packed variable-length sequences).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     allocates no device memory and keeps no pointer after a call returns.
 *   - Element types: q, k, v, o, dO, dq, dk, dv are bfloat16 (passed as void*);
 *     lse and workspaces are float32.
 *   - Layout is token-major: q, o, dO, dq are [T, Hq, d] and k, v, dk, dv are
 *     [T, Hkv, d], contiguous, head dimension innermost.  lse is [Hq, T].
 *   - Batched mode (cu_seqlens == NULL): B sequences of N tokens, T = B * N.
 *     Packed mode (cu_seqlens != NULL): cu_seqlens is a DEVICE int32 array of
 *     B + 1 non-decreasing offsets with cu_seqlens[0] = 0 and
 *     cu_seqlens[B] = T; sequence s is tokens cu_seqlens[s] .. cu_seqlens[s+1]-1
 *     and no sequence may be longer than N.  Offsets outside [0, T] are
 *     detected on the device: the affected sequence is skipped and the next
 *     fa_stream_status() reports FA_ERR_INVALID_ARG.
 *   - Query head h reads K/V head h / (Hq / Hkv).
 *   - Causal masking uses positions relative to each sequence's start; key j
 *     is visible from query i when j <= i.
 *   - scale multiplies the raw scores; it must be positive and finite.
 *   - lse is the natural-log LogSumExp of the scaled, masked scores of each
 *     query row.
 *   - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 *     stream).  Outputs are fully overwritten.  Calls on distinct buffers are
 *     independent; calls that share an output buffer must be ordered by the
 *     caller.
 *
 * Errors: every function returns 0 (FA_OK) or an FA_ERR_* code and never
 * prints or aborts.  Devices with an index of 64 or more are rejected
 * (FA_ERR_INVALID_ARG).  Argument errors are found on the host before any launch.
 * fa_last_error_string() describes the most recent failure of the calling
 * thread.  Device-side conditions (a bounded wait that ran out, bad packed
 * offsets) are latched in a device word that fa_stream_status() reads.
 */
#ifndef EXACT_ATTENTION_FA_H
#define EXACT_ATTENTION_FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,        /* null or misaligned pointer, bad size or shape */
  FA_ERR_UNSUPPORTED_DEVICE = 2, /* current device is not compute capability 10.3 */
  FA_ERR_LAUNCH = 3,             /* a CUDA runtime call or kernel launch failed */
  FA_ERR_TIMEOUT = 4,            /* a device-side bounded wait gave up */
  FA_ERR_UNSUPPORTED = 5         /* valid request this build does not implement */
};

/*
 * Forward pass.  Tiled exact attention with the online-softmax recurrence
 * ("FlashAttention：从 Safe Softmax 到分块计算", sections 3.2 and 7), causal
 * tile skipping ("Attention 算子优化…", section 四), GQA and packed sequences.
 *
 *   q   [T, Hq, d]  bf16, 16-byte aligned          (in)
 *   k   [T, Hkv, d] bf16, 16-byte aligned          (in)
 *   v   [T, Hkv, d] bf16, 16-byte aligned          (in)
 *   o   [T, Hq, d]  bf16, 16-byte aligned          (out)
 *   lse [Hq, T]     f32, 4-byte aligned            (out)
 *   B, Hq, Hkv, N, d: batch (or sequence count), query heads, K/V heads,
 *       sequence length (or longest packed sequence), head dimension.
 *       Requires B, Hq, Hkv, N >= 1, Hq % Hkv == 0, d in {64, 128}.
 *   T   total tokens: B * N in batched mode, cu_seqlens[B] in packed mode.
 *   scale  score multiplier (1/sqrt(d) for standard attention), > 0.
 *   causal 0 or 1.
 *   cu_seqlens  NULL (batched) or device int32 [B + 1] (packed).
 *   stream      cudaStream_t.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int Hq, int Hkv, int N, int d, long long T, float scale, int causal,
           const int* cu_seqlens, void* stream);

/*
 * Backward pass.  Recomputes S and P tile by tile from the saved LSE and
 * applies dV = P^T dO, dP = dO V^T, dS = P * (dP - D) with
 * D = rowsum(dO * O) (equal to rowsum(dP * P)), dQ = scale dS K,
 * dK = scale dS^T Q ("企业官网建设流程全解析", section 2.3; "Attention 算子优化…",
 * section 四 on recomputation).  dK and dV of a K/V head are summed over the
 * query heads that share it.
 *
 *   q, k, v, o, lse  as produced for / by fa_fwd with the same shape arguments (in)
 *   dout [T, Hq, d]  bf16 upstream gradient dO                     (in)
 *   dq [T, Hq, d], dk [T, Hkv, d], dv [T, Hkv, d]  bf16            (out)
 *   workspace        device scratch of at least
 *                    fa_bwd_workspace_size(Hq, T, d) bytes, 256-byte aligned;
 *                    its contents on entry are ignored.
 *   Other arguments as for fa_fwd (d in {64, 128}).
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv,
           int B, int Hq, int Hkv, int N, int d, long long T, float scale, int causal,
           const int* cu_seqlens, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass with results that do not depend on the order in which the
 * GPU runs thread blocks: bitwise identical outputs for identical inputs.
 * fa_bwd sums dQ over key tiles with bulk reduce-adds whose order varies from
 * run to run (an f32 sum is not associative); here dK and dV come from the
 * same kernel without its dQ part, and each query tile's dQ is accumulated by
 * one thread block over the key tiles in ascending order, recomputing S and
 * dP for it ("Attention 算子优化…", section 四: recomputation).  About 1.4x the
 * tensor-core work of fa_bwd.  Arguments, workspace and errors as for fa_bwd.
 */
int fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv,
                         int B, int Hq, int Hkv, int N, int d, long long T, float scale, int causal,
                         const int* cu_seqlens, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Forward pass (prefill) over a paged K/V cache ("Attention 算子优化…",
 * section 五, PagedAttention: the cache is a pool of fixed-size pages and each
 * sequence reaches its pages through a page table, so its K/V need not be
 * contiguous).  The queries are packed as in fa_fwd's packed mode; sequence b
 * has Lq = cu_seqlens_q[b+1] - cu_seqlens_q[b] queries, its newest tokens,
 * and Lk = seqlens_k[b] keys: logical key j is row
 *     block_table[b * max_pages + j / page_size] * page_size + j % page_size
 * of the pool.  Lk may exceed Lq (an earlier part of the sequence already in
 * the cache, e.g. chunked prefill or a cached prompt prefix): query i is then
 * the token at position Lk - Lq + i, and under the causal mask it sees keys
 * j <= Lk - Lq + i (the mask aligned at the newest token; Lk = Lq gives the
 * ordinary mask).  A query row that sees no key (causal with Lk < Lq) gets
 * O = 0 and LSE = -inf.  Tiles wholly under the mask are skipped.
 *
 *   q         [Tq, Hq, d] bf16, 16-byte aligned                     (in)
 *   k_pages, v_pages  [num_pages * page_size, Hkv, d] bf16 page pool,
 *             16-byte aligned (in).  Pool rows that hold no key of any
 *             sequence may hold anything finite: they are read (and
 *             multiplied by zero probabilities) when they share a page or a
 *             128-key tile with live keys.
 *   block_table  device int32 [B, max_pages]                        (in)
 *   cu_seqlens_q device int32 [B + 1] query offsets, as in fa_fwd    (in)
 *   seqlens_k    device int32 [B]: keys of each sequence, at most
 *                max_pages * page_size                              (in)
 *   o [Tq, Hq, d] bf16, lse [Hq, Tq] f32                             (out)
 *   max_seqlen_q  longest query chunk (grid sizing); Tq = cu_seqlens_q[B].
 *   page_size     8, 16, 32, 64 or 128 tokens.
 *   Other arguments as for fa_fwd.  A length out of range, or a table entry
 *   inside a cache that is not a page of the pool, is detected on the device:
 *   that sequence's result is not valid (a bad length skips it, a bad entry
 *   reads page 0 instead) and the next fa_stream_status() reports
 *   FA_ERR_INVALID_ARG.
 */
int fa_fwd_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                 const int* cu_seqlens_q, const int* seqlens_k, void* o, float* lse,
                 int B, int Hq, int Hkv, int max_seqlen_q, int d, long long Tq, float scale, int causal,
                 int page_size, int num_pages, int max_pages, void* stream);

/*
 * fa_fwd and fa_bwd with the kernels' own count of the work they did: the
 * thread that issues the score products adds, for each sequence, the number
 * of (query tile, key tile) pairs whose scores it computed, summed over the
 * query heads, into tile_counts[sequence].  Under the causal mask the tiles
 * entirely above the diagonal are skipped ("Attention 算子优化…", section 四:
 * about half the tiles lie wholly under the mask), so with 128 x 128 tiles a
 * sequence of L tokens counts Hq * sum_{i < ceil(L/128)} min(i + 1, ceil(L/128))
 * pairs (Hq * ceil(L/128)^2 without the mask), the value fa_tile_counts gives
 * per query head.  This measures what the kernels processed, not what the
 * host expects them to.
 *
 *   tile_counts  device int64 [B], 8-byte aligned (out): zeroed on `stream`
 *                by the call, then accumulated by the kernel.
 *   Other arguments, results and errors as for fa_fwd / fa_bwd.  The outputs
 *   are the same as fa_fwd's / fa_bwd's; only the counts are added.
 */
int fa_fwd_counted(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int Hq, int Hkv, int N, int d, long long T, float scale, int causal,
                   const int* cu_seqlens, long long* tile_counts, void* stream);
int fa_bwd_counted(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv,
                   int B, int Hq, int Hkv, int N, int d, long long T, float scale, int causal,
                   const int* cu_seqlens, void* workspace, size_t workspace_bytes,
                   long long* tile_counts, void* stream);

/* Bytes of workspace fa_bwd needs: the row dots D (f32 [Hq, T]) and the f32 dQ
 * accumulator ([T, Hq, d]), each rounded up to 256 bytes.  Returns 0 for
 * non-positive arguments. */
size_t fa_bwd_workspace_size(int Hq, long long T, int d);

/*
 * One decoding step with the K/V cache split into chunks ("Flash-Decoding").
 * Every sequence b has one new query token whose query q[b] attends to all
 * of the sequence's cached keys and values; the result for each query head
 * is O = softmax(scale * K q) V and its LSE ("Attention 算子优化…", section 五:
 * the new token's query against the cached K/V of all earlier tokens, a
 * matrix-vector product bound by HBM bandwidth; "FlashAttention：从 Safe
 * Softmax 到分块计算", section 10: one or a few queries against a long cache
 * call for a split-K/V strategy).  The cache of each sequence is processed in
 * splits whose partial (O, LSE) are merged with the online-softmax rule of
 * section 3 of the same page, which is exact.
 *
 *   q   [B, Hq, d]  bf16, 16-byte aligned: the new token's query of each sequence (in)
 *   k   [T, Hkv, d] bf16, 16-byte aligned: the K cache                      (in)
 *   v   [T, Hkv, d] bf16, 16-byte aligned: the V cache                      (in)
 *   o   [B, Hq, d]  bf16, 16-byte aligned                                   (out)
 *   lse [Hq, B]     f32, 4-byte aligned: natural-log LSE of the scaled scores (out)
 *   B, Hq, Hkv, d   as for fa_fwd; Hq / Hkv must be at most 16
 *                   (FA_ERR_UNSUPPORTED otherwise).
 *   N   longest cache (batched mode: every sequence caches N tokens).
 *   T   cached tokens in all: B * N in batched mode, cu_seqlens_k[B] in packed mode.
 *   cu_seqlens_k  NULL (batched) or device int32 [B + 1] offsets of each
 *                 sequence's cache in k / v (packed); an empty cache gives
 *                 O = 0 and LSE = -inf.
 *   workspace     device scratch of at least fa_decode_workspace_size(B, Hq,
 *                 d, N) bytes, 256-byte aligned (per-split partial results);
 *                 contents on entry are ignored.
 *   Other conventions, errors and asynchrony as for fa_fwd.  The query is the
 *   newest token of its sequence, so no key is masked.
 */
int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse,
              int B, int Hq, int Hkv, int N, int d, long long T, float scale,
              const int* cu_seqlens_k, void* workspace, size_t workspace_bytes, void* stream);

/*
 * E4M3 quantisation of K/V cache rows, as written back to the cache
 * ("Attention 算子优化…", section 六: FP8 K/V cache with per-token scales).
 * Each row of d elements (one token of one K/V head) gets the f32 scale
 * s = max|x| / 448 (1 for an all-zero row) and the codes e4m3(x / s), rounded
 * to nearest even and saturated to +-448 (the "fn" E4M3 variant: no infinities).
 *
 *   x      [rows, d] bf16, 16-byte aligned, e.g. a [T, Hkv, d] cache (rows = T * Hkv)  (in)
 *   x8     [rows, d] E4M3 codes (one byte each), 16-byte aligned                      (out)
 *   scale  [rows] f32, 4-byte aligned                                                 (out)
 *   d      64 or 128.
 * Asynchronous on `stream`; errors as for fa_fwd.
 */
int fa_kv_quantize_fp8(const void* x, void* x8, float* scale, long long rows, int d, void* stream);

/*
 * One decoding step (as fa_decode) over an E4M3 K/V cache produced by
 * fa_kv_quantize_fp8: the cache stays compressed in HBM ("Attention 算子优化…",
 * section 六) and the tensor cores read its K and V tiles as they arrive, in
 * E4M3 x E4M3 products against the query and the probabilities, each written
 * as three E4M3 terms (2^-12 relative for the larger elements, finer than
 * bf16); the per-token scales, the softmax and the accumulation are f32.
 * The result is the attention of q over the dequantised cache k8 * k_scale,
 * v8 * v_scale.
 *
 *   k8, v8    [T, Hkv, d] E4M3 codes, 16-byte aligned                 (in)
 *   k_scale, v_scale  [T, Hkv] f32 per-token scales, 4-byte aligned   (in)
 *   Other arguments as for fa_decode.  d = 128; or d = 64 with an even Hkv
 *   and Hq / Hkv <= 8 (two adjacent K/V heads then form one 128-byte row of
 *   the cache); FA_ERR_UNSUPPORTED otherwise.
 */
int fa_decode_fp8(const void* q, const void* k8, const void* v8, const float* k_scale, const float* v_scale,
                  void* o, float* lse, int B, int Hq, int Hkv, int N, int d, long long T, float scale,
                  const int* cu_seqlens_k, void* workspace, size_t workspace_bytes, void* stream);

/*
 * One decoding step (as fa_decode) over a paged K/V cache ("Attention 算子优化…",
 * section 五, PagedAttention): the cache is a pool of fixed-size pages and each
 * sequence reaches its pages through a page table, so caches need not be
 * contiguous.  Logical key j of sequence b is row
 *     block_table[b * max_pages + j / page_size] * page_size + j % page_size
 * of the pool.  Table entries past a sequence's cache are not read.
 *
 *   k_pages, v_pages  [num_pages * page_size, Hkv, d] bf16 page pool, 16-byte aligned (in)
 *   block_table       device int32 [B, max_pages]: physical page of each logical page (in)
 *   seqlens           device int32 [B]: cache length of each sequence, at most
 *                     max_pages * page_size (in)
 *   page_size         8, 16, 32, 64 or 128 tokens.
 *   workspace         at least fa_decode_workspace_size(B, Hq, d, max_pages * page_size) bytes.
 *   Other arguments as for fa_decode.  A length out of range, or a table
 *   entry inside a cache that is not a page of the pool, is detected on the
 *   device: that sequence's result is not valid and the next
 *   fa_stream_status() reports FA_ERR_INVALID_ARG.
 */
int fa_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                    const int* seqlens, void* o, float* lse, int B, int Hq, int Hkv, int d, int page_size,
                    int num_pages, int max_pages, float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_decode_paged over an E4M3 page pool (codes from fa_kv_quantize_fp8 and
 * f32 per-token scales k_scale, v_scale [num_pages * page_size, Hkv], laid
 * out like the pool).  Head dimensions as for fa_decode_fp8.
 */
int fa_decode_paged_fp8(const void* q, const void* k8_pages, const void* v8_pages, const float* k_scale,
                        const float* v_scale, const int* block_table, const int* seqlens, void* o, float* lse, int B,
                        int Hq, int Hkv, int d, int page_size, int num_pages, int max_pages, float scale,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace fa_decode needs for B sequences, Hq query heads, head
 * dimension d and caches of at most max_seqlen_k tokens (an upper bound over
 * every split length the library picks).  Returns 0 for non-positive
 * arguments. */
size_t fa_decode_workspace_size(int B, int Hq, int d, int max_seqlen_k);

/*
 * Host-side count of the (query tile, key tile) pairs the forward kernel
 * processes per query head, for each sequence, with the kernel's 128 x 128
 * tiles: under the causal mask tiles entirely above the diagonal are skipped
 * ("Attention 算子优化…", section 四).  lengths: host int32 [B]; out: host
 * int64 [B].  Uses the same tile-range function as the kernels.
 */
int fa_tile_counts(int B, const int* lengths, int causal, long long* out);

/*
 * Backward pass for callers that cannot allocate device memory.  No passage of
 * the source pages has a counterpart: this is a library convenience.
 *
 * fa_bwd needs a caller-allocated workspace.  Some callers cannot provide one
 * at the point where they need gradients — for example code running under a
 * runtime whose memory pool forbids cudaMalloc outside its own allocator, or a
 * plugin inside a host program that owns all device memory.  fa_bwd_noalloc
 * takes the same arguments as fa_bwd minus the workspace and uses instead a
 * scratch array of FA_BWD_NOALLOC_SCRATCH_BYTES compiled into the library.
 * It allocates nothing and calls no allocating routine.
 *
 *   - Size limit: fa_bwd_workspace_size(Hq, T, d) must not exceed
 *     FA_BWD_NOALLOC_SCRATCH_BYTES; larger problems get FA_ERR_INVALID_ARG
 *     (and a message from fa_last_error_string) and must use fa_bwd.
 *   - The array stays resident on every GPU that loads the library until the
 *     process exits.
 *   - The first call on each device looks up that device's copy of the array
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.  The address is kept for the rest of the
 *     process: after a cudaDeviceReset of that device the array is unusable
 *     (as is the library's device status word, looked up the same way).
 *   - All calls share the one array and it keeps what the last call left in
 *     it; each call re-initialises what must start at zero.  Calls whose
 *     kernels overlap on the GPU (different streams, no ordering) race on the
 *     array and give wrong gradients: order them.
 *   - Other arguments, layouts and errors as for fa_bwd.
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (64ull * 1024ull * 1024ull)

int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv,
                   int B, int Hq, int Hkv, int N, int d, long long T, float scale, int causal,
                   const int* cu_seqlens, void* stream);

/*
 * Self-test of failure detection (no passage of the source pages has a
 * counterpart).  Every wait inside the kernels is bounded: a wait that runs
 * out latches a bit in the device status word, the kernel winds down without
 * trapping, and the next fa_stream_status() returns FA_ERR_TIMEOUT while the
 * CUDA context stays usable.  This launches one block whose bounded wait, the
 * kernels' own, waits on a barrier nothing ever completes, with a limit of
 * limit_ms milliseconds (1..10000) instead of the kernels' 2 s, so that a
 * caller or a test can exercise that path on demand.  After it,
 * fa_stream_status(stream) returns FA_ERR_TIMEOUT (and clears the word).
 */
int fa_selftest_wait_timeout(int limit_ms, void* stream);

/* Synchronises `stream`, then reports and clears the device status word:
 * FA_ERR_TIMEOUT if a bounded wait gave up, FA_ERR_INVALID_ARG if packed
 * offsets were out of range, FA_ERR_LAUNCH if the stream itself failed. */
int fa_stream_status(void* stream);

/* Text of the calling thread's most recent error (empty string if none). */
const char* fa_last_error_string(void);

/* Number of kernels this library has launched in the calling process, counted
 * on the host at each launch (every entry point above, all devices and
 * streams together).  The difference of two readings around a region is the
 * number of this library's kernels launched in it; a call that fails before
 * launching adds nothing.  Never fails. */
unsigned long long fa_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTENTION_FA_H */
