// C ABI of the attention library: argument validation, TMA descriptor setup,
// work-grid sizing and kernel launch.  Declarations and the contract of each
// entry point are in include/fa.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "fa_common.cuh"

namespace fa {
int launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
               const FwdParams& p, cudaStream_t stream);
int launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk, const CUtensorMap& tdv,
               const BwdParams& p, bool deterministic,
               cudaStream_t stream);
int launch_decode(int d, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, cudaStream_t stream);
int launch_decode_fp8(int d, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                      cudaStream_t stream);
int launch_quantize_fp8(int d, const void* x, void* x8, float* scale, long long rows, cudaStream_t stream);
}  // namespace fa

namespace fa {
// A wait that nothing ever completes, through the kernels' own bounded wait:
// warp 1 waits on an mbarrier that warp 0 initialises and never arrives on;
// when the wait gives up it latches the timeout bit in the status word and
// raises the CTA's abort flag, as a kernel role would, and warp 0 (which
// waits on the abort flag) winds down with it.
__global__ void __launch_bounds__(64) fa_selftest_timeout_kernel(unsigned* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* ab = &abort_flag;
  if (threadIdx.x == 32) {
    if (!mbar_wait_limit(&bar, 0, ab, limit_ns)) {
      atomicOr(status, kStatusTimeout);
      *ab = 1;
    }
  } else if (threadIdx.x == 0) {
    // a role that would arrive on the barrier once its work is done; it only
    // waits for the abort, with a bound of its own
    const uint64_t t0 = globaltimer_ns();
    while (!*ab && globaltimer_ns() - t0 < 4 * limit_ns) {
    }
  }
  __syncthreads();
}
}  // namespace fa

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

// Device status word: bits from kStatusTimeout / kStatusBadOffsets / kStatusSmemAlign.
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;
struct DeviceState {
  int checked = 0;       // 0 = not yet, 1 = supported, -1 = unsupported
  unsigned* status = nullptr;
  int sms = 0;           // streaming multiprocessors
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Checks the current device (compute capability 10.3) and finds its status
// word; done once per device.
int device_state(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return fail(FA_ERR_LAUNCH, "cudaGetDevice failed");
  if (dev >= kMaxDevices)
    return fail(FA_ERR_INVALID_ARG, "device index %d exceeds the library limit of %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceState& st = g_dev[dev];
  if (st.checked == 0) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) {
      st.checked = -1;
    } else {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess)
        return fail(FA_ERR_LAUNCH, "cudaGetSymbolAddress(status) failed");
      st.status = static_cast<unsigned*>(addr);
      cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev);
      if (st.sms < 1) st.sms = 1;
      st.checked = 1;
    }
  }
  if (st.checked < 0) return fail(FA_ERR_UNSUPPORTED_DEVICE, "device %d is not compute capability 10.3", dev);
  *out = &st;
  return FA_OK;
}

// [T, H, d] bf16 viewed as a 3-D tensor (d, H, T); box = 64 columns x 1 head
// x 128 tokens with the 128-byte swizzle, which is the K-major SW128 operand
// layout the MMAs read.  Rows past T read as zeros.
int make_map(CUtensorMap* map, const void* base, long long T, int H, int d, const char* what, int box_rows = fa::kTile) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(FA_ERR_LAUNCH, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H) * d * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_INVALID_ARG, "tensor map for %s rejected (CUresult %d)", what, (int)r);
  return FA_OK;
}

// E4M3 [T, H, d] (one byte per element) viewed as (d, H, T); box = 128 columns
// (one 128-byte row) x 1 head x 128 tokens with the 128-byte swizzle.  Rows
// past T read as zeros.
int make_map_u8(CUtensorMap* map, const void* base, long long T, int H, int d, const char* what,
                int box_rows = fa::kTile) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(FA_ERR_LAUNCH, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H) * d};
  cuuint32_t box[3] = {128, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_INVALID_ARG, "tensor map for %s rejected (CUresult %d)", what, (int)r);
  return FA_OK;
}

// f32 [T, H, d] accumulator viewed as (d, H, T); box = 32 columns (128 bytes)
// x 1 head x 128 tokens with the 128-byte swizzle, the layout the backward
// kernel stages dQ tiles in before its bulk reduce-add.
int make_map_f32(CUtensorMap* map, void* base, long long T, int H, int d, const char* what) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(FA_ERR_LAUNCH, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(H) * d * 4};
  cuuint32_t box[3] = {32, 1, static_cast<cuuint32_t>(fa::kTile)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_INVALID_ARG, "tensor map for %s rejected (CUresult %d)", what, (int)r);
  return FA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Shape {
  int B, Hq, Hkv, N, d;
  long long T;
  int n_tiles;  // ceil(N / 128)
};

int check_shape(int B, int Hq, int Hkv, int N, int d, long long T, float scale, int causal, const int* cu,
                Shape* s) {
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 1) return fail(FA_ERR_INVALID_ARG, "B, Hq, Hkv, N must be >= 1");
  if (Hq % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (d != 64 && d != 128) return fail(FA_ERR_INVALID_ARG, "d must be 64 or 128 (got %d)", d);
  if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(FA_ERR_INVALID_ARG, "scale must be positive and finite");
  if (T < 1 || T > (1ll << 31) - 1) return fail(FA_ERR_INVALID_ARG, "T must be in [1, 2^31)");
  if (cu == nullptr && T != static_cast<long long>(B) * N)
    return fail(FA_ERR_INVALID_ARG, "batched mode needs T == B * N");
  if (cu != nullptr && !aligned(cu, 4)) return fail(FA_ERR_INVALID_ARG, "cu_seqlens must be 4-byte aligned");
  if (B > 65535) return fail(FA_ERR_INVALID_ARG, "B must be <= 65535");
  if (static_cast<long long>(Hq) * T * d > (1ll << 40)) return fail(FA_ERR_INVALID_ARG, "problem too large");
  *s = Shape{B, Hq, Hkv, N, d, T, (N + fa::kTile - 1) / fa::kTile};
  if (s->n_tiles > 65535) return fail(FA_ERR_INVALID_ARG, "N too large");
  return FA_OK;
}

// 128-key tiles per decode split.  Decode CTAs are resident one per SM, so a
// grid of (split, K/V head, sequence) CTAs runs in ceil(CTAs / SMs) waves, and
// each CTA costs its tiles plus item_cost tiles of start-up (barrier set-up
// and the latency of its first loads; measured at about four tiles for an
// item of paired d = 64 heads, whose query and output cover two heads, and
// one otherwise).  Picks the split length with the lowest modelled time;
// packed caches are modelled as sequences of the mean length.
// Packed caches numbered compactly (every item exists and the CTAs take
// consecutive ones): the split length with the smallest modelled time of the
// busiest CTA, ceil(items / SMs) items of the split's tiles plus about half a
// tile each, where the items are estimated from the total cached tokens T
// (each sequence's last tile and last split counted as half on average).
int decode_split_tiles_compact(int B, int Hkv, int max_tiles, long long T, int sms) {
  const double tiles = static_cast<double>(T) / fa::kTile + 0.5 * B;
  int best = 1;
  double best_time = 0.0;
  for (int st = 1; st <= std::max(max_tiles, 1); ++st) {
    const double items = Hkv * (tiles / st + 0.5 * B);
    const double time = std::ceil(items / sms) * (std::min<double>(st, tiles / B) + 0.5);
    if (st == 1 || time < best_time) {
      best = st;
      best_time = time;
    }
  }
  return best;
}

int decode_split_tiles(int B, int Hkv, int max_tiles, long long T, bool packed, int sms, double item_cost) {
  const double mean_tiles =
      packed ? std::max(1.0, static_cast<double>(T) / B / fa::kTile) : static_cast<double>(max_tiles);
  int best = 1;
  double best_time = 0.0;
  for (int st = 1; st <= 2 * max_tiles && st <= (1 << 20); st *= 2) {
    const long long per_seq = static_cast<long long>(std::ceil(mean_tiles / st));
    const long long ctas = static_cast<long long>(B) * Hkv * per_seq;
    const long long waves = (ctas + sms - 1) / sms;
    const double time = static_cast<double>(waves) * (std::min<double>(st, mean_tiles) + item_cost);
    if (st == 1 || time < best_time) {
      best = st;
      best_time = time;
    }
  }
  return std::min(best, std::max(max_tiles, 1));
}

}  // namespace

namespace fa {
int record_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace fa

extern "C" {

const char* fa_last_error_string(void) { return g_err; }

unsigned long long fa_launch_count(void) { return fa::launch_counter().load(std::memory_order_relaxed); }

}  // extern "C"

// Shared by fa_fwd and fa_fwd_counted (tile_count == nullptr: no counting).
static int fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                      int N, int d, long long T, float scale, int causal, const int* cu_seqlens,
                      long long* tile_count, void* stream) {
  Shape s{};
  int rc = check_shape(B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens, &s);
  if (rc) return rc;
  if (!q || !k || !v || !o || !lse) return fail(FA_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(FA_ERR_INVALID_ARG, "q, k, v, o must be 16-byte aligned");
  if (!aligned(lse, 4)) return fail(FA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  DeviceState* dev = nullptr;
  if ((rc = device_state(&dev))) return rc;
  CUtensorMap tq, tk, tv, to;
  if ((rc = make_map(&tq, q, T, Hq, d, "q")) || (rc = make_map(&tk, k, T, Hkv, d, "k")) ||
      (rc = make_map(&tv, v, T, Hkv, d, "v")) || (rc = make_map(&to, o, T, Hq, d, "o")))
    return rc;
  fa::FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.cu = cu_seqlens;
  p.status = dev->status;
  p.T = T;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.group = Hq / Hkv;
  p.causal = causal;
  p.n_qtiles = s.n_tiles;
  p.scale_log2 = scale * 1.4426950408889634f;
  if (tile_count != nullptr) {
    if (!aligned(tile_count, 8)) return fail(FA_ERR_INVALID_ARG, "tile_counts must be 8-byte aligned");
    const cudaError_t z = cudaMemsetAsync(tile_count, 0, sizeof(long long) * B, static_cast<cudaStream_t>(stream));
    if (z != cudaSuccess) return fail(FA_ERR_LAUNCH, "zeroing tile_counts failed: %s", cudaGetErrorString(z));
    p.tile_count = reinterpret_cast<unsigned long long*>(tile_count);
  }
  int e = fa::launch_fwd(d, tq, tk, tv, to, p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FA_ERR_LAUNCH, "forward launch failed: %s", cudaGetErrorString((cudaError_t)e));
  return FA_OK;
}

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N, int d,
           long long T, float scale, int causal, const int* cu_seqlens, void* stream) {
  g_err[0] = '\0';
  return fwd_common(q, k, v, o, lse, B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens, nullptr, stream);
}

int fa_fwd_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                 const int* cu_seqlens_q, const int* seqlens_k, void* o, float* lse, int B, int Hq, int Hkv,
                 int max_seqlen_q, int d, long long Tq, float scale, int causal, int page_size, int num_pages,
                 int max_pages, void* stream) {
  g_err[0] = '\0';
  if (!block_table || !cu_seqlens_q || !seqlens_k)
    return fail(FA_ERR_INVALID_ARG, "block_table, cu_seqlens_q and seqlens_k must be non-null");
  if (page_size != 8 && page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128)
    return fail(FA_ERR_INVALID_ARG, "page_size must be 8, 16, 32, 64 or 128 (got %d)", page_size);
  if (num_pages < 1 || max_pages < 1) return fail(FA_ERR_INVALID_ARG, "num_pages and max_pages must be >= 1");
  if (static_cast<long long>(max_pages) * page_size > (1ll << 30) ||
      static_cast<long long>(num_pages) * page_size > (1ll << 31) - 1)
    return fail(FA_ERR_INVALID_ARG, "page pool or page table too large");
  if (!aligned(block_table, 4) || !aligned(seqlens_k, 4))
    return fail(FA_ERR_INVALID_ARG, "block_table and seqlens_k must be 4-byte aligned");
  Shape s{};
  int rc = check_shape(B, Hq, Hkv, max_seqlen_q, d, Tq, scale, causal, cu_seqlens_q, &s);
  if (rc) return rc;
  if (!q || !k_pages || !v_pages || !o || !lse) return fail(FA_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(o, 16))
    return fail(FA_ERR_INVALID_ARG, "q, k_pages, v_pages, o must be 16-byte aligned");
  if (!aligned(lse, 4)) return fail(FA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  DeviceState* dev = nullptr;
  if ((rc = device_state(&dev))) return rc;
  const long long rows = static_cast<long long>(num_pages) * page_size;
  CUtensorMap tq, tk, tv, to;
  if ((rc = make_map(&tq, q, Tq, Hq, d, "q")) || (rc = make_map(&tk, k_pages, rows, Hkv, d, "k_pages", page_size)) ||
      (rc = make_map(&tv, v_pages, rows, Hkv, d, "v_pages", page_size)) || (rc = make_map(&to, o, Tq, Hq, d, "o")))
    return rc;
  fa::FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.cu = cu_seqlens_q;
  p.status = dev->status;
  p.T = Tq;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = max_seqlen_q;
  p.group = Hq / Hkv;
  p.causal = causal;
  p.n_qtiles = s.n_tiles;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.block_table = block_table;
  p.seqlens_k = seqlens_k;
  p.page_size = page_size;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  int e = fa::launch_fwd(d, tq, tk, tv, to, p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FA_ERR_LAUNCH, "forward launch failed: %s", cudaGetErrorString((cudaError_t)e));
  return FA_OK;
}

int fa_fwd_counted(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
                   int d, long long T, float scale, int causal, const int* cu_seqlens, long long* tile_counts,
                   void* stream) {
  g_err[0] = '\0';
  if (!tile_counts) return fail(FA_ERR_INVALID_ARG, "null tile_counts");
  return fwd_common(q, k, v, o, lse, B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens, tile_counts, stream);
}

size_t fa_bwd_workspace_size(int Hq, long long T, int d) {
  if (Hq < 1 || T < 1 || d < 1) return 0;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  return up(static_cast<size_t>(Hq) * T * 4) + up(static_cast<size_t>(T) * Hq * d * 4);
}

// Shared by fa_bwd and fa_bwd_deterministic.
static int bwd_common(const void* q, const void* k, const void* v, const void* o, const void* dout,
                      const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d,
                      long long T, float scale, int causal, const int* cu_seqlens, void* workspace,
                      size_t workspace_bytes, bool deterministic, long long* tile_count, void* stream) {
  Shape s{};
  int rc = check_shape(B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens, &s);
  if (rc) return rc;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace)
    return fail(FA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16))
    return fail(FA_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
  if (!aligned(lse, 4)) return fail(FA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  if (!aligned(workspace, 256)) return fail(FA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const size_t need = fa_bwd_workspace_size(Hq, T, d);
  if (workspace_bytes < need)
    return fail(FA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
  DeviceState* dev = nullptr;
  if ((rc = device_state(&dev))) return rc;
  void* dq_acc = static_cast<char*>(workspace) + (static_cast<size_t>(Hq) * T * 4 + 255) / 256 * 256;
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  if ((rc = make_map(&tq, q, T, Hq, d, "q")) || (rc = make_map(&tk, k, T, Hkv, d, "k")) ||
      (rc = make_map(&tv, v, T, Hkv, d, "v")) || (rc = make_map(&tdo, dout, T, Hq, d, "dout")) ||
      (rc = make_map_f32(&tdq, dq_acc, T, Hq, d, "dq accumulator")) || (rc = make_map(&tdk, dk, T, Hkv, d, "dk")) ||
      (rc = make_map(&tdv, dv, T, Hkv, d, "dv")))
    return rc;
  fa::BwdParams p{};
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.rowdot = static_cast<float*>(workspace);
  p.dq_acc = static_cast<float*>(dq_acc);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.cu = cu_seqlens;
  p.status = dev->status;
  p.T = T;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.group = Hq / Hkv;
  p.causal = causal;
  p.n_kvtiles = s.n_tiles;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  if (tile_count != nullptr) {
    if (!aligned(tile_count, 8)) return fail(FA_ERR_INVALID_ARG, "tile_counts must be 8-byte aligned");
    const cudaError_t z = cudaMemsetAsync(tile_count, 0, sizeof(long long) * B, static_cast<cudaStream_t>(stream));
    if (z != cudaSuccess) return fail(FA_ERR_LAUNCH, "zeroing tile_counts failed: %s", cudaGetErrorString(z));
    p.tile_count = reinterpret_cast<unsigned long long*>(tile_count);
  }
  int e = fa::launch_bwd(d, tq, tk, tv, tdo, tdq, tdk, tdv, p, deterministic, static_cast<cudaStream_t>(stream));
  if (e == -1) return fail(FA_ERR_UNSUPPORTED, "backward kernel unavailable for d = %d", d);
  if (e != cudaSuccess) return fail(FA_ERR_LAUNCH, "backward launch failed: %s", cudaGetErrorString((cudaError_t)e));
  return FA_OK;
}

size_t fa_decode_workspace_size(int B, int Hq, int d, int max_seqlen_k) {
  if (B < 1 || Hq < 1 || d < 1 || max_seqlen_k < 1) return 0;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = static_cast<size_t>(B) * Hq * ((max_seqlen_k + fa::kTile - 1) / fa::kTile);
  return up(rows * d * 4) + up(rows * 4);
}

// Page table of a paged cache (block_table == nullptr: packed or batched cache).
struct Paging {
  const int* block_table = nullptr;
  const int* seqlens = nullptr;
  int page_size = 0, num_pages = 0, max_pages = 0;
};

// Shared by the four decoding entry points (k_scale == nullptr: bf16 cache).
static int decode_common(const void* q, const void* k, const void* v, const float* k_scale, const float* v_scale,
                         void* o, float* lse, int B, int Hq, int Hkv, int N, int d, long long T, float scale,
                         const int* cu_seqlens_k, const Paging& pg, void* workspace, size_t workspace_bytes,
                         void* stream) {
  const bool fp8 = k_scale != nullptr;
  const bool paged = pg.block_table != nullptr;
  if (paged) {
    if (pg.page_size != 8 && pg.page_size != 16 && pg.page_size != 32 && pg.page_size != 64 && pg.page_size != 128)
      return fail(FA_ERR_INVALID_ARG, "page_size must be 8, 16, 32, 64 or 128 (got %d)", pg.page_size);
    if (pg.num_pages < 1 || pg.max_pages < 1) return fail(FA_ERR_INVALID_ARG, "num_pages and max_pages must be >= 1");
    if (static_cast<long long>(pg.max_pages) * pg.page_size > (1ll << 30) ||
        static_cast<long long>(pg.num_pages) * pg.page_size > (1ll << 31) - 1)
      return fail(FA_ERR_INVALID_ARG, "page pool or page table too large");
    if (!pg.seqlens || !aligned(pg.block_table, 4) || !aligned(pg.seqlens, 4))
      return fail(FA_ERR_INVALID_ARG, "block_table and seqlens must be non-null and 4-byte aligned");
  }
  Shape s{};
  int rc = check_shape(B, Hq, Hkv, N, d, T, scale, 0, paged ? pg.seqlens : cu_seqlens_k, &s);
  if (rc) return rc;
  if (Hq / Hkv > 16) return fail(FA_ERR_UNSUPPORTED, "decode supports up to 16 query heads per K/V head");
  if (fp8 && d != 128 && !(d == 64 && Hkv % 2 == 0 && Hq / Hkv <= 8))
    return fail(FA_ERR_UNSUPPORTED,
                "the E4M3 cache is supported for d = 128, and for d = 64 with an even Hkv and Hq / Hkv <= 8");
  if (!q || !k || !v || !o || !lse || !workspace || (fp8 && !v_scale)) return fail(FA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(FA_ERR_INVALID_ARG, "q, k, v, o must be 16-byte aligned");
  if (!aligned(lse, 4) || (fp8 && (!aligned(k_scale, 4) || !aligned(v_scale, 4))))
    return fail(FA_ERR_INVALID_ARG, "lse and the scales must be 4-byte aligned");
  if (!aligned(workspace, 256)) return fail(FA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const size_t need = fa_decode_workspace_size(B, Hq, d, N);
  if (workspace_bytes < need)
    return fail(FA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
  DeviceState* dev = nullptr;
  if ((rc = device_state(&dev))) return rc;
  // d = 64 with an even number of K/V heads and at most 8 query heads per K/V
  // head: adjacent K/V heads are paired, [T, Hkv, 64] read as [T, Hkv / 2, 128],
  // and the 128-row tensor-core kernel runs on the pairs
  const bool pair = d == 64 && Hkv % 2 == 0 && Hq / Hkv <= 8;
  const int Hmap = pair ? Hkv / 2 : Hkv, dmap = pair ? 128 : d;
  CUtensorMap tk, tv;
  const int box = paged ? pg.page_size : fa::kTile;
  if (fp8) {
    if ((rc = make_map_u8(&tk, k, T, Hmap, dmap, "k", box)) || (rc = make_map_u8(&tv, v, T, Hmap, dmap, "v", box)))
      return rc;
  } else if ((rc = make_map(&tk, k, T, Hmap, dmap, "k", box)) || (rc = make_map(&tv, v, T, Hmap, dmap, "v", box))) {
    return rc;
  }
  fa::DecodeParams p{};
  p.q = q;
  p.o = o;
  p.lse = lse;
  p.cu = cu_seqlens_k;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.block_table = pg.block_table;
  p.seqlens = pg.seqlens;
  p.page_size = pg.page_size;
  p.max_pages = pg.max_pages;
  p.num_pages = pg.num_pages;
  p.status = dev->status;
  p.T = T;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.group = Hq / Hkv;
  if (pair) {
    p.pair = 1;
    p.Hkv = Hkv / 2;
    p.group = 2 * (Hq / Hkv);
  }
  // packed caches of up to the kernel's prefix size: compact item numbering
  const bool packed = !paged && cu_seqlens_k != nullptr;
  const bool tc = d == 128 || pair;
  p.compact = (tc && packed && B <= (fp8 ? 192 : 1024)) ? 1 : 0;
  p.split_tiles = p.compact ? decode_split_tiles_compact(B, p.Hkv, s.n_tiles, T, dev->sms)
                            : decode_split_tiles(B, p.Hkv, s.n_tiles, T, packed, dev->sms, pair ? 4.0 : 1.0);
  p.n_splits = (s.n_tiles + p.split_tiles - 1) / p.split_tiles;
  // one split per row of a batched cache (every sequence has N >= 1 keys):
  // the tensor-core kernel writes O and the LSE itself and no combine runs
  p.direct = (tc && !paged && cu_seqlens_k == nullptr && p.n_splits == 1) ? 1 : 0;
  p.sms = dev->sms;
  const size_t rows = static_cast<size_t>(B) * Hq * p.n_splits;
  p.o_part = static_cast<float*>(workspace);
  p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + (rows * d * 4 + 255) / 256 * 256);
  p.scale_log2 = scale * 1.4426950408889634f;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int e = fp8 ? fa::launch_decode_fp8(d, tk, tv, p, st) : fa::launch_decode(d, tk, tv, p, st);
  if (e == -1) return fail(FA_ERR_UNSUPPORTED, "decode kernel unavailable for d = %d, group %d", d, p.group);
  if (e != cudaSuccess) return fail(FA_ERR_LAUNCH, "decode launch failed: %s", cudaGetErrorString((cudaError_t)e));
  return FA_OK;
}

int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
              int d, long long T, float scale, const int* cu_seqlens_k, void* workspace, size_t workspace_bytes,
              void* stream) {
  g_err[0] = '\0';
  return decode_common(q, k, v, nullptr, nullptr, o, lse, B, Hq, Hkv, N, d, T, scale, cu_seqlens_k, Paging{},
                       workspace, workspace_bytes, stream);
}

int fa_decode_fp8(const void* q, const void* k8, const void* v8, const float* k_scale, const float* v_scale,
                  void* o, float* lse, int B, int Hq, int Hkv, int N, int d, long long T, float scale,
                  const int* cu_seqlens_k, void* workspace, size_t workspace_bytes, void* stream) {
  g_err[0] = '\0';
  if (!k_scale || !v_scale) return fail(FA_ERR_INVALID_ARG, "null scale pointer");
  return decode_common(q, k8, v8, k_scale, v_scale, o, lse, B, Hq, Hkv, N, d, T, scale, cu_seqlens_k, Paging{},
                       workspace, workspace_bytes, stream);
}

int fa_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                    const int* seqlens, void* o, float* lse, int B, int Hq, int Hkv, int d, int page_size,
                    int num_pages, int max_pages, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  g_err[0] = '\0';
  if (!block_table) return fail(FA_ERR_INVALID_ARG, "null block_table");
  if (page_size < 1 || max_pages < 1 || num_pages < 1 || static_cast<long long>(max_pages) * page_size > (1ll << 30) ||
      static_cast<long long>(num_pages) * page_size > (1ll << 31) - 1)
    return fail(FA_ERR_INVALID_ARG, "page_size, num_pages and max_pages must be >= 1 and the pool below 2^31 rows");
  Paging pg{block_table, seqlens, page_size, num_pages, max_pages};
  const long long rows = static_cast<long long>(num_pages) * page_size;
  return decode_common(q, k_pages, v_pages, nullptr, nullptr, o, lse, B, Hq, Hkv, max_pages * page_size, d, rows,
                       scale, nullptr, pg, workspace, workspace_bytes, stream);
}

int fa_decode_paged_fp8(const void* q, const void* k8_pages, const void* v8_pages, const float* k_scale,
                        const float* v_scale, const int* block_table, const int* seqlens, void* o, float* lse, int B,
                        int Hq, int Hkv, int d, int page_size, int num_pages, int max_pages, float scale,
                        void* workspace, size_t workspace_bytes, void* stream) {
  g_err[0] = '\0';
  if (!block_table) return fail(FA_ERR_INVALID_ARG, "null block_table");
  if (!k_scale || !v_scale) return fail(FA_ERR_INVALID_ARG, "null scale pointer");
  if (page_size < 1 || max_pages < 1 || num_pages < 1 || static_cast<long long>(max_pages) * page_size > (1ll << 30) ||
      static_cast<long long>(num_pages) * page_size > (1ll << 31) - 1)
    return fail(FA_ERR_INVALID_ARG, "page_size, num_pages and max_pages must be >= 1 and the pool below 2^31 rows");
  Paging pg{block_table, seqlens, page_size, num_pages, max_pages};
  const long long rows = static_cast<long long>(num_pages) * page_size;
  return decode_common(q, k8_pages, v8_pages, k_scale, v_scale, o, lse, B, Hq, Hkv, max_pages * page_size, d, rows,
                       scale, nullptr, pg, workspace, workspace_bytes, stream);
}

int fa_kv_quantize_fp8(const void* x, void* x8, float* scale, long long rows, int d, void* stream) {
  g_err[0] = '\0';
  if (d != 64 && d != 128) return fail(FA_ERR_INVALID_ARG, "d must be 64 or 128 (got %d)", d);
  if (rows < 1 || rows > (1ll << 40) / d) return fail(FA_ERR_INVALID_ARG, "rows must be in [1, 2^40 / d]");
  if (!x || !x8 || !scale) return fail(FA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(x, 16) || !aligned(x8, 16) || !aligned(scale, 4))
    return fail(FA_ERR_INVALID_ARG, "x and x8 must be 16-byte aligned, scale 4-byte aligned");
  DeviceState* dev = nullptr;
  int rc = device_state(&dev);
  if (rc) return rc;
  int e = fa::launch_quantize_fp8(d, x, x8, scale, rows, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FA_ERR_LAUNCH, "quantize launch failed: %s", cudaGetErrorString((cudaError_t)e));
  return FA_OK;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse, void* dq,
           void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, long long T, float scale, int causal,
           const int* cu_seqlens, void* workspace, size_t workspace_bytes, void* stream) {
  g_err[0] = '\0';
  return bwd_common(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens, workspace,
                    workspace_bytes, false, nullptr, stream);
}

int fa_bwd_counted(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                   void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, long long T, float scale,
                   int causal, const int* cu_seqlens, void* workspace, size_t workspace_bytes,
                   long long* tile_counts, void* stream) {
  g_err[0] = '\0';
  if (!tile_counts) return fail(FA_ERR_INVALID_ARG, "null tile_counts");
  return bwd_common(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens, workspace,
                    workspace_bytes, false, tile_counts, stream);
}

int fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d,
                         long long T, float scale, int causal, const int* cu_seqlens, void* workspace,
                         size_t workspace_bytes, void* stream) {
  g_err[0] = '\0';
  return bwd_common(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens, workspace,
                    workspace_bytes, true, nullptr, stream);
}

int fa_selftest_wait_timeout(int limit_ms, void* stream) {
  g_err[0] = '\0';
  if (limit_ms < 1 || limit_ms > 10000) return fail(FA_ERR_INVALID_ARG, "limit_ms must be in [1, 10000]");
  DeviceState* dev = nullptr;
  int rc = device_state(&dev);
  if (rc) return rc;
  fa::note_launch();
  fa::fa_selftest_timeout_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(
      dev->status, static_cast<unsigned long long>(limit_ms) * 1000000ull);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FA_ERR_LAUNCH, "self-test launch failed: %s", cudaGetErrorString(e));
  return FA_OK;
}

int fa_tile_counts(int B, const int* lengths, int causal, long long* out) {
  g_err[0] = '\0';
  if (B < 0 || (B > 0 && (!lengths || !out))) return fail(FA_ERR_INVALID_ARG, "bad arguments");
  for (int s = 0; s < B; ++s) {
    const int L = lengths[s];
    if (L < 0) return fail(FA_ERR_INVALID_ARG, "negative length");
    const int nq = (L + fa::kTile - 1) / fa::kTile;
    long long n = 0;
    for (int i = 0; i < nq; ++i) n += fa::kv_tiles_for(i, L, causal != 0);
    out[s] = n;
  }
  return FA_OK;
}

int fa_stream_status(void* stream) {
  g_err[0] = '\0';
  DeviceState* dev = nullptr;
  int rc = device_state(&dev);
  if (rc) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FA_ERR_LAUNCH, "stream failed: %s", cudaGetErrorString(e));
  unsigned word = 0;
  if (cudaMemcpy(&word, dev->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return fail(FA_ERR_LAUNCH, "reading the status word failed");
  if (word == 0) return FA_OK;
  const unsigned zero = 0;
  cudaMemcpy(dev->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
  if (word & fa::kStatusTimeout) return fail(FA_ERR_TIMEOUT, "a device-side wait timed out");
  if (word & fa::kStatusSmemAlign)
    return fail(FA_ERR_LAUNCH, "dynamic shared memory of a kernel was not 1024-byte aligned; the kernel did nothing");
  return fail(FA_ERR_INVALID_ARG, "packed sequence offsets out of range");
}

}  // extern "C"
