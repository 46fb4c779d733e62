// Allocation-free variant of the backward pass.
//
// fa_bwd needs a device workspace (the per-row dots D and the f32 dQ
// accumulator) that the caller allocates.  Some callers cannot allocate device
// memory at the point where they need gradients: code running inside a
// memory-pool-managed runtime that forbids cudaMalloc outside its own
// allocator, plugins loaded into a host program that owns all device memory,
// or callers that must not add allocation latency or fragmentation to a tight
// loop.  fa_bwd_noalloc serves them by taking its scratch from a fixed array
// compiled into this library instead of from the caller.
//
// The array lives in device global memory for as long as the library is
// loaded, on every GPU that loads it, and every call shares it.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/fa.h"

namespace fa {
// Records an error message for fa_last_error_string (defined in fa_api.cu).
int record_error(int code, const char* msg);
}  // namespace fa

namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(FA_BWD_NOALLOC_SCRATCH_BYTES);

// The scratch array.  In host code this name is only a stand-in for the
// symbol: its device address must be fetched with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of this device's copy of the scratch array; looked up once
// per device, with that device current, and kept for the life of the process
// (a cudaDeviceReset unloads the module and leaves the kept address stale).
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
    return fa::record_error(FA_ERR_LAUNCH, "fa_bwd_noalloc: cudaGetDevice failed");
  if (dev >= kMaxDevices) {
    char msg[120];
    snprintf(msg, sizeof msg, "fa_bwd_noalloc: device index %d exceeds the library limit of %d", dev, kMaxDevices);
    return fa::record_error(FA_ERR_INVALID_ARG, msg);
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[160];
      snprintf(msg, sizeof msg, "fa_bwd_noalloc: cudaGetSymbolAddress(scratch) failed: %s", cudaGetErrorString(e));
      return fa::record_error(FA_ERR_LAUNCH, msg);
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d,
                              long long T, float scale, int causal, const int* cu_seqlens, void* stream) {
  const size_t need = fa_bwd_workspace_size(Hq, T, d);
  if (need > kScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof msg,
             "fa_bwd_noalloc: this problem needs %zu bytes of scratch but the built-in array holds %zu; "
             "use fa_bwd with a caller-allocated workspace",
             need, kScratchBytes);
    return fa::record_error(FA_ERR_INVALID_ARG, msg);
  }
  void* scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc != FA_OK) return rc;
  // The backward's row-dot pass rewrites D and zeroes the dQ accumulator on
  // every call, so what an earlier call left in the array does not matter.
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens, scratch,
                kScratchBytes, stream);
}
