// sdpa_decode_noalloc: the split-KV decode for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run attention: allocator-free
// embedded runtimes, hosts that hand out device memory only through their own pool and forbid
// library allocations, and serving loops that must not call cudaMalloc on the hot path (it can
// synchronize the device).  sdpa_decode
// already allocates nothing, but it needs a caller-provided workspace for the per-split
// partial results.  This entry point takes that workspace from a fixed array in the
// library's own device memory instead, so the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ variable: every GPU that loads this library holds
// kNoAllocScratchBytes of device memory for it until the process exits.  All calls on a
// device share it, and it keeps whatever the last call left in it; the decode writes every
// partial it later reads, so nothing needs clearing between calls.  Two calls whose kernels
// overlap on the GPU (different streams, no ordering between them) race on the array.
#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "sdpa.h"

namespace sdpa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kMaxScratchDevices = 64;
float* g_noalloc_ptr[kMaxScratchDevices] = {};
std::mutex g_noalloc_mu;

// Device address of this device's scratch array.  The host-side name of the array is only a
// stand-in; the address a kernel can use comes from cudaGetSymbolAddress, resolved once per
// device with that device current.
cudaError_t noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<float*>(ptr);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace sdpa

using namespace sdpa;

extern "C" int sdpa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_len,
                                   void* o, float* lse, int B, int Hq, int Hkv, int max_kv, int D, int Dv,
                                   const int64_t* strides, float scale, sdpa_dtype dtype, void* stream) {
  DecodeCall call;
  const int rc = decode_check(q, k_cache, v_cache, nullptr, kv_len, o, lse, B, Hq, Hkv, max_kv, 0, 0, 0, D, Dv,
                              strides, scale, dtype, &call);
  if (rc != SDPA_OK) return rc;
  // the partials must fit the fixed scratch array
  if (decode_partials_bytes(B, Hq, max_kv, Dv) > kNoAllocScratchBytes) return SDPA_ERR_UNSUPPORTED;
  float* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return SDPA_ERR_CUDA;
  return decode_launch(call, scratch, static_cast<cudaStream_t>(stream));
}
