// sdpa_decode_noalloc: the split-KV decode for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run attention: code that runs
// while a CUDA graph is being captured, allocator-free embedded runtimes, and hosts that hand
// out device memory only through their own pool and forbid library allocations.  sdpa_decode
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

bool aligned16_na(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool stride_ok_na(int64_t s) { return s >= 0 && s % 8 == 0 && s < (int64_t(1) << 36); }

}  // namespace
}  // namespace sdpa

using namespace sdpa;

extern "C" int sdpa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_len,
                                   void* o, float* lse, int B, int Hq, int Hkv, int max_kv, int D, int Dv,
                                   const int64_t* strides, float scale, sdpa_dtype dtype, void* stream) {
  if (!q || !k_cache || !v_cache || !kv_len || !o) return SDPA_ERR_INVALID;
  if (B < 1 || Hq < 1 || Hkv < 1 || max_kv < 1 || D < 1 || Dv < 1) return SDPA_ERR_INVALID;
  if (Hq % Hkv != 0) return SDPA_ERR_INVALID;
  if (!(std::isfinite(scale) && scale > 0.f)) return SDPA_ERR_INVALID;
  if (dtype != SDPA_F16 && dtype != SDPA_BF16) return SDPA_ERR_UNSUPPORTED;
  if (D != 128 || Dv != kDecodeDv) return SDPA_ERR_UNSUPPORTED;
  const int group = Hq / Hkv;
  if (group > 8) return SDPA_ERR_UNSUPPORTED;
  if (B > 65535 || Hkv > 65535) return SDPA_ERR_UNSUPPORTED;
  // the partials must fit the fixed scratch array
  const size_t n_splits = (size_t)((max_kv + kDecodeSplit - 1) / kDecodeSplit);
  const size_t need = (size_t)B * (size_t)Hq * n_splits * (size_t)(Dv + 2) * sizeof(float);
  if (need > kNoAllocScratchBytes) return SDPA_ERR_UNSUPPORTED;
  int64_t st[SDPA_DECODE_NSTRIDES];
  if (strides) {
    std::memcpy(st, strides, sizeof(st));
  } else {
    const int64_t cs[SDPA_DECODE_NSTRIDES] = {(int64_t)Hq * D, D, (int64_t)max_kv * Hkv * D, (int64_t)Hkv * D, D,
                                              (int64_t)max_kv * Hkv * Dv, (int64_t)Hkv * Dv, Dv, (int64_t)Hq * Dv,
                                              Dv};
    std::memcpy(st, cs, sizeof(st));
  }
  for (int i = 0; i < SDPA_DECODE_NSTRIDES; ++i)
    if (!stride_ok_na(st[i])) return SDPA_ERR_UNSUPPORTED;
  if (!aligned16_na(q) || !aligned16_na(k_cache) || !aligned16_na(v_cache) || !aligned16_na(o))
    return SDPA_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(kv_len) & 3u) return SDPA_ERR_INVALID;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SDPA_ERR_INVALID;

  const CUtensorMapDataType dt = dtype == SDPA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  alignas(64) CUtensorMap tk, tv;
  if (!encode_bshd(&tk, k_cache, dt, 2, B, max_kv, Hkv, D, st[2], st[3], st[4], 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_bshd(&tv, v_cache, dt, 2, B, max_kv, Hkv, Dv, st[5], st[6], st[7], 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return SDPA_ERR_CUDA;
  float* scratch = nullptr;
  uint32_t* status = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess || device_status_ptr(&status) != cudaSuccess) return SDPA_ERR_CUDA;

  DecodeParams p{};
  p.q = q, p.k = k_cache, p.v = v_cache, p.kv_len = kv_len, p.o = o, p.lse = lse;
  p.ws = scratch;
  p.status = status;
  p.q_b = st[0], p.q_h = st[1], p.k_b = st[2], p.k_s = st[3], p.k_h = st[4];
  p.v_b = st[5], p.v_s = st[6], p.v_h = st[7], p.o_b = st[8], p.o_h = st[9];
  p.B = B, p.Hq = Hq, p.Hkv = Hkv, p.max_kv = max_kv, p.group = group;
  p.n_splits_max = (int)n_splits;
  p.scale2 = (float)((double)scale * 1.4426950408889634);
  const cudaError_t e =
      launch_decode(dtype == SDPA_BF16 ? kBF16 : kF16, p, tk, tv, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}
