// Widening of int8 codes to 16-bit copies ahead of the int8-code prefill.  sm_103a has no int8
// tensor-core MMA, so the codes meet in the 16-bit MMA instead: every int8 value is exact in f16
// and bf16, and a dot product of up to 192 code pairs (|sum| <= 192 * 128 * 128 < 2^24) is exact
// in the fp32 accumulator, so the scores equal an int32 accumulation.  The pass is bound by HBM:
// 16 codes (one 16-byte load) become two 16-byte stores per thread and step.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace sdpa {
namespace {

__device__ __forceinline__ uint32_t widen_pair(int a, int b, int to_bf16) {
  if (to_bf16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(static_cast<float>(a), static_cast<float>(b));
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  const __half2 h = __floats2half2_rn(static_cast<float>(a), static_cast<float>(b));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// signed byte i of word w
__device__ __forceinline__ int sbyte(uint32_t w, int i) { return static_cast<int>(static_cast<int8_t>(w >> (8 * i))); }

__global__ void __launch_bounds__(256) widen_kernel(const WidenParams p) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int si = 0; si < p.n_seg; ++si) {
    const WidenSeg sg = p.seg[si];
    const int per_row = sg.Dh / 16;  // 16-code groups per (b, s, h) row
    const long long n = static_cast<long long>(sg.B) * sg.S * sg.H * per_row;
    uint4* dst = static_cast<uint4*>(sg.dst);
    for (long long g = tid; g < n; g += stride) {
      long long r = g / per_row;
      const int d16 = static_cast<int>(g - r * per_row);
      const int h = static_cast<int>(r % sg.H);
      r /= sg.H;
      const int s = static_cast<int>(r % sg.S);
      const int b = static_cast<int>(r / sg.S);
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(sg.src + b * sg.sb + s * sg.ss + h * sg.sh + d16 * 16));
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
      uint32_t out[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        out[2 * i] = widen_pair(sbyte(w[i], 0), sbyte(w[i], 1), p.to_bf16);
        out[2 * i + 1] = widen_pair(sbyte(w[i], 2), sbyte(w[i], 3), p.to_bf16);
      }
      dst[2 * g] = make_uint4(out[0], out[1], out[2], out[3]);
      dst[2 * g + 1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
  }
}

}  // namespace

cudaError_t launch_widen(const WidenParams& p, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  long long groups = 0;
  for (int i = 0; i < p.n_seg; ++i)
    groups = max(groups, static_cast<long long>(p.seg[i].B) * p.seg[i].S * p.seg[i].H * (p.seg[i].Dh / 16));
  const long long want = (groups + 255) / 256;
  const int grid = static_cast<int>(want < 8LL * sms ? (want > 0 ? want : 1) : 8LL * sms);
  widen_kernel<<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace sdpa
