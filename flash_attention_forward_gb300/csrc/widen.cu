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

__device__ __forceinline__ void widen16(const int8_t* src, uint4* dst, int to_bf16) {
  const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src));
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t out[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[2 * i] = widen_pair(sbyte(w[i], 0), sbyte(w[i], 1), to_bf16);
    out[2 * i + 1] = widen_pair(sbyte(w[i], 2), sbyte(w[i], 3), to_bf16);
  }
  dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
  dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
}

// Group g (16 codes) of a segment: contiguous sources index directly; strided ones split g into
// (b, s, h, 16-code column) with 32-bit arithmetic (rows = B*S*H < 2^31, checked on the host).
__device__ __forceinline__ const int8_t* group_src(const WidenSeg& sg, long long g, int per_row) {
  if (sg.contig) return sg.src + g * 16;
  const uint32_t r = static_cast<uint32_t>(g / per_row);
  const int d16 = static_cast<int>(g - static_cast<long long>(r) * per_row);
  const uint32_t h = r % static_cast<uint32_t>(sg.H);
  const uint32_t bs = r / static_cast<uint32_t>(sg.H);
  const uint32_t sq = bs % static_cast<uint32_t>(sg.S);
  const uint32_t b = bs / static_cast<uint32_t>(sg.S);
  return sg.src + b * sg.sb + sq * sg.ss + h * sg.sh + d16 * 16;
}

__global__ void __launch_bounds__(256) widen_kernel(const WidenParams p) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int si = 0; si < p.n_seg; ++si) {
    const WidenSeg sg = p.seg[si];
    const int per_row = sg.Dh / 16;  // 16-code groups per (b, s, h) row
    const long long n = static_cast<long long>(sg.B) * sg.S * sg.H * per_row;
    uint4* dst = static_cast<uint4*>(sg.dst);
    long long g = tid;
    // four groups per thread and step: four 16-byte loads in flight
    for (; g + 3 * stride < n; g += 4 * stride) {
      const int8_t* s0 = group_src(sg, g, per_row);
      const int8_t* s1 = group_src(sg, g + stride, per_row);
      const int8_t* s2 = group_src(sg, g + 2 * stride, per_row);
      const int8_t* s3 = group_src(sg, g + 3 * stride, per_row);
      widen16(s0, dst + 2 * g, p.to_bf16);
      widen16(s1, dst + 2 * (g + stride), p.to_bf16);
      widen16(s2, dst + 2 * (g + 2 * stride), p.to_bf16);
      widen16(s3, dst + 2 * (g + 3 * stride), p.to_bf16);
    }
    for (; g < n; g += stride) widen16(group_src(sg, g, per_row), dst + 2 * g, p.to_bf16);
  }
}

}  // namespace

cudaError_t launch_widen(const WidenParams& p, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = current_device_sms(&dev, &sms)) != cudaSuccess) return e;
  long long groups = 0;
  for (int i = 0; i < p.n_seg; ++i)
    groups = max(groups, static_cast<long long>(p.seg[i].B) * p.seg[i].S * p.seg[i].H * (p.seg[i].Dh / 16));
  const long long want = (groups + 255) / 256;
  const int grid = static_cast<int>(want < 8LL * sms ? (want > 0 ? want : 1) : 8LL * sms);
  widen_kernel<<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace sdpa
