// Two-phase split-KV decode (one query token per sequence) for sm_103a, plus the kernel
// that condenses an fp16 additive mask for the prefill kernels.
//
// Phase 1 (decode_split_kernel): a CTA owns one (sequence b, KV head, split of
// kDecodeSplit keys); its four warps stream disjoint quarters of the split straight from
// HBM with 128-bit loads.  All Hq/Hkv query heads of the KV head ride in the rows of one
// m16n8k16 tensor-core tile, so every K/V byte is read once per KV head.  Each warp runs
// the online softmax over its keys (running max, lazy rescale, running sum), the four
// warps merge in shared memory, and the CTA writes one partial (unnormalised O, max, sum).
// Phase 2 (decode_combine_kernel): per (b, query head) the partials of all splits are
// merged with a log-sum-exp weighting and normalised.
// (page "Xe2 ESIMD Flash Attention - SDP Prefill & Decode", section "Assets": the
// production decode is two-phase; section "kv_len alignment": lengths are not aligned to
// the split size, and keys past kv_len are clamped out.)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace sdpa {

namespace {

constexpr float kDecodeRescaleLog2 = 8.0f;
constexpr float kLn2f = 0.6931471805599453f;

template <int ELEM>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  // rows 8..15 of A (a1, a3) are zero: only the first 8 rows carry query heads
  if constexpr (ELEM == kBF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
  }
}

template <int ELEM>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (ELEM == kBF16)
    return pack_bf16x2(lo, hi);
  else
    return pack_f16x2(lo, hi);
}

template <int ELEM>
__device__ __forceinline__ float sum2(uint32_t w) {
  if constexpr (ELEM == kBF16) {
    return bf16lo_f32(w) + bf16hi_f32(w);
  } else {
    const __half2 h = *reinterpret_cast<const __half2*>(&w);
    return __low2float(h) + __high2float(h);
  }
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

__device__ __forceinline__ uint4 ldg128(const uint16_t* ptr) {
  return __ldg(reinterpret_cast<const uint4*>(ptr));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Thread layout inside a warp (m16n8k16 fragments): g = lane / 4 is the query head of the
// group for A/C rows and the key (QK) or value column (PV) for B; t = lane % 4.
//
// The head dimension is permuted consistently for Q and K, so that each thread's B operand
// for the 8 QK k-steps is exactly four 16-byte loads of its key row: thread t owns dims
// [32 i + 8 t, 32 i + 8 t + 8) for i = 0..3, k-step kk uses chunk i = kk / 2, words 2 (kk%2)
// (virtual k 2t, 2t+1) and 2 (kk%2) + 1 (virtual k 2t+8, 2t+9).  A dot product does not
// depend on the order of its terms, so S is unchanged.
//
// The value dimension is permuted too: PV n-tile nt, column g holds value dim 16 g + nt, so
// each thread's B operand for all 16 n-tiles is one 32-byte run of a value row, and the C
// fragment of thread (g, t) ends up holding value dims [32 t, 32 t + 32) of query head g.
template <int ELEM>
__global__ void __launch_bounds__(kDecodeWarps * 32) decode_split_kernel(const DecodeParams p) {
  constexpr int kWarpKeys = kDecodeSplit / kDecodeWarps;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int L = min(max(__ldg(p.kv_len + b), 0), p.max_kv);
  const int start = split * kDecodeSplit;
  if (start >= L) return;
  const int w_begin = start + warp * kWarpKeys;
  const int w_end = min(w_begin + kWarpKeys, L);
  const int G = p.group;
  const float scale2 = p.scale2;

  uint32_t qf[4][4];
  if (g < G) {
    const uint16_t* qrow = reinterpret_cast<const uint16_t*>(p.q) + b * p.q_b + (int64_t)(kvh * G + g) * p.q_h;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = ldg128(qrow + 32 * i + 8 * t);
      qf[i][0] = v.x, qf[i][1] = v.y, qf[i][2] = v.z, qf[i][3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) qf[i][0] = qf[i][1] = qf[i][2] = qf[i][3] = 0u;
  }

  float acc[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  float m = -INFINITY, l = 0.f;

  const uint16_t* kb = reinterpret_cast<const uint16_t*>(p.k) + b * p.k_b + (int64_t)kvh * p.k_h;
  const uint16_t* vb = reinterpret_cast<const uint16_t*>(p.v) + b * p.v_b + (int64_t)kvh * p.v_h;
  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);

  for (int t0 = w_begin; t0 < w_end; t0 += 16) {
    // keys t0 + g and t0 + 8 + g: four 16-byte pieces each (never past w_end)
    uint4 kr[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int tok = t0 + 8 * nt + g;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        kr[nt][i] = zero4;
        if (tok < w_end) kr[nt][i] = ldg128(kb + (int64_t)tok * p.k_s + 32 * i + 8 * t);
      }
    }
    // values of keys t0 + {2t, 2t+1, 2t+8, 2t+9}, dims [16 g, 16 g + 16)
    uint4 vr[4][2];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int tok = t0 + 2 * t + (u & 1) + 8 * (u >> 1);
      const uint16_t* vp = vb + (int64_t)tok * p.v_s + 16 * g;
      vr[u][0] = zero4;
      vr[u][1] = zero4;
      if (tok < w_end) {
        vr[u][0] = ldg128(vp);
        vr[u][1] = ldg128(vp + 8);
      }
    }
    // S = Q K^T for 16 keys
    float sc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int i = kk >> 1, hs = kk & 1;
        mma16816<ELEM>(sc[nt], qf[i][2 * hs], qf[i][2 * hs + 1], word(kr[nt][i], 2 * hs), word(kr[nt][i], 2 * hs + 1));
      }
    }
    float x[4] = {sc[0][0] * scale2, sc[0][1] * scale2, sc[1][0] * scale2, sc[1][1] * scale2};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int tok = t0 + 2 * t + (u & 1) + 8 * (u >> 1);
      if (tok >= w_end) x[u] = -INFINITY;
    }
    float mb = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    const float m_cand = fmaxf(m, mb);
    if (__any_sync(0xffffffffu, m_cand > m + kDecodeRescaleLog2)) {
      const float alpha = (m_cand == -INFINITY) ? 1.f : ex2(m - m_cand);
      l *= alpha;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) acc[nt][0] *= alpha, acc[nt][1] *= alpha;
      m = m_cand;
    }
    const float neg_m = (m == -INFINITY) ? 0.f : -m;
    const uint32_t a0 = pack2<ELEM>(ex2(x[0] + neg_m), ex2(x[1] + neg_m));
    const uint32_t a2 = pack2<ELEM>(ex2(x[2] + neg_m), ex2(x[3] + neg_m));
    l += sum2<ELEM>(a0) + sum2<ELEM>(a2);
    // O += P V over the 16 keys, 16 n-tiles of 8 (permuted) value columns
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int wi = (nt & 7) >> 1, hv = nt >> 3;
      const uint32_t sel = (nt & 1) ? 0x7632u : 0x5410u;
      const uint32_t b0 = prmt(word(vr[0][hv], wi), word(vr[1][hv], wi), sel);
      const uint32_t b1 = prmt(word(vr[2][hv], wi), word(vr[3][hv], wi), sel);
      mma16816<ELEM>(acc[nt], a0, a2, b0, b1);
    }
  }

  // per-row sum over the four threads sharing a query head
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);

  __shared__ float sm_m[kDecodeWarps][8];
  __shared__ float sm_l[kDecodeWarps][8];
  __shared__ float sm_o[kDecodeWarps][8][kDecodeDv];
  if (g < G) {
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      sm_o[warp][g][32 * t + nt] = acc[nt][0];
      sm_o[warp][g][32 * t + 16 + nt] = acc[nt][1];
    }
    if (t == 0) {
      sm_m[warp][g] = m;
      sm_l[warp][g] = l;
    }
  }
  __syncthreads();
  const int n_splits = p.n_splits_max;
  const int dv = threadIdx.x;  // kDecodeWarps * 32 == kDecodeDv
  for (int r = 0; r < G; ++r) {
    float M = -INFINITY;
#pragma unroll
    for (int wi = 0; wi < kDecodeWarps; ++wi) M = fmaxf(M, sm_m[wi][r]);
    float o = 0.f, ls = 0.f;
#pragma unroll
    for (int wi = 0; wi < kDecodeWarps; ++wi) {
      const float mw = sm_m[wi][r];
      const float e = (mw == -INFINITY) ? 0.f : ex2(mw - M);
      o += e * sm_o[wi][r][dv];
      ls += e * sm_l[wi][r];
    }
    const int h = kvh * G + r;
    float* part = p.ws + ((int64_t)(b * p.Hq + h) * n_splits + split) * (kDecodeDv + 2);
    part[dv] = o;
    if (dv == 0) {
      part[kDecodeDv] = M;
      part[kDecodeDv + 1] = ls;
    }
  }
}

template <int ELEM>
__global__ void __launch_bounds__(kDecodeDv) decode_combine_kernel(const DecodeParams p) {
  const int h = blockIdx.x, b = blockIdx.y, dv = threadIdx.x;
  const int L = min(max(__ldg(p.kv_len + b), 0), p.max_kv);
  const int ns = (L + kDecodeSplit - 1) / kDecodeSplit;
  const float* base = p.ws + (int64_t)(b * p.Hq + h) * p.n_splits_max * (kDecodeDv + 2);
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, base[s * (kDecodeDv + 2) + kDecodeDv]);
  float o = 0.f, ls = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float* part = base + s * (kDecodeDv + 2);
    const float ms = part[kDecodeDv];
    const float e = (ms == -INFINITY) ? 0.f : ex2(ms - M);
    o += e * part[dv];
    ls += e * part[kDecodeDv + 1];
  }
  const float out = ls > 0.f ? o / ls : 0.f;
  uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + b * p.o_b + (int64_t)h * p.o_h;
  if constexpr (ELEM == kBF16)
    orow[dv] = __bfloat16_as_ushort(__float2bfloat16_rn(out));
  else
    orow[dv] = __half_as_ushort(__float2half_rn(out));
  if (p.lse != nullptr && dv == 0) p.lse[b * p.Hq + h] = ls > 0.f ? (M + __log2f(ls)) * kLn2f : -INFINITY;
}

// One warp per mask row: for every 128-key block, a 128-bit word with bit c set where
// mask[b, i, 128 j + c] is -inf, and a flag set where the block row holds any finite
// non-zero value (those are added to the scores by the prefill kernel from the original
// mask).  Keys past Sk read as 0.
__global__ void __launch_bounds__(128) mask_convert_kernel(const MaskConvertParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 4 + warp;
  if (row >= (int64_t)p.B * p.Sq) return;
  const int b = (int)(row / p.Sq), i = (int)(row % p.Sq);
  const uint16_t* src = p.mask + b * p.mask_b + (int64_t)i * p.mask_i;
  for (int jb = 0; jb < p.n_kblocks; ++jb) {
    uint32_t wd[4];
    bool general = false;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int col = jb * 128 + q * 32 + lane;
      const uint16_t v = col < p.Sk ? src[col] : (uint16_t)0;
      const bool neg_inf = v == 0xFC00u;
      general |= !(neg_inf || v == 0u || v == 0x8000u);
      wd[q] = __ballot_sync(0xffffffffu, neg_inf);
    }
    general = __any_sync(0xffffffffu, general);
    if (lane == 0) {
      p.bits[row * p.n_kblocks + jb] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      p.flags[row * p.n_kblocks + jb] = general ? 1 : 0;
    }
  }
}

}  // namespace

cudaError_t launch_decode(int elem, const DecodeParams& p, cudaStream_t st) {
  const dim3 g1(p.n_splits_max, p.Hkv, p.B), g2(p.Hq, p.B);
  if (elem == kBF16) {
    decode_split_kernel<kBF16><<<g1, kDecodeWarps * 32, 0, st>>>(p);
    decode_combine_kernel<kBF16><<<g2, kDecodeDv, 0, st>>>(p);
  } else {
    decode_split_kernel<kF16><<<g1, kDecodeWarps * 32, 0, st>>>(p);
    decode_combine_kernel<kF16><<<g2, kDecodeDv, 0, st>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_mask_convert(const MaskConvertParams& p, cudaStream_t st) {
  const int64_t rows = (int64_t)p.B * p.Sq;
  mask_convert_kernel<<<(unsigned)((rows + 3) / 4), 128, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace sdpa
