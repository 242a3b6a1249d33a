// Two-phase split-KV decode (one query token per sequence) for sm_103a, plus the kernel
// that condenses an fp16 additive mask for the prefill kernels.
//
// Phase 1 (decode_split_kernel): a CTA owns one (sequence b, KV head, split of
// kDecodeSplit keys).  A producer warp streams the split's K and V rows with TMA into a
// shared-memory ring; four consumer warps each take a quarter of every chunk.  All Hq/Hkv
// query heads of the KV head ride in the rows of one m16n8k16 tensor-core tile, so every
// K/V byte is read from HBM once.  Each warp runs the online softmax over its keys (running
// max, lazy rescale, running sum), the four warps merge in shared memory, and the CTA
// writes one partial (unnormalised O, max, sum).
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

// D (16 x 8, fp32) += A (16 x 16) B (16 x 8): A rows 0-7 are query heads g of the GQA group
// (a0, a2), rows 8-15 heads g + 8 (a1, a3; zero for groups of at most 8 heads).
template <int ELEM>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  if constexpr (ELEM == kBF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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

// Phase 1 layout.  A CTA is 4 consumer warps plus one producer warp.  The producer streams the
// split's keys in chunks of kDecChunk rows: D / 64 64-column TMA boxes of K and two of V per
// chunk (128-byte swizzle) into a DecCfg<D, WIDE>::STAGES-deep shared-memory ring.  Consumer warp w
// takes rows [16 w, 16 w + 16) of every chunk, copies its fragments to registers and releases
// the stage.
//
// Fragments (m16n8k16): g = lane / 4 is the query head of the group for A/C rows (rows 0-7:
// heads g; rows 8-15: heads g + 8, used by groups of 9-16 heads) and the key (QK) or value
// column (PV) for B; t = lane % 4.
//  * Head dimension, permuted consistently for Q and K: thread t owns dims [32 i + 8 t, +8)
//    for i = 0 .. D/32 - 1; k-step kk uses chunk i = kk / 2, words 2 (kk%2) and 2 (kk%2) + 1.
//    A dot product does not depend on the order of its terms.
//  * Keys: QK n-index n of n-tile nt is key 8 nt + kSigma[n] of the warp's 16, and P.V k-index
//    k is the same key as QK's (nt, n) = (k / 8, k % 8).  Any fixed order of keys gives the
//    same softmax; this one spreads the eight rows a quarter-warp reads over all swizzle phases.
//  * Value dims: P.V n-tile nt, column g is value dim 16 kBeta[g] + nt, so each thread's B
//    operand for all 16 n-tiles is one 32-byte run of a value row; the C fragment of thread
//    (g, t) ends up holding value dims 16 kBeta[2t] + nt and 16 kBeta[2t + 1] + nt.
constexpr int kDecChunk = 64;                           // keys per TMA chunk
constexpr int kDecBox = kDecChunk * 64 * 2;             // one 64-column box of 16-bit rows: 8 KB
constexpr int kDecThreads = (kDecodeWarps + 1) * 32;
// The D = 128 kernel for groups of up to 8 heads fits two CTAs per SM (at most ~200 registers a
// thread) with a 3-stage ring each; the wider variants (groups of 9-16 heads, or D = 192) need
// more registers, run one CTA per SM and keep about as many bytes in flight with a deeper ring.
template <int D, bool WIDE>
struct DecCfg {
  static constexpr int KBOX = D / 64;                       // K boxes per chunk (V: 2, Dv = 128)
  static constexpr int QCH = D / 32;                        // 8-dim runs of the head dim per thread
  static constexpr int STAGE = (KBOX + 2) * kDecBox;        // 32 KB (D = 128) or 40 KB (D = 192)
  static constexpr bool TWO_CTAS = D == 128 && !WIDE;
  static constexpr int STAGES = TWO_CTAS ? 3 : (D == 128 ? 6 : 5);
  static constexpr int SMEM = STAGES * STAGE + 256 + 1024;
  static_assert(D % 64 == 0 && STAGES * STAGE >= kDecodeWarps * 16 * kDecodeDv * 4, "merge buffer fits the ring");
};
__constant__ int kSigma[8] = {0, 4, 1, 5, 2, 6, 3, 7};
__constant__ int kBeta[8] = {0, 2, 1, 3, 4, 6, 5, 7};

// byte offset of the 16-byte unit `unit` (0..7) of row `row` in a 128-byte-swizzled box
__device__ __forceinline__ uint32_t swz(int row, int unit) {
  return static_cast<uint32_t>(row * 128 + ((unit ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

// WIDE: groups of 9-16 query heads per KV head (rows 8-15 of the tiles carry heads 8-15).
template <int ELEM, bool PAGED, int D, bool WIDE>
__global__ void __launch_bounds__(kDecThreads) decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                      const __grid_constant__ CUtensorMap tm_v,
                                                                      const DecodeParams p) {
  using C = DecCfg<D, WIDE>;
  constexpr int ST = C::STAGES;
  constexpr int RH = WIDE ? 2 : 1;  // row halves of the tiles that carry heads
  constexpr int R = 8 * RH;         // heads per warp in the merge buffer
  extern __shared__ uint8_t dsmem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ST * C::STAGE);
  uint64_t* empty = full + ST;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + ST);

  // the combine kernel may be scheduled once every CTA here has started; it waits for this
  // grid's completion before it reads the partials
  pdl_launch_dependents();
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = min(max(__ldg(p.kv_len + b), 0), p.max_kv);
  const int start = split * kDecodeSplit;
  if (start >= L) return;
  const int end = min(start + kDecodeSplit, L);
  const int nchunks = (end - start + kDecChunk - 1) / kDecChunk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecodeWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  __shared__ float sm_m[kDecodeWarps][R];
  __shared__ float sm_l[kDecodeWarps][R];
  const int G = p.group;

  if (warp == kDecodeWarps) {
    // ---------------------------------------------------------- producer (one warp)
    // A chunk is KBOX + 2 boxes (the 64-column parts of K and of V) for contiguous caches and
    // pages of at least 64 rows: lane 0 issues them.  Pages of fewer rows need (KBOX + 2) x 64 /
    // page_size boxes per chunk, one page each: lane 0 posts the byte count and the boxes are
    // issued by separate lanes, so that their page-table reads and issues overlap.
    constexpr int PARTS = C::KBOX + 2;
    const int rows = PAGED ? min(kDecChunk, p.page_size) : kDecChunk;  // rows per box
    const int nsub = kDecChunk / rows;                                 // boxes per operand part
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    int c = 0;
    for (; c < nchunks; ++c) {
      const int s = c % ST, r = c / ST;
      uint8_t* st = smem + s * C::STAGE;
      const int row = start + c * kDecChunk;  // rows past max_kv read as zeros
      if (nsub == 1) {
        if (lane == 0) {
          if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, abort_flag, p.status)) break;
          mbar_arrive_expect_tx(&full[s], C::STAGE);
          int c3 = b, c2 = row;
          if constexpr (PAGED) {
            const int lp = row >> p.log2_page;
            // logical pages past the table read a page index outside the pool: zero rows, masked
            c3 = lp < p.max_pages ? __ldg(p.page_table + b * p.pt_b + lp) : p.n_pages;
            c2 = row & (p.page_size - 1);
          }
#pragma unroll
          for (int kb = 0; kb < C::KBOX; ++kb) tma_load_4d(st + kb * kDecBox, &tm_k, &full[s], 64 * kb, kvh, c2, c3);
          tma_load_4d(st + C::KBOX * kDecBox, &tm_v, &full[s], 0, kvh, c2, c3);
          tma_load_4d(st + (C::KBOX + 1) * kDecBox, &tm_v, &full[s], 64, kvh, c2, c3);
        }
      } else {
        if (r > 0 && !mbar_wait_warp(&empty[s], (r - 1) & 1, abort_flag, p.status)) break;
        if (lane == 0) mbar_arrive_expect_tx(&full[s], C::STAGE);
        __syncwarp();
        if (lane < PARTS * nsub) {
          // part: the 64-column parts of K (KBOX of them), then V columns 0-63 and 64-127
          const int part = lane % PARTS, sub = lane / PARTS;
          const int key = row + sub * rows;
          const int lp = key >> p.log2_page;
          const int phys = lp < p.max_pages ? __ldg(p.page_table + b * p.pt_b + lp) : p.n_pages;
          const bool is_k = part < C::KBOX;
          // page_size is a power of two >= 16, so every box starts 2 KB-aligned in the stage
          tma_load_4d(st + part * kDecBox + sub * rows * 128, is_k ? &tm_k : &tm_v, &full[s],
                      64 * (is_k ? part : part - C::KBOX), kvh, 0, phys);
        }
      }
    }
    if (c < nchunks && lane == 0)  // aborted: let the copies in flight land
      for (int j = max(0, c - ST); j < c; ++j) mbar_drain(&full[j % ST], (j / ST) & 1);
  } else {
    // ---------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;
    const float scale2 = p.scale2;
    uint32_t qf[RH][C::QCH][4];
#pragma unroll
    for (int rh = 0; rh < RH; ++rh) {
      const int head = g + 8 * rh;
      if (head < G) {
        const uint16_t* qrow = reinterpret_cast<const uint16_t*>(p.q) + b * p.q_b + (int64_t)(kvh * G + head) * p.q_h;
#pragma unroll
        for (int i = 0; i < C::QCH; ++i) {
          const uint4 v = ldg128(qrow + 32 * i + 8 * t);
          qf[rh][i][0] = v.x, qf[rh][i][1] = v.y, qf[rh][i][2] = v.z, qf[rh][i][3] = v.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < C::QCH; ++i) qf[rh][i][0] = qf[rh][i][1] = qf[rh][i][2] = qf[rh][i][3] = 0u;
      }
    }
    const int beta_g = kBeta[g];
    int sig_k[2], sig_v[4];  // chunk rows of this thread's K (per n-tile) and V (per u) keys
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) sig_k[nt] = 16 * warp + 8 * nt + kSigma[g];
#pragma unroll
    for (int u = 0; u < 4; ++u) sig_v[u] = 16 * warp + 8 * (u >> 1) + kSigma[2 * t + (u & 1)];

    // acc[nt][0..1]: heads g, acc[nt][2..3]: heads g + 8 (zero products unless WIDE)
    float acc[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    float m[RH], l[RH];
#pragma unroll
    for (int rh = 0; rh < RH; ++rh) m[rh] = -INFINITY, l[rh] = 0.f;
    bool ok = true;

    for (int c = 0; c < nchunks; ++c) {
      const int s = c % ST;
      if (!mbar_wait_warp(&full[s], (c / ST) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      const uint8_t* kS = smem + s * C::STAGE;
      const uint8_t* vS = kS + C::KBOX * kDecBox;
      const int row0 = start + c * kDecChunk;  // key index of chunk row 0
      // every fragment of the chunk goes to registers first, so that the stage refills while the
      // tensor cores and the softmax work on them
      uint4 kr[2][C::QCH];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < C::QCH; ++i) kr[nt][i] = lds128(kS + (i >> 1) * kDecBox + swz(sig_k[nt], (i & 1) * 4 + t));
      uint4 vr[4][2];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool valid = row0 + sig_v[u] < end;  // rows past kv_len may hold anything (NaN)
#pragma unroll
        for (int hv = 0; hv < 2; ++hv) {
          const uint4 x = lds128(vS + (beta_g >> 2) * kDecBox + swz(sig_v[u], 2 * (beta_g & 3) + hv));
          vr[u][hv] = valid ? x : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // fragments are in registers: the stage may refill

      // S = Q K^T for this warp's 16 keys of the chunk
      float sc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int i = kk >> 1, hs = kk & 1;
          mma16816<ELEM>(sc[nt], qf[0][i][2 * hs], WIDE ? qf[RH - 1][i][2 * hs] : 0u, qf[0][i][2 * hs + 1],
                         WIDE ? qf[RH - 1][i][2 * hs + 1] : 0u, word(kr[nt][i], 2 * hs), word(kr[nt][i], 2 * hs + 1));
        }
      }

      // x[rh][u]: score of head g + 8 rh with key u ((nt, n) = (u / 2, 2t + u % 2), V row u)
      float x[RH][4];
#pragma unroll
      for (int rh = 0; rh < RH; ++rh) {
        x[rh][0] = sc[0][2 * rh] * scale2, x[rh][1] = sc[0][2 * rh + 1] * scale2;
        x[rh][2] = sc[1][2 * rh] * scale2, x[rh][3] = sc[1][2 * rh + 1] * scale2;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (row0 + sig_v[u] >= end) x[rh][u] = -INFINITY;
      }
      float m_cand[RH];
      bool need = false;
#pragma unroll
      for (int rh = 0; rh < RH; ++rh) {
        float mb = fmaxf(fmaxf(x[rh][0], x[rh][1]), fmaxf(x[rh][2], x[rh][3]));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
        m_cand[rh] = fmaxf(m[rh], mb);
        need |= m_cand[rh] > m[rh] + kDecodeRescaleLog2;
      }
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int rh = 0; rh < RH; ++rh) {
          const float alpha = (m_cand[rh] == -INFINITY) ? 1.f : ex2(m[rh] - m_cand[rh]);
          l[rh] *= alpha;
#pragma unroll
          for (int nt = 0; nt < 16; ++nt) acc[nt][2 * rh] *= alpha, acc[nt][2 * rh + 1] *= alpha;
          m[rh] = m_cand[rh];
        }
      }
      uint32_t a[RH][2];  // P as the A operand: keys (2t, 2t + 1) and (2t + 8, 2t + 9) of each head row
#pragma unroll
      for (int rh = 0; rh < RH; ++rh) {
        const float neg_m = (m[rh] == -INFINITY) ? 0.f : -m[rh];
        a[rh][0] = pack2<ELEM>(ex2(x[rh][0] + neg_m), ex2(x[rh][1] + neg_m));
        a[rh][1] = pack2<ELEM>(ex2(x[rh][2] + neg_m), ex2(x[rh][3] + neg_m));
        l[rh] += sum2<ELEM>(a[rh][0]) + sum2<ELEM>(a[rh][1]);
      }
      // O += P V over the 16 keys, 16 n-tiles of 8 (permuted) value columns
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const int wi = (nt & 7) >> 1, hv = nt >> 3;
        const uint32_t sel = (nt & 1) ? 0x7632u : 0x5410u;
        const uint32_t b0 = prmt(word(vr[0][hv], wi), word(vr[1][hv], wi), sel);
        const uint32_t b1 = prmt(word(vr[2][hv], wi), word(vr[3][hv], wi), sel);
        mma16816<ELEM>(acc[nt], a[0][0], WIDE ? a[RH - 1][0] : 0u, a[0][1], WIDE ? a[RH - 1][1] : 0u, b0, b1);
      }
    }

#pragma unroll
    for (int rh = 0; rh < RH; ++rh) {
      l[rh] += __shfl_xor_sync(0xffffffffu, l[rh], 1);
      l[rh] += __shfl_xor_sync(0xffffffffu, l[rh], 2);
      if (!ok) {
        m[rh] = -INFINITY;
        l[rh] = 0.f;
      }
    }
    // merge the four warps: per-warp O goes to the (now idle) ring memory
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"n"(kDecodeWarps * 32));  // all consumers are past the ring
    float* sm_o = reinterpret_cast<float*>(smem);               // [warp][head][dv]
#pragma unroll
    for (int rh = 0; rh < RH; ++rh) {
      const int head = g + 8 * rh;
      if (head < G) {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          sm_o[(warp * R + head) * kDecodeDv + 16 * kBeta[2 * t] + nt] = acc[nt][2 * rh];
          sm_o[(warp * R + head) * kDecodeDv + 16 * kBeta[2 * t + 1] + nt] = acc[nt][2 * rh + 1];
        }
        if (t == 0) {
          sm_m[warp][head] = m[rh];
          sm_l[warp][head] = l[rh];
        }
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kDecodeWarps * 32));
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
        o += e * sm_o[(wi * R + r) * kDecodeDv + dv];
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
}

template <int ELEM>
__global__ void __launch_bounds__(kDecodeDv) decode_combine_kernel(const DecodeParams p) {
  const int h = blockIdx.x, b = blockIdx.y, dv = threadIdx.x;
  const int L = min(max(__ldg(p.kv_len + b), 0), p.max_kv);
  const int ns = (L + kDecodeSplit - 1) / kDecodeSplit;
  constexpr int kPart = kDecodeDv + 2;  // floats per partial: O, then max, then sum
  constexpr int kGroup = 8;             // partials whose loads are in flight together
  const float* base = p.ws + (int64_t)(b * p.Hq + h) * p.n_splits_max * kPart;
  pdl_wait();  // the partials come from the split kernel launched before
  float M = -INFINITY;
  for (int s0 = 0; s0 < ns; s0 += kGroup) {
    float m[kGroup];
#pragma unroll
    for (int i = 0; i < kGroup; ++i) m[i] = (s0 + i < ns) ? __ldg(base + (s0 + i) * kPart + kDecodeDv) : -INFINITY;
#pragma unroll
    for (int i = 0; i < kGroup; ++i) M = fmaxf(M, m[i]);
  }
  float o = 0.f, ls = 0.f;
  for (int s0 = 0; s0 < ns; s0 += kGroup) {
    float m[kGroup], x[kGroup], l[kGroup];
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {
      const bool in = s0 + i < ns;
      const float* part = base + (s0 + i) * kPart;
      m[i] = in ? __ldg(part + kDecodeDv) : -INFINITY;
      x[i] = in ? __ldg(part + dv) : 0.f;
      l[i] = in ? __ldg(part + kDecodeDv + 1) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {  // splits in order, as a sequential loop would take them
      const float e = (m[i] == -INFINITY) ? 0.f : ex2(m[i] - M);
      o += e * x[i];
      ls += e * l[i];
    }
  }
  const float out = ls > 0.f ? o / ls : 0.f;
  uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + b * p.o_b + (int64_t)h * p.o_h;
  if constexpr (ELEM == kBF16)
    orow[dv] = __bfloat16_as_ushort(__float2bfloat16_rn(out));
  else
    orow[dv] = __half_as_ushort(__float2half_rn(out));
  if (p.lse != nullptr && dv == 0) p.lse[b * p.Hq + h] = ls > 0.f ? (M + __log2f(ls)) * kLn2f : -INFINITY;
}

// For every (row, 128-key block): a 128-bit word with bit c set where mask[b, i, 128 j + c] is
// -inf, and a flag set where the block row holds any finite non-zero value (those are added to
// the scores by the prefill kernel from the original mask).  Keys past Sk read as 0.
// One warp per (row, group of kMaskGroup blocks): all of the group's loads are issued before
// the first ballot, so each warp keeps kMaskGroup x 4 coalesced 64-byte reads in flight (mask
// rows need only 2-byte alignment, which rules out wider loads).
constexpr int kMaskGroup = 4;

__global__ void __launch_bounds__(128) mask_convert_kernel(const MaskConvertParams p) {
  // the prefill that reads the bits may be scheduled as soon as every CTA here has started; it
  // waits for this grid's completion before its first read of them
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_groups = (p.n_kblocks + kMaskGroup - 1) / kMaskGroup;
  const int64_t item = (int64_t)blockIdx.x * 4 + warp;
  if (item >= (int64_t)p.B * p.Sq * n_groups) return;
  const int64_t row = item / n_groups;
  const int jb0 = static_cast<int>(item % n_groups) * kMaskGroup;
  const int b = (int)(row / p.Sq), i = (int)(row % p.Sq);
  const uint16_t* src = p.mask + b * p.mask_b + (int64_t)i * p.mask_i;
  uint16_t v[kMaskGroup][4];
#pragma unroll
  for (int g = 0; g < kMaskGroup; ++g)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int col = (jb0 + g) * 128 + q * 32 + lane;
      v[g][q] = col < p.Sk ? __ldg(src + col) : (uint16_t)0;
    }
#pragma unroll
  for (int g = 0; g < kMaskGroup; ++g) {
    const int jb = jb0 + g;
    if (jb >= p.n_kblocks) break;  // the same for the whole warp
    uint32_t wd[4];
    bool general = false;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const bool neg_inf = v[g][q] == 0xFC00u;
      general |= !(neg_inf || v[g][q] == 0u || v[g][q] == 0x8000u);
      wd[q] = __ballot_sync(0xffffffffu, neg_inf);
    }
    general = __any_sync(0xffffffffu, general);
    if (lane == 0) {
      p.bits[row * p.n_kblocks + jb] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      p.flags[row * p.n_kblocks + jb] = general ? 1 : 0;
    }
  }
}

// Work-tile prefix of packed variable-length sequences: tile_prefix[b] is the number of work
// tiles (2 x 128 query rows) of the sequences before b, tile_prefix[B] of all of them.  One CTA
// scans the B counts 1024 at a time.  Offsets that are not non-decreasing within [0, total], or
// more tiles than the launch was sized for, raise kStatusBadSeqlens and leave every count zero,
// so the prefill that follows stores nothing.
__global__ void __launch_bounds__(1024) varlen_prep_kernel(const VarlenPrepParams p) {
  __shared__ long long warp_sum[32];  // 64-bit sums: invalid offsets must not overflow them
  __shared__ long long carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  int bad = 0;
  for (int base = 0; base < p.B; base += 1024) {
    const int b = base + tid;
    long long v = 0;
    if (b < p.B) {
      const int q0 = __ldg(p.cu_q + b), q1 = __ldg(p.cu_q + b + 1);
      const int k0 = __ldg(p.cu_k + b), k1 = __ldg(p.cu_k + b + 1);
      if (q1 < q0 || k1 < k0) bad = 1;
      if (b == 0 && (q0 < 0 || k0 < 0)) bad = 1;
      if (b == p.B - 1 && (q1 > p.total_q || k1 > p.total_k)) bad = 1;
      v = (max(0ll, (long long)q1 - q0) + kCtaRows - 1) / kCtaRows;
    }
    long long x = v;  // inclusive scan inside the warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    if (lane == 31) warp_sum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      long long w = warp_sum[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, w, d);
        if (lane >= d) w += y;
      }
      warp_sum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const long long incl = x + (warp > 0 ? warp_sum[warp - 1] : 0ll);
    if (b < p.B) p.tile_prefix[b] = static_cast<int32_t>(carry + incl - v);
    __syncthreads();
    if (tid == 1023) carry += incl;
    __syncthreads();
  }
  const bool fail = __syncthreads_or(bad) || carry > p.max_tiles;
  if (fail) {
    for (int b = tid; b <= p.B; b += 1024) p.tile_prefix[b] = 0;
    if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
  } else if (tid == 0) {
    p.tile_prefix[p.B] = static_cast<int32_t>(carry);
  }
}

template <int ELEM, bool PAGED, int D, bool WIDE>
cudaError_t launch_split_instance(dim3 grid, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                                  cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = current_device_sms(&dev, &sms);
  if (e != cudaSuccess) return e;
  static std::atomic<uint64_t> opted{0};
  auto kern = decode_split_kernel<ELEM, PAGED, D, WIDE>;
  if ((e = smem_opt_in(kern, DecCfg<D, WIDE>::SMEM, dev, opted)) != cudaSuccess) return e;
  kern<<<grid, kDecThreads, DecCfg<D, WIDE>::SMEM, st>>>(tk, tv, p);
  return cudaGetLastError();
}

template <int ELEM, int D>
cudaError_t launch_split(dim3 grid, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                         cudaStream_t st) {
  const bool wide = p.group > 8;
  if (p.page_table)
    return wide ? launch_split_instance<ELEM, true, D, true>(grid, tk, tv, p, st)
                : launch_split_instance<ELEM, true, D, false>(grid, tk, tv, p, st);
  return wide ? launch_split_instance<ELEM, false, D, true>(grid, tk, tv, p, st)
              : launch_split_instance<ELEM, false, D, false>(grid, tk, tv, p, st);
}

}  // namespace

cudaError_t launch_decode(int elem, int D, const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                          cudaStream_t st) {
  const dim3 g1(p.n_splits_max, p.Hkv, p.B);
  cudaError_t e;
  if (elem == kBF16)
    e = D == 192 ? launch_split<kBF16, 192>(g1, tk, tv, p, st) : launch_split<kBF16, 128>(g1, tk, tv, p, st);
  else
    e = D == 192 ? launch_split<kF16, 192>(g1, tk, tv, p, st) : launch_split<kF16, 128>(g1, tk, tv, p, st);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the combine's CTAs are scheduled while the split grid drains
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.Hq, p.B);
  cfg.blockDim = dim3(kDecodeDv);
  cfg.stream = st;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  e = elem == kBF16 ? cudaLaunchKernelEx(&cfg, decode_combine_kernel<kBF16>, p)
                    : cudaLaunchKernelEx(&cfg, decode_combine_kernel<kF16>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_mask_convert(const MaskConvertParams& p, cudaStream_t st) {
  const int64_t warps = (int64_t)p.B * p.Sq * ((p.n_kblocks + kMaskGroup - 1) / kMaskGroup);
  if ((warps + 3) / 4 > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  mask_convert_kernel<<<(unsigned)((warps + 3) / 4), 128, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_varlen_prep(const VarlenPrepParams& p, cudaStream_t st) {
  varlen_prep_kernel<<<1, 1024, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace sdpa
