// Fused attention prefill for sm_103a: TMA -> shared-memory ring -> tcgen05 MMAs with
// accumulators in tensor memory -> blocked online softmax -> P.V, warp-specialised.
//
// The algorithm is the blocked online softmax of the page "Xe SDPA Forward Mainloop"
// (sections "mainloop_body(K)", "softmax() helper" and "Full simplified pseudocode"):
// per K/V block, S = Q K^T accumulated over the head dim, mask, new row max, rescale of
// the running O and l, P = exp2(scale*log2(e)*S - max), l += rowsum(P), O += P V.  What is
// laid out differently for this GPU:
//   * one CTA owns two 128-row query tiles that share every K/V block; each tile has its
//     own 128-column S and O accumulators in tensor memory (4 x 128 = 512 columns);
//   * one thread issues every tcgen05.mma; the two softmax warpgroups ping-pong, so the
//     tensor core works on one tile while the other tile's softmax runs;
//   * P overwrites its own S columns in tensor memory (16-bit, packed in pairs) and feeds
//     the P.V MMA directly from there;
//   * the O rescale is lazy: the stale row max is kept until the max grows by more than
//     kRescaleLog2 (log2 units), which is exact because O and l always share the max;
//   * masking touches only the blocks that need it (the causal diagonal and the ragged
//     last block); fully hidden causal blocks are never loaded.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace sdpa {

constexpr float kRescaleLog2 = 8.0f;
// Register split (launch: 384 threads x 168): the load/MMA warpgroup gives registers to the
// two softmax warpgroups.  128 * 96 + 256 * 200 = 63488 <= 384 * 168 = 64512.  The e4m3
// kernels' softmax takes 192 (measured faster there: +1.2%; 176 +0.8%, 184 -0.2%).
constexpr uint32_t kRegsControl = 96;
constexpr uint32_t kRegsSoftmax = 200;
constexpr uint32_t kRegsSoftmaxE4m3 = 192;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kPrefillThreads * 168, "register split exceeds launch");
static_assert(kRegsSoftmaxE4m3 > 168 && kRegsSoftmaxE4m3 <= kRegsSoftmax, "e4m3 softmax registers out of range");
constexpr float kLn2 = 0.6931471805599453f;

template <int ELEM, int D, int DV>
struct PrefillCfg {
  static constexpr int ESZ = (ELEM == kE4M3) ? 1 : 2;  // Q and K element bytes
  static constexpr int CH = 64;                 // elements per swizzle chunk (TMA box width)
  static constexpr int CHB = CH * ESZ;          // 128 B (16-bit) or 64 B (e4m3)
  static constexpr uint32_t SW = (CHB == 128) ? kSwizzle128B : kSwizzle64B;
  static constexpr int NCH_D = D / CH;
  static constexpr int NCH_V = DV / 64;         // V is always 16-bit in shared memory
  // ring depth: 4 stages for D = 64, 2 otherwise; 16-bit D = 192 has room for one stage only
  // (two Q tiles of 48 KB plus one K + V stage of 80 KB), so its loads and MMAs take turns
  static constexpr int STAGES = (D <= 64) ? 4 : (ESZ == 2 && D > 128) ? 1 : 2;
  static constexpr int Q_BYTES = kBlockQ * D * ESZ;
  static constexpr int K_BYTES = kBlockK * D * ESZ;
  static constexpr int V_BYTES = kBlockK * DV * 2;
  static constexpr int VRAW_BYTES = (ELEM == kE4M3) ? kBlockK * DV : 0;
  static constexpr int KSTEP_BYTES = 32;        // K extent of one MMA: 16 x 16-bit or 32 x e4m3
  static constexpr int STEPS_PER_CH = CHB / KSTEP_BYTES;
  static constexpr int QK_STEPS = D * ESZ / KSTEP_BYTES;
  static constexpr int PV_STEPS = kBlockK / 16;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + kTilesPerCta * Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * K_BYTES;
  static constexpr int OFF_VRAW = OFF_V + STAGES * V_BYTES;
  // output staging: one 64-column box of 16-bit rows (128 x 128 B) per softmax warpgroup
  static constexpr bool TMA_EPILOGUE = true;
  static constexpr int OST_BYTES = TMA_EPILOGUE ? kBlockQ * 128 : 0;
  static constexpr int OFF_OST = OFF_VRAW + STAGES * VRAW_BYTES;
  static constexpr int OFF_BAR = OFF_OST + kTilesPerCta * OST_BYTES;
  // barriers, tmem base, abort flag; then 1 KB of slack so that the 1024-B alignment of the
  // dynamic shared window never pushes the last byte past the allocation
  static constexpr int SMEM = OFF_BAR + 512 + 1024;
  static_assert(D % CH == 0 && DV % 64 == 0, "head dims must be multiples of 64");
  static_assert(Q_BYTES % 1024 == 0 && K_BYTES % 1024 == 0 && V_BYTES % 1024 == 0, "1 KB tile alignment");
  static_assert(SMEM <= 227 * 1024, "more shared memory than a CTA may opt in to");
};

template <int ELEM>
struct ElemTraits;
template <>
struct ElemTraits<kF16> {
  static constexpr uint32_t qk_fmt = 0, pv_fmt = 0;  // f16 x f16, P f16
};
template <>
struct ElemTraits<kBF16> {
  static constexpr uint32_t qk_fmt = 1, pv_fmt = 1;  // bf16 x bf16, P bf16
};
template <>
struct ElemTraits<kE4M3> {
  static constexpr uint32_t qk_fmt = 0, pv_fmt = 0;  // e4m3 x e4m3 (kind::f8f6f4), P and V f16
};


template <int ELEM>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
  if constexpr (ELEM == kBF16)
    return pack_bf16x2(lo, hi);
  else
    return pack_f16x2(lo, hi);
}

// Output element packing (bf16 unless the inputs are f16).
template <int ELEM>
__device__ __forceinline__ uint32_t pack_out(float lo, float hi) {
  if constexpr (ELEM == kF16)
    return pack_f16x2(lo, hi);
  else
    return pack_bf16x2(lo, hi);
}

// Eight e4m3 codes (two 32-bit words) -> eight f16 values (four f16x2 words); exact.
__device__ __forceinline__ uint4 e4m3x8_to_f16x8(uint2 in) {
  uint4 out;
  asm("{\n\t.reg .b16 a, b, c, d;\n\t"
      "mov.b32 {a, b}, %4;\n\t"
      "mov.b32 {c, d}, %5;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t"
      "cvt.rn.f16x2.e4m3x2 %2, c;\n\t"
      "cvt.rn.f16x2.e4m3x2 %3, d;\n\t}"
      : "=r"(out.x), "=r"(out.y), "=r"(out.z), "=r"(out.w)
      : "r"(in.x), "r"(in.y));
  return out;
}

// One work unit: two consecutive 128-row query tiles of one (batch, query head) against the
// key blocks [jb0, jb0 + n_blocks), which is every block the tiles need unless the work tile is
// split (split >= 0: part `part` of p.split_parts key ranges of split work tile `split`).
struct WorkTile {
  int b, h, kvh, q0;
  int n_t[kTilesPerCta];  // K/V blocks each query tile needs (0 = tile entirely past Sq)
  int n_blocks;           // blocks streamed for the unit = max over its query tiles
  int jb0;                // first key block
  int split, part;        // split work tile and key range, or split = -1
  int sq, sk;             // query and key rows of the sequence
  int q_off, k_off, cb;   // TMA coordinates: first query / key row and batch index of the sequence
};

// Element offset of O row qrow of work tile w, and the index of its LSE entry.
template <bool VARLEN>
__device__ __forceinline__ int64_t o_offset(const PrefillParams& p, const WorkTile& w, int qrow) {
  if constexpr (VARLEN)
    return static_cast<int64_t>(w.q_off + qrow) * p.o_s + static_cast<int64_t>(w.h) * p.o_h;
  else
    return static_cast<int64_t>(w.b) * p.o_b + static_cast<int64_t>(qrow) * p.o_s + static_cast<int64_t>(w.h) * p.o_h;
}
template <bool VARLEN>
__device__ __forceinline__ int64_t lse_index(const PrefillParams& p, const WorkTile& w, int qrow) {
  if constexpr (VARLEN)
    return static_cast<int64_t>(w.h) * p.total_q + w.q_off + qrow;
  else
    return (static_cast<int64_t>(w.b) * p.Hq + w.h) * p.lse_ld + qrow;
}

// Work tiles in launch order.  A KV unit is one (batch, KV head): its K/V are shared by the
// Hq/Hkv query heads of the group and all their query tiles.  Units are taken in groups of
// p.units_per_group (sized on the host so that a group fills whole pairs of snake rounds and its
// K/V fits in L2), so the K/V that the CTAs running at the same time need stays resident in L2.
// Inside a group, causal tiles at the bottom of the matrix see the most keys and come first;
// tiles of one row band are ordered by unit, then query head.
// FAST: divide by the launch constants with precomputed reciprocals.  Every role decodes every
// work tile, the single MMA-issuing thread included, for which the decode is pure overhead
// between MMA groups.  The masked kernels divide plainly: with the reciprocals their softmax
// spills (measured slower there, faster on the unmasked kernels).
template <bool CAUSAL, bool VARLEN, bool FAST = true>
__device__ __forceinline__ WorkTile work_tile(const PrefillParams& p, int work_unit) {
  WorkTile w;
  w.split = -1, w.part = 0, w.jb0 = 0;
  int jb1 = p.n_kblocks;
  if constexpr (VARLEN) {
    // unit = (tile of the packed sequences) * Hq + head; a sequence's tiles run longest first
    // when causal.  Units past the last tile are empty.
    const int total_tiles = __ldg(p.tile_prefix + p.B);
    const int tg = FAST ? static_cast<int>(fast_div(static_cast<uint32_t>(work_unit), p.div_heads)) : work_unit / p.Hq;
    w.h = work_unit - tg * p.Hq;
    w.kvh = FAST ? static_cast<int>(fast_div(static_cast<uint32_t>(w.h), p.div_group)) : w.h / p.group;
    if (tg >= total_tiles) {
      w.b = 0, w.q0 = 0, w.sq = 0, w.sk = 0, w.q_off = 0, w.k_off = 0, w.cb = 0;
      w.n_t[0] = w.n_t[1] = 0;
      w.n_blocks = 0;
      return w;
    }
    int lo = 0, hi = p.B;  // tile_prefix[lo] <= tg < tile_prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.tile_prefix + mid) <= tg) lo = mid; else hi = mid;
    }
    const int first = __ldg(p.tile_prefix + lo), n_tiles = __ldg(p.tile_prefix + lo + 1) - first;
    const int local = tg - first;
    w.b = lo;
    w.q0 = (CAUSAL ? n_tiles - 1 - local : local) * kCtaRows;
    w.q_off = __ldg(p.cu_q + lo);
    w.sq = __ldg(p.cu_q + lo + 1) - w.q_off;
    w.k_off = __ldg(p.cu_k + lo);
    w.sk = __ldg(p.cu_k + lo + 1) - w.k_off;
    w.cb = 0;
    // a sequence without keys still gets one (fully masked) block: its rows come out O = 0, LSE = -inf
    jb1 = max(1, (w.sk + kBlockK - 1) / kBlockK);
  } else {
    // work units past the whole work tiles are key ranges of the split tail (never causal)
    int item = work_unit;
    if (!CAUSAL && work_unit >= p.n_full) {
      const int r = work_unit - p.n_full;
      const int parts = p.split_parts;
      w.split = r / parts;
      w.part = r - w.split * parts;
      item = p.n_full + w.split;
      w.jb0 = w.part * p.n_kblocks / parts;
      jb1 = (w.part + 1) * p.n_kblocks / parts;
    }
    const int G = p.group;                           // query heads per KV head
    const int units = p.B * p.Hkv;
    const int gsize = static_cast<int>(p.div_gsize.d);  // work tiles of a full group
    const int gi = FAST ? static_cast<int>(fast_div(static_cast<uint32_t>(item), p.div_gsize)) : item / gsize;
    const int base = gi * p.units_per_group;
    const bool last = units - base < p.units_per_group;  // the last group may hold fewer units
    FastDiv band;
    band.m = last ? p.div_band_last.m : p.div_band.m;
    band.sh1 = last ? p.div_band_last.sh1 : p.div_band.sh1;
    band.sh2 = last ? p.div_band_last.sh2 : p.div_band.sh2;
    band.d = last ? p.div_band_last.d : p.div_band.d;
    const int r = item - gi * gsize;
    // row band, longest first when causal
    const int rank = FAST ? static_cast<int>(fast_div(static_cast<uint32_t>(r), band)) : r / static_cast<int>(band.d);
    const int q = r - rank * static_cast<int>(band.d);
    const int qg = FAST ? static_cast<int>(fast_div(static_cast<uint32_t>(q), p.div_group)) : q / G;
    const int unit = base + qg;
    const int ctile = CAUSAL ? (p.n_cta_tiles - 1 - rank) : rank;
    w.b = FAST ? static_cast<int>(fast_div(static_cast<uint32_t>(unit), p.div_heads)) : unit / p.Hkv;
    w.kvh = unit - w.b * p.Hkv;
    w.h = w.kvh * G + (q - qg * G);
    w.q0 = ctile * kCtaRows;
    w.sq = p.Sq, w.sk = p.Sk;
    w.q_off = 0, w.k_off = 0, w.cb = w.b;
  }
  w.n_blocks = 0;
#pragma unroll
  for (int t = 0; t < kTilesPerCta; ++t) {
    const int r0 = w.q0 + t * kBlockQ;
    int n = 0;
    if (r0 < w.sq) {
      n = jb1 - w.jb0;
      if (CAUSAL) {
        const int last_row = min(r0 + kBlockQ - 1, w.sq - 1);
        n = min(n, (last_row + p.causal_off) / kBlockK + 1);
      }
    }
    w.n_t[t] = n;
    w.n_blocks = max(w.n_blocks, n);
  }
  return w;
}

// The k-th work unit of CTA c (snake order over the longest-first list: forward on even
// rounds, backward on odd ones, which evens out the per-CTA totals of a causal schedule).
__device__ __forceinline__ int nth_item(int k) {
  const int G = gridDim.x;
  return (k & 1) ? (k + 1) * G - 1 - (int)blockIdx.x : k * G + (int)blockIdx.x;
}

// Persistent kernel: CTA c processes work tiles nth_item(0), nth_item(1), ...  Every role walks
// the same sequence; the mbarrier phases continue from one work tile to the next, counted per
// role:
//   q_full[t]  / q_empty[t] : Q tile t landed / its last QK MMA finished (Q buffer reusable)
//   16-bit inputs, one ring whose step j holds what MMA step j reads:
//   in_full[s]              : K(j) (j < n_blocks) and V(j-1) (j >= 1) landed in stage s
//   released[s]             : every MMA that read stage s has finished (one commit per step)
//   e4m3 inputs, where V(j) must also be converted to f16 before P V(j), K(j) and V(j) load
//   together one step ahead of their P.V:
//   in_full[s] / released[s]: K(j) landed / its QK MMAs finished
//   v_full[s] / vraw_free[s]: raw V(j) landed / raw V(j) read by the converter (raw buffer free)
//   v_free[s]               : P V(j) finished (converted buffer free)
//   v_ready[s]              : V(j) converted to f16
//   s_full[t]               : S_t = Q_t K^T finished
//   p_half[t]               : keys 0-63 of P_t written to tensor memory (and O_t rescaled if needed)
//   p_full[t]               : all of P_t written
//   o_full[t]               : the last P_t V of the work tile finished (epilogue may read O_t)
// A rescale of O_t needs no barrier of its own: the commit behind s_full[t] for block j also
// covers the P_t V of block j-1, which the same thread issued earlier.
//   o_empty[t]              : the epilogue has read O_t (the next work tile may overwrite it)
template <int ELEM, int D, int DV, bool CAUSAL, bool MASK, int VAR>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const PrefillParams p) {
  using C = PrefillCfg<ELEM, D, DV>;
  constexpr bool VARLEN = VAR == kVarlen;
  constexpr bool SCALED = VAR == kBlockScaled;
  // Without a mask, tile 0's softmax waits for what the MMA thread's step j+1 reads before it
  // signals P_0(j) (16-bit: ring step j+1 landed; e4m3: V(j) converted and K(j+1) landed), which
  // spares the MMA thread those waits (with a mask the longer softmax would then hold it up)
  constexpr bool T0_COVERS_STEP = !MASK;
  constexpr bool FAST_DIV = !MASK;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sVraw = smem + C::OFF_VRAW;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;                 // [2]
  uint64_t* q_empty = q_full + 2;          // [2]
  uint64_t* in_full = q_empty + 2;         // [ST] 16-bit: K(j) + V(j-1); e4m3: K(j)
  uint64_t* released = in_full + ST;       // [ST] 16-bit: stage free; e4m3: K stage free
  uint64_t* v_full = released + ST;        // [ST] e4m3: raw V(j) landed
  uint64_t* v_free = v_full + ST;          // [ST] e4m3: V stage (raw and converted) free
  uint64_t* v_ready = v_free + ST;         // [ST] e4m3: V(j) converted to f16
  uint64_t* vraw_free = v_ready + ST;      // [ST] e4m3: raw V(j) converted (raw buffer free)
  uint64_t* s_full = vraw_free + ST;       // [2]
  uint64_t* p_full = s_full + 2;           // [2]
  uint64_t* o_full = p_full + 2;           // [2]
  uint64_t* o_empty = o_full + 2;          // [2]
  uint64_t* mma_done = o_empty + 2;        // [1]
  uint64_t* p_half = mma_done + 1;         // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(p_half + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int n_items = p.n_units;
  // the split merge, if any, may be scheduled early (it waits for this grid's completion)
  if constexpr (!CAUSAL && !VARLEN) pdl_launch_dependents();

  if (tid == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&q_empty[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
      mbar_init(&p_half[t], 128);
      mbar_init(&o_full[t], 1);
      mbar_init(&o_empty[t], 128);
    }
    for (int s = 0; s < ST; ++s) {
      mbar_init(&in_full[s], 1);
      mbar_init(&released[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_free[s], 1);
      mbar_init(&v_ready[s], 64);
      mbar_init(&vraw_free[s], 64);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    regs_dec<kRegsControl>();
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int qn[2] = {0, 0};  // Q loads issued per tile slot
      int g = 0;           // ring steps issued
      bool ok = true;
      for (int k = 0, item = nth_item(0); ok && item < n_items; item = nth_item(++k)) {
        const WorkTile w = work_tile<CAUSAL, VARLEN, FAST_DIV>(p, item);
        if (VARLEN && w.n_blocks == 0) continue;  // an empty unit (past the packed sequences' tiles)
        for (int t = 0; t < kTilesPerCta && ok; ++t) {
          if (w.n_t[t] == 0) continue;
          if (qn[t] > 0 && !mbar_wait(&q_empty[t], (qn[t] - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&q_full[t], C::Q_BYTES);
          for (int c = 0; c < C::NCH_D; ++c)
            tma_load_4d(sQ + t * C::Q_BYTES + c * kBlockQ * C::CHB, &tm_q, &q_full[t], c * C::CH, w.h,
                        w.q_off + w.q0 + t * kBlockQ, w.cb);
          ++qn[t];
        }
        if constexpr (ELEM == kE4M3) {
          // step j brings K(j) and raw V(j)
          for (int j = 0; ok && j < w.n_blocks; ++j, ++g) {
            const int s = g % ST, r = g / ST;
            if (r > 0 && !mbar_wait(&released[s], (r - 1) & 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            if (p.stall_first_stage && g == 0) continue;  // test hook: stage 0 never fills
            mbar_arrive_expect_tx(&in_full[s], C::K_BYTES);
            for (int c = 0; c < C::NCH_D; ++c)
              tma_load_4d(sK + s * C::K_BYTES + c * kBlockK * C::CHB, &tm_k, &in_full[s], c * C::CH, w.kvh,
                          w.k_off + (w.jb0 + j) * kBlockK, w.cb);
            // the raw buffer frees as soon as the converter has read it
            if (r > 0 && !mbar_wait(&vraw_free[s], (r - 1) & 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&v_full[s], C::VRAW_BYTES);
            tma_load_4d(sVraw + s * C::VRAW_BYTES, &tm_v, &v_full[s], 0, w.kvh, w.k_off + (w.jb0 + j) * kBlockK,
                        w.cb);
          }
        } else {
          // step j of the work tile brings K(j) and V(j-1)
          for (int j = 0; ok && j <= w.n_blocks; ++j, ++g) {
            const int s = g % ST, r = g / ST;
            const bool has_k = j < w.n_blocks, has_v = j >= 1;
            if (r > 0 && !mbar_wait(&released[s], (r - 1) & 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            if (p.stall_first_stage && g == 0) continue;  // test hook: stage 0 never fills
            mbar_arrive_expect_tx(&in_full[s], (has_k ? C::K_BYTES : 0) + (has_v ? C::V_BYTES : 0));
            if (has_k) {
              for (int c = 0; c < C::NCH_D; ++c)
                tma_load_4d(sK + s * C::K_BYTES + c * kBlockK * C::CHB, &tm_k, &in_full[s], c * C::CH, w.kvh,
                            w.k_off + (w.jb0 + j) * kBlockK, w.cb);
            }
            if (has_v) {
              for (int c = 0; c < C::NCH_V; ++c)
                tma_load_4d(sV + s * C::V_BYTES + c * kBlockK * 128, &tm_v, &in_full[s], c * 64, w.kvh,
                            w.k_off + (w.jb0 + j - 1) * kBlockK, w.cb);
            }
          }
        }
      }
      if (!ok) {
        // let every copy already in flight land before the CTA's shared memory goes away
        for (int t = 0; t < kTilesPerCta; ++t)
          if (qn[t] > 0) mbar_drain(&q_full[t], (qn[t] - 1) & 1);
        for (int j = max(0, g - ST); j < g; ++j) {
          mbar_drain(&in_full[j % ST], (j / ST) & 1);
          if (ELEM == kE4M3) mbar_drain(&v_full[j % ST], (j / ST) & 1);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (one thread)
    regs_dec<kRegsControl>();
    if (lane == 0) {
      constexpr uint32_t idesc_qk =
          make_idesc(ElemTraits<ELEM>::qk_fmt, ElemTraits<ELEM>::qk_fmt, 0, 0, kBlockQ, kBlockK);
      constexpr uint32_t idesc_pv = make_idesc(ElemTraits<ELEM>::pv_fmt, ElemTraits<ELEM>::pv_fmt, 0, 1, kBlockQ, DV);
      // Descriptors are built once; a k-step or stage only moves the start address, whose
      // field holds (address >> 4) in the low 14 bits of the low word.  For shared addresses
      // below 256 KB an add of (offset >> 4) to the low word is exact and never carries out
      // of the field, so the high words stay fixed.
      const uint64_t dq0 = make_smem_desc(smem_u32(sQ), 16, 8 * C::CHB, C::SW);
      const uint64_t dk0 = make_smem_desc(smem_u32(sK), 16, 8 * C::CHB, C::SW);
      const uint64_t dv0 = make_smem_desc(smem_u32(sV), kBlockK * 128, 1024, kSwizzle128B);
      const uint32_t q_lo = static_cast<uint32_t>(dq0), q_hi = static_cast<uint32_t>(dq0 >> 32);
      const uint32_t k_lo = static_cast<uint32_t>(dk0), k_hi = static_cast<uint32_t>(dk0 >> 32);
      const uint32_t v_lo = static_cast<uint32_t>(dv0), v_hi = static_cast<uint32_t>(dv0 >> 32);
      int qn[2] = {0, 0};   // work tiles seen per tile slot (q_full / q_empty / o_full / o_empty phases)
      int pn[2] = {0, 0};   // P.V blocks issued per tile slot (p_full phases)
      int g = 0;            // ring steps consumed
      bool ok = true;
      for (int k = 0, item = nth_item(0); ok && item < n_items; item = nth_item(++k)) {
        const WorkTile w = work_tile<CAUSAL, VARLEN, FAST_DIV>(p, item);
        if (VARLEN && w.n_blocks == 0) continue;  // an empty unit: skipped by every role
        for (int t = 0; t < kTilesPerCta && ok; ++t)
          if (w.n_t[t] > 0) ok = mbar_wait(&q_full[t], qn[t] & 1, abort_flag, p.status);
        // Ring block of step j: e4m3 uses block g + j for K(j) and g + j - 1 for V(j-1); the
        // 16-bit ring holds both operands of step j in one stage.
        for (int j = 0; ok && j <= w.n_blocks; ++j) {
          // Steady steps 2 <= j < min(n_t) - 1: both tiles take P.V of block j - 1 (neither the
          // first nor the last of the tile) and QK of block j (not the last), so no o_empty wait,
          // o_full or q_empty commit is due.  The same waits and commits as the general step
          // below, in the same order, without its per-step case analysis: every instruction the
          // issuing thread spends between MMA groups can leave the tensor pipe idle.
          if (j == 2) {
            const int j_end = min(w.n_t[0], w.n_t[1]) - 1;
            for (; j < j_end; ++j) {
              const int gk = (ELEM == kE4M3) ? g + j : g;      // stage of K(j)
              const int gv = (ELEM == kE4M3) ? g + j - 1 : g;  // stage of V(j-1)
              const int s = gk % ST, sv = gv % ST;
              bool k_ready = ELEM != kE4M3 || T0_COVERS_STEP;
              if constexpr (!T0_COVERS_STEP) {
                if (!mbar_wait(ELEM == kE4M3 ? &v_ready[sv] : &in_full[s], ((ELEM == kE4M3 ? gv : gk) / ST) & 1,
                               abort_flag, p.status)) {
                  ok = false;
                  break;
                }
              }
              tc_fence_after();
              const uint32_t dv = v_lo + static_cast<uint32_t>((sv * C::V_BYTES) >> 4);
              const uint32_t dk = k_lo + static_cast<uint32_t>((s * C::K_BYTES) >> 4);
#pragma unroll
              for (int t = 0; t < kTilesPerCta; ++t) {
                const uint32_t tS = tmem_base + t * 128;
                const uint32_t tO = tmem_base + 256 + t * 128;
                // P.V in two halves: keys 0-63 as soon as the softmax has written them
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  if (!mbar_wait(h == 0 ? &p_half[t] : &p_full[t], pn[t] & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                  }
                  tc_fence_after();
#pragma unroll
                  for (int kk = h * C::PV_STEPS / 2; kk < (h + 1) * C::PV_STEPS / 2; ++kk)
                    mma_f16_ts(tO, tS + kk * 8, dv + static_cast<uint32_t>((kk * 16 * 128) >> 4), v_hi, idesc_pv, 1u);
                }
                if (!ok) break;
                ++pn[t];
                if (ELEM == kE4M3 && t == kTilesPerCta - 1) mma_commit(&v_free[sv]);
                if (!k_ready) {
                  if (!mbar_wait(&in_full[s], (gk / ST) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                  }
                  tc_fence_after();
                  k_ready = true;
                }
                const uint32_t dq = q_lo + static_cast<uint32_t>((t * C::Q_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < C::QK_STEPS; ++kk) {
                  constexpr int kCh = kBlockQ * C::CHB;
                  const uint32_t off = static_cast<uint32_t>(
                      ((kk / C::STEPS_PER_CH) * kCh + (kk % C::STEPS_PER_CH) * C::KSTEP_BYTES) >> 4);
                  if constexpr (ELEM == kE4M3)
                    mma_f8_ss(tS, dq + off, q_hi, dk + off, k_hi, idesc_qk, kk > 0 ? 1u : 0u);
                  else
                    mma_f16_ss(tS, dq + off, q_hi, dk + off, k_hi, idesc_qk, kk > 0 ? 1u : 0u);
                }
                mma_commit(&s_full[t]);
              }
              if (!ok) break;
              mma_commit(&released[s]);
              if (ELEM != kE4M3) ++g;
            }
            if (!ok) break;
          }
          const int gk = (ELEM == kE4M3) ? g + j : g;            // stage of K(j)
          const int gv = (ELEM == kE4M3) ? g + j - 1 : g;        // stage of V(j-1)
          const int s = gk % ST, r = gk / ST;
          const int sv = gv % ST, rv = gv / ST;
          // e4m3: K(j) is waited for just before the first QK, unless tile 0's softmax covered it
          const bool covered = T0_COVERS_STEP && j >= 1 && j - 1 < w.n_t[0];
          bool k_ready = ELEM != kE4M3 || covered;
          if constexpr (ELEM == kE4M3) {
            if (j >= 1 && !covered && !mbar_wait(&v_ready[sv], rv & 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
          } else {
            // A step that starts with P_0(j-1) V(j-1) needs no wait of its own: tile 0's softmax
            // saw this stage land before it signalled P_0(j-1).
            if (!covered && !mbar_wait(&in_full[s], r & 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          for (int t = 0; t < kTilesPerCta; ++t) {
            const uint32_t tS = tmem_base + t * 128;
            const uint32_t tO = tmem_base + 256 + t * 128;
            // O_t += P_t(j-1) V(j-1), with P read from tensor memory
            if (j >= 1 && j - 1 < w.n_t[t]) {
              // the first P.V of a work tile overwrites O_t: the previous epilogue must be done
              if (j == 1 && qn[t] > 0 && !mbar_wait(&o_empty[t], (qn[t] - 1) & 1, abort_flag, p.status)) {
                ok = false;
                break;
              }
              const uint32_t dv = v_lo + static_cast<uint32_t>((sv * C::V_BYTES) >> 4);
              const uint32_t acc0 = (j - 1 > 0) ? 1u : 0u;
              // P.V in two halves: keys 0-63 as soon as the softmax has written them
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                if (!mbar_wait(h == 0 ? &p_half[t] : &p_full[t], pn[t] & 1, abort_flag, p.status)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = h * C::PV_STEPS / 2; kk < (h + 1) * C::PV_STEPS / 2; ++kk)
                  mma_f16_ts(tO, tS + kk * 8, dv + static_cast<uint32_t>((kk * 16 * 128) >> 4), v_hi, idesc_pv,
                             kk > 0 ? 1u : acc0);
              }
              if (!ok) break;
              if (j == w.n_t[t]) mma_commit(&o_full[t]);  // O_t of this work tile complete
              ++pn[t];
            }
            // e4m3: the V stage of block j-1 is free once both P.V MMAs of this step complete
            if (ELEM == kE4M3 && t == kTilesPerCta - 1 && j >= 1) mma_commit(&v_free[sv]);
            // S_t = Q_t K(j)^T
            if (j < w.n_t[t]) {
              if (!k_ready) {
                if (!mbar_wait(&in_full[s], r & 1, abort_flag, p.status)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                k_ready = true;
              }
              const uint32_t dq = q_lo + static_cast<uint32_t>((t * C::Q_BYTES) >> 4);
              const uint32_t dk = k_lo + static_cast<uint32_t>((s * C::K_BYTES) >> 4);
#pragma unroll
              for (int kk = 0; kk < C::QK_STEPS; ++kk) {
                constexpr int kCh = kBlockQ * C::CHB;  // bytes per 64-element chunk (Q and K tiles alike)
                const uint32_t off =
                    static_cast<uint32_t>(((kk / C::STEPS_PER_CH) * kCh + (kk % C::STEPS_PER_CH) * C::KSTEP_BYTES) >> 4);
                if constexpr (ELEM == kE4M3)
                  mma_f8_ss(tS, dq + off, q_hi, dk + off, k_hi, idesc_qk, kk > 0 ? 1u : 0u);
                else
                  mma_f16_ss(tS, dq + off, q_hi, dk + off, k_hi, idesc_qk, kk > 0 ? 1u : 0u);
              }
              mma_commit(&s_full[t]);
              if (j == w.n_t[t] - 1) mma_commit(&q_empty[t]);  // Q_t of this work tile fully used
            }
          }
          if constexpr (ELEM == kE4M3) {
            if (ok && j < w.n_blocks) mma_commit(&released[s]);  // K(j) free once its QKs complete
          } else {
            // everything this step read from ring stage s is free once these MMAs complete
            if (ok) mma_commit(&released[s]);
            ++g;
          }
        }
        if (ELEM == kE4M3) g += w.n_blocks;
        for (int t = 0; t < kTilesPerCta; ++t)
          if (w.n_t[t] > 0) ++qn[t];
      }
      // every MMA issued so far has finished before tensor memory is released
      mma_commit(mma_done);
      mbar_drain(mma_done, 0);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ e4m3 V -> f16 converter
    regs_dec<kRegsControl>();
    if constexpr (ELEM == kE4M3) {
      const int ct = tid - 64;  // 0..63
      int g = 0;
      bool ok = true;
      for (int k = 0, item = nth_item(0); ok && item < n_items; item = nth_item(++k)) {
        const WorkTile w = work_tile<CAUSAL, VARLEN, FAST_DIV>(p, item);
        for (int j = 0; j < w.n_blocks; ++j, ++g) {
          const int s = g % ST, r = g / ST;
          if (!mbar_wait(&v_full[s], r & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          // the converted buffer of this stage is free once the previous P.V that read it finished
          if (r > 0 && !mbar_wait(&v_free[s], (r - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint8_t* src = sVraw + s * C::VRAW_BYTES;
          uint8_t* dst = sV + s * C::V_BYTES;
          constexpr int UNITS = kBlockK * DV / 8;  // 8 values per unit
#pragma unroll 4
          for (int u = ct; u < UNITS; u += 64) {
            const int row = u / (DV / 8), du = u % (DV / 8);
            const int ch = du >> 3, uc = du & 7;
            const uint2 raw = *reinterpret_cast<const uint2*>(src + row * DV + du * 8);
            *reinterpret_cast<uint4*>(dst + ch * kBlockK * 128 + row * 128 + ((uc ^ (row & 7)) << 4)) =
                e4m3x8_to_f16x8(raw);
          }
          fence_proxy_async_smem();
          mbar_arrive(&v_ready[s]);
          mbar_arrive(&vraw_free[s]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    regs_inc<ELEM == kE4M3 ? kRegsSoftmaxE4m3 : kRegsSoftmax>();
    if constexpr (MASK) pdl_wait();  // the condensed mask comes from the kernel launched before
    const int t = (warp - 4) >> 2;           // query tile slot of this warpgroup
    const int wq = warp & 3;                 // tensor-memory lane quarter
    const int row = wq * 32 + lane;          // row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem_base + lane_off + t * 128;
    const uint32_t tO = tmem_base + lane_off + 256 + t * 128;
    const bool wg_leader = wq == 0 && lane == 0;  // issues this warpgroup's output stores
    const float scale2 = p.scale2;
    int sn = 0;     // S blocks consumed (s_full / p_full phases)
    int on = 0;     // work tiles finished (o_full phases)
    int gbase = 0;  // ring index of the current work tile's first step (tile 0 uses it)
    bool ok = true;
    for (int k = 0, item = nth_item(0); ok && item < n_items; item = nth_item(++k)) {
      const WorkTile w = work_tile<CAUSAL, VARLEN, FAST_DIV>(p, item);
      const int g0 = gbase;
      // every role skips empty units; the 16-bit ring takes n_blocks + 1 steps, e4m3 n_blocks
      gbase += w.n_blocks > 0 ? w.n_blocks + (ELEM == kE4M3 ? 0 : 1) : 0;
      const int n = w.n_t[t];
      if (n == 0) continue;
      const int qrow = w.q0 + t * kBlockQ + row;
      const bool row_valid = qrow < w.sq;
      // int8 codes: this tile's Q block scale folded into the exp2 scale; K block scales per block
      float tile_scale2 = scale2;
      const float* ks_row = nullptr;
      if constexpr (SCALED) {
        tile_scale2 = scale2 * __ldg(p.q_scale + (static_cast<int64_t>(w.b) * p.Hq + w.h) * p.n_qblocks +
                                     (w.q0 + t * kBlockQ) / kBlockQ);
        ks_row = p.k_scale + (static_cast<int64_t>(w.b) * p.Hkv + w.kvh) * p.n_kblocks + w.jb0;
      }
      float m_used = -INFINITY;
      float l = 0.f;
      const uint4* bits_row = nullptr;
      const uint8_t* flags_row = nullptr;
      if constexpr (MASK) {
        const int qr = row_valid ? qrow : 0;
        bits_row = p.mask_bits + (static_cast<int64_t>(w.b) * p.Sq + qr) * p.n_kblocks;
        flags_row = p.mask_flags + (static_cast<int64_t>(w.b) * p.Sq + qr) * p.n_kblocks;
      }

      for (int j = 0; j < n; ++j, ++sn) {
        float blk_scale2 = tile_scale2;  // exp2 units per unit of s in this block
        if constexpr (SCALED) blk_scale2 = tile_scale2 * __ldg(ks_row + j);
        uint4 mbits = make_uint4(0u, 0u, 0u, 0u);
        uint32_t mflag = 0;
        if constexpr (MASK) {
          if (row_valid) {
            mbits = __ldg(bits_row + w.jb0 + j);
            mflag = __ldg(flags_row + w.jb0 + j);
          }
        }
        if (!mbar_wait_warp(&s_full[t], sn & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[kBlockK];
        {
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tmem_ld32(tS + 0, r0);
          tmem_ld32(tS + 32, r1);
          tmem_ld32(tS + 64, r2);
          tmem_ld32(tS + 96, r3);
          tmem_ld_wait();
          reg_fence(r0);
          reg_fence(r1);
          reg_fence(r2);
          reg_fence(r3);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            s[c] = __uint_as_float(r0[c]);
            s[32 + c] = __uint_as_float(r1[c]);
            s[64 + c] = __uint_as_float(r2[c]);
            s[96 + c] = __uint_as_float(r3[c]);
          }
        }
        // the causal diagonal and the ragged last block: hide keys past the row / past Sk
        const int k0 = (w.jb0 + j) * kBlockK;
        const bool edge = (CAUSAL && (k0 + kBlockK - 1 > w.q0 + t * kBlockQ + p.causal_off)) || (k0 + kBlockK > w.sk);
        if (edge) {
          const int lim = (CAUSAL ? min(w.sk, qrow + p.causal_off + 1) : w.sk) - k0;
#pragma unroll
          for (int c = 0; c < kBlockK; ++c)
            if (c >= lim) s[c] = -INFINITY;
        }
        if constexpr (MASK) {
          if (mflag) {
            // block row with finite non-zero mask values: add them (rare path)
            const uint16_t* mrow =
                p.mask + static_cast<int64_t>(w.b) * p.mask_b + static_cast<int64_t>(qrow) * p.mask_i;
#pragma unroll
            for (int c = 0; c < kBlockK; ++c) {
              if (k0 + c < w.sk) {
                const float mv = __half2float(__ushort_as_half(__ldg(mrow + k0 + c)));
                s[c] += mv * p.inv_scale;
              }
            }
          }
          __syncwarp();
          const uint32_t mw[4] = {mbits.x, mbits.y, mbits.z, mbits.w};
#pragma unroll
          for (int c = 0; c < kBlockK; ++c)
            if ((mw[c >> 5] >> (c & 31)) & 1u) s[c] = -INFINITY;
        }
        // block row max (blk_scale2 > 0, so the max of s orders like the max of blk_scale2 * s)
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[i], s[8 + i]);
#pragma unroll
        for (int gi = 1; gi < kBlockK / 16; ++gi)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[16 * gi + i], s[16 * gi + 8 + i]);
        const float mb = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        const float m_cand = fmaxf(m_used, mb * blk_scale2);
        const bool need = m_cand > m_used + kRescaleLog2;
        const bool rescale = __any_sync(0xffffffffu, need);
        float alpha = 1.f;
        if (rescale) {
          alpha = (m_cand == -INFINITY) ? 1.f : ex2(m_used - m_cand);
          l *= alpha;
          m_used = m_cand;
        }
        // P = exp2(blk_scale2 * s - m), rounded to 16 bits for the P.V product; l sums the fp32
        // values, two at a time by one packed add (one instruction a pair, against two for
        // sums of the rounded values).  P goes to tensor memory in two halves of 64 keys, each
        // signalled as soon as it is written (p_half, then p_full), so that the MMA thread
        // starts P.V on the first half while the second is computed.
        const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int w2 = 0; w2 < 32; ++w2) {
            const int c = half * 64 + 2 * w2;
            float x0, x1;
            ffma2_scalar(x0, x1, s[c], s[c + 1], blk_scale2, neg_m);
            const float p0 = ex2(x0), p1 = ex2(x1);
            pk[w2] = pack_p<ELEM>(p0, p1);
            if (w2 & 1)
              fadd2(ls[2], ls[3], p0, p1);
            else
              fadd2(ls[0], ls[1], p0, p1);
          }
          tmem_st32(tS + half * 32, pk);
          if (half == 1) break;
          if (rescale && j > 0) {
            // O holds P.V of blocks < j at the old max (finished: s_full(j) covers it); scale it
            // before the first P.V of block j
#pragma unroll 1
            for (int c = 0; c < DV / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_ld_wait();
              reg_fence(o);
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                float a = __uint_as_float(o[i]), b = __uint_as_float(o[i + 1]);
                fmul2_scalar(a, b, alpha);
                o[i] = __float_as_uint(a);
                o[i + 1] = __float_as_uint(b);
              }
              tmem_st32(tO + c * 32, o);
            }
          }
          // P_0(j) also stands for what the MMA thread's step j+1 reads (V(j) among it, which the
          // first half of P_0(j) V(j) already reads), so it skips its own waits at that step.
          // Tile 0 is active in every work tile, and the MMA thread waits for itself at every
          // step tile 0 does not cover, so these waits never fall two phases behind.
          if (T0_COVERS_STEP && t == 0) {
            if constexpr (ELEM == kE4M3) {
              const int gv = g0 + j;  // V(j) converted; K(j+1) landed when there is a block j+1
              if (!mbar_wait_warp(&v_ready[gv % ST], (gv / ST) & 1, abort_flag, p.status) ||
                  (j + 1 < w.n_blocks &&
                   !mbar_wait_warp(&in_full[(gv + 1) % ST], ((gv + 1) / ST) & 1, abort_flag, p.status))) {
                ok = false;
                break;
              }
            } else {
              const int g_next = g0 + j + 1;
              if (!mbar_wait_warp(&in_full[g_next % ST], (g_next / ST) & 1, abort_flag, p.status)) {
                ok = false;
                break;
              }
            }
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&p_half[t]);
        }
        if (!ok) break;
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[t]);
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue: O / l, LSE
      if (!mbar_wait_warp(&o_full[t], on & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      ++on;
      tc_fence_after();
      uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) + 2 * o_offset<VARLEN>(p, w, qrow);
      float* lse_out = p.lse ? p.lse + lse_index<VARLEN>(p, w, qrow) : nullptr;
      if (w.split >= 0) {
        // one key range of a split work tile: store this part's unnormalised O row, row max
        // and row sum for split_combine_kernel
        const int prow = t * kBlockQ + row;
        const size_t slot = (static_cast<size_t>(w.split) * p.split_parts + w.part) * kCtaRows + prow;
        float* po = p.split_o + slot * DV;
#pragma unroll 1
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait();
          reg_fence(o);
          if (row_valid) {
            uint4* dst = reinterpret_cast<uint4*>(po + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          }
          __syncwarp();
        }
        tc_fence_before();
        mbar_arrive(&o_empty[t]);
        if (row_valid) *reinterpret_cast<float2*>(p.split_ml + slot * 2) = make_float2(m_used, l);
        continue;
      }
      const float inv = (l > 0.f) ? p.out_scale / l : 0.f;
      const float* vs_row = nullptr;  // int8 V codes: per-channel scales
      if constexpr (SCALED)
        if (p.v_scale != nullptr) vs_row = p.v_scale + (static_cast<int64_t>(w.b) * p.Hkv + w.kvh) * DV;
      if constexpr (!VARLEN && C::TMA_EPILOGUE) {
        // O leaves through shared memory: each 64-column half of the tile goes to this
        // warpgroup's staging box (128-byte swizzle, conflict-free rows) and out by one TMA store,
        // which writes whole rows of global memory (rows past Sq clipped) and runs on while the
        // warpgroup starts its next work tile.  A thread storing its own row straight from
        // registers writes 16-byte pieces of 32 rows per instruction instead.
        uint8_t* ost = smem + C::OFF_OST + t * C::OST_BYTES;
#pragma unroll 1
        for (int hb = 0; hb < DV / 64; ++hb) {
          // the staging box is free once the previous store from it has read it
          if (wg_leader) bulk_wait_read_all();
          named_barrier_sync(1 + t, 128);
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * hb + cc;
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait();
            reg_fence(o);
            if constexpr (SCALED) {
              if (vs_row != nullptr) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float4 f = __ldg(reinterpret_cast<const float4*>(vs_row + c * 32) + i);
                  o[4 * i] = __float_as_uint(__uint_as_float(o[4 * i]) * f.x);
                  o[4 * i + 1] = __float_as_uint(__uint_as_float(o[4 * i + 1]) * f.y);
                  o[4 * i + 2] = __float_as_uint(__uint_as_float(o[4 * i + 2]) * f.z);
                  o[4 * i + 3] = __float_as_uint(__uint_as_float(o[4 * i + 3]) * f.w);
                }
              }
            }
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_out<ELEM>(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              *reinterpret_cast<uint4*>(ost + row * 128 + (((4 * cc + i) ^ (row & 7)) << 4)) =
                  make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
          fence_proxy_async_smem();
          named_barrier_sync(1 + t, 128);
          if (wg_leader) {
            tma_store_4d(&tm_o, ost, hb * 64, w.h, w.q_off + w.q0 + t * kBlockQ, w.cb);
            bulk_commit_group();
          }
        }
      } else {
        // packed sequences (a tile's rows past its sequence belong to the next one) and the e4m3
        // kernels: each thread stores its own row
#pragma unroll 1
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait();
          reg_fence(o);
          if constexpr (SCALED) {
            if (vs_row != nullptr) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 f = __ldg(reinterpret_cast<const float4*>(vs_row + c * 32) + i);
                o[4 * i] = __float_as_uint(__uint_as_float(o[4 * i]) * f.x);
                o[4 * i + 1] = __float_as_uint(__uint_as_float(o[4 * i + 1]) * f.y);
                o[4 * i + 2] = __float_as_uint(__uint_as_float(o[4 * i + 2]) * f.z);
                o[4 * i + 3] = __float_as_uint(__uint_as_float(o[4 * i + 3]) * f.w);
              }
            }
          }
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_out<ELEM>(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
          if (row_valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 64);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
          __syncwarp();
        }
      }
      // O_t has been read: the next work tile's first P.V may overwrite it
      tc_fence_before();
      mbar_arrive(&o_empty[t]);
      if (lse_out != nullptr && row_valid) *lse_out = (l > 0.f) ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
    }
    // the shared-memory staging must outlive every output store issued from it
    if (wg_leader) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// Merges the split_parts partial results of every row of the split work tiles and writes the
// normalised O and LSE (runs after prefill_kernel in the same stream).  One thread per (split
// tile, row, 8 output columns):
//   M = max_q m_q,  w_q = 2^(m_q - M),  O = sum_q w_q O_q / sum_q w_q l_q,  LSE = (M + log2 L) ln 2,
// parts taken in order, so the result does not depend on which part finished first.
template <int ELEM, int DV>
__global__ void __launch_bounds__(128) split_combine_kernel(const PrefillParams p) {
  constexpr int kChunks = DV / 8;
  pdl_wait();  // the partials come from the prefill launched before
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(p.split_tail) * kCtaRows * kChunks) return;
  const int chunk = static_cast<int>(idx % kChunks);
  const int prow = static_cast<int>((idx / kChunks) % kCtaRows);
  const int split = static_cast<int>(idx / (static_cast<long long>(kChunks) * kCtaRows));
  const int P = p.split_parts;
  const WorkTile w = work_tile<false, false>(p, p.n_full + split * P);
  const int qrow = w.q0 + prow;
  if (qrow >= w.sq) return;
  const size_t slot0 = static_cast<size_t>(split) * P * kCtaRows + prow;
  float m[kMaxSplitParts], l[kMaxSplitParts];
  float M = -INFINITY;
#pragma unroll
  for (int q = 0; q < kMaxSplitParts; ++q) {
    if (q < P) {
      const float2 ml = *reinterpret_cast<const float2*>(p.split_ml + (slot0 + static_cast<size_t>(q) * kCtaRows) * 2);
      m[q] = ml.x, l[q] = ml.y;
    } else {
      m[q] = -INFINITY, l[q] = 0.f;
    }
    M = fmaxf(M, m[q]);
  }
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float L = 0.f;
#pragma unroll
  for (int q = 0; q < kMaxSplitParts; ++q) {
    if (q < P) {
      const float wq = (m[q] == -INFINITY) ? 0.f : ex2(m[q] - M);
      L += wq * l[q];
      const float4* src = reinterpret_cast<const float4*>(p.split_o + (slot0 + static_cast<size_t>(q) * kCtaRows) * DV) + 2 * chunk;
      const float4 a = src[0], b = src[1];
      acc[0] += wq * a.x, acc[1] += wq * a.y, acc[2] += wq * a.z, acc[3] += wq * a.w;
      acc[4] += wq * b.x, acc[5] += wq * b.y, acc[6] += wq * b.z, acc[7] += wq * b.w;
    }
  }
  if (p.v_scale != nullptr) {  // int8 V codes: per-channel scales (set only for int8 inputs)
    const float4* vs = reinterpret_cast<const float4*>(p.v_scale + (static_cast<int64_t>(w.b) * p.Hkv + w.kvh) * DV) +
                       2 * chunk;
    const float4 a = __ldg(vs), b = __ldg(vs + 1);
    acc[0] *= a.x, acc[1] *= a.y, acc[2] *= a.z, acc[3] *= a.w;
    acc[4] *= b.x, acc[5] *= b.y, acc[6] *= b.z, acc[7] *= b.w;
  }
  const float inv = (L > 0.f) ? p.out_scale / L : 0.f;
  uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) + 2 * o_offset<false>(p, w, qrow);
  *reinterpret_cast<uint4*>(orow + chunk * 16) =
      make_uint4(pack_out<ELEM>(acc[0] * inv, acc[1] * inv), pack_out<ELEM>(acc[2] * inv, acc[3] * inv),
                 pack_out<ELEM>(acc[4] * inv, acc[5] * inv), pack_out<ELEM>(acc[6] * inv, acc[7] * inv));
  if (chunk == 0 && p.lse != nullptr)
    p.lse[lse_index<false>(p, w, qrow)] = (L > 0.f) ? (M + __log2f(L)) * kLn2 : -INFINITY;
}

}  // namespace sdpa
