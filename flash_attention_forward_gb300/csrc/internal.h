// Host/device parameter blocks and the launch functions each kernel file exports to the
// C-ABI layer.  Internal: not part of the public header.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sdpa {

// Status bits a kernel ORs into the device status word.
enum : uint32_t { kStatusTimeout = 1u, kStatusBadSeqlens = 2u };

// Prefill tile geometry shared by host and device.
constexpr int kBlockQ = 128;           // query rows per tile (one TMEM lane each)
constexpr int kTilesPerCta = 2;        // two query tiles per CTA share every K/V block
constexpr int kCtaRows = kBlockQ * kTilesPerCta;
constexpr int kBlockK = 128;           // keys per K/V block
static_assert(kBlockQ == kBlockK, "Q and K tiles share the descriptor chunk stride");
constexpr int kPrefillThreads = 384;   // 12 warps: load, MMA, 2 helpers, 2 x 4 softmax

enum ElemKind : int { kF16 = 0, kBF16 = 1, kE4M3 = 2 };

// Prefill kernel variants: a dense batch, packed variable-length sequences, or int8 codes widened
// to 16 bits whose scores are scaled per (128-row Q block, 128-key K block) and whose O columns
// may be scaled per channel.
enum PrefillVariant : int { kDense = 0, kVarlen = 1, kBlockScaled = 2 };

// Division by a launch constant d >= 1 with one multiply-high, two adds and two shifts, exact
// for every 32-bit numerator (the unsigned scheme of Granlund and Montgomery, "Division by
// Invariant Integers using Multiplication", 1994, figure 4.1): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, t = umulhi(m, n) and n / d = (t + ((n - t) >> min(l, 1)))
// >> max(l - 1, 0).  The work-tile decode runs on the single MMA-issuing thread and on every
// softmax warp at each new work tile, where a general integer division costs tens of
// instructions; 32-bit arithmetic keeps it from holding register pairs.
struct FastDiv {
  uint32_t m = 1, sh1 = 0, sh2 = 0;
  uint32_t d = 1;
};
inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  uint32_t l = 0;
  while ((uint64_t(1) << l) < d) ++l;  // l <= 31 for d < 2^31
  f.m = static_cast<uint32_t>(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
  f.sh1 = l < 1 ? l : 1;
  f.sh2 = l > 1 ? l - 1 : 0;
  f.d = d;
  return f;
}
#ifdef __CUDACC__
__host__ __device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
#ifdef __CUDA_ARCH__
  const uint32_t t = __umulhi(f.m, n);
#else
  const uint32_t t = static_cast<uint32_t>((static_cast<uint64_t>(f.m) * n) >> 32);
#endif
  return (t + ((n - t) >> f.sh1)) >> f.sh2;
}
#endif

struct PrefillParams {
  void* o;                 // [B, Sq, Hq, Dv] out dtype
  float* lse;              // [B, Hq, Sq] or null
  int64_t o_b, o_s, o_h;   // element strides of o
  int B, Hq, Hkv, Sq, Sk;
  int causal_off;          // causal: key j visible to query row i iff j <= i + causal_off (top-left: 0)
  int64_t lse_ld;          // dense LSE layout [B, Hq, lse_ld] (lse_ld >= Sq)
  int group;               // Hq / Hkv
  int n_cta_tiles;         // ceil(Sq / kCtaRows)
  int units_per_group;     // KV units (batch x KV head) whose work tiles are scheduled together
  // divisors of the work-tile decode: a full group's work tiles, a row band of a full group and of
  // the last group, the query heads per KV head, Hkv (dense) or Hq (packed sequences)
  FastDiv div_gsize, div_band, div_band_last, div_group, div_heads;
  int n_kblocks;           // ceil(Sk / kBlockK)
  float scale2;            // scale * log2(e) (times descale_q * descale_k for e4m3)
  float inv_scale;         // 1 / (scale * descale_q * descale_k): mask values enter s in score units
  float out_scale;         // descale_v for e4m3, else 1
  // condensed additive mask (null when there is none)
  const uint4* mask_bits;  // [B, Sq, n_kblocks] x 128 bits, bit set = -inf
  const uint8_t* mask_flags;  // [B, Sq, n_kblocks], 1 = block row holds finite non-zero values
  const uint16_t* mask;    // original fp16 mask, read only for flagged block rows
  int64_t mask_b, mask_i;  // element strides of the original mask
  uint32_t* status;        // device status word
  int stall_first_stage;   // test hook: the producer never fills the first K/V stage
  // Work units: n_full whole work tiles, then split_tail work tiles cut into split_parts key
  // ranges each (see prefill_split_plan); n_units = n_full + split_tail * split_parts.
  int n_units, n_full, split_tail, split_parts;
  float* split_o;          // [split_tail, split_parts, kCtaRows, DV] unnormalised fp32 O
  float* split_ml;         // [split_tail, split_parts, kCtaRows, 2] row max (log2 units), row sum
  // packed variable-length sequences (varlen != 0): q/o rows cu_q[b] .. cu_q[b+1] and k/v rows
  // cu_k[b] .. cu_k[b+1] belong to sequence b; tile_prefix[b] counts the work tiles (2 x 128 query
  // rows) of the sequences before b, tile_prefix[B] all of them; lse is [Hq, total_q]
  int varlen, total_q;
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* tile_prefix;
  // int8 codes (kBlockScaled): score of (row i, key j) = scale2 * q_scale[b, h, i / 128] *
  // k_scale[b, kvh, j / 128] * (integer dot product); O column c times v_scale[b, kvh, c] if given
  const float* q_scale;    // [B, Hq, n_qblocks]
  const float* k_scale;    // [B, Hkv, n_kblocks]
  const float* v_scale;    // [B, Hkv, DV] or null
  int n_qblocks;
};

struct VarlenPrepParams {
  const int32_t* cu_q;     // [B + 1] query row offsets
  const int32_t* cu_k;     // [B + 1] key row offsets
  int B, total_q, total_k;
  int max_tiles;           // work tiles the prefill launch has units for
  int32_t* tile_prefix;    // [B + 1]
  uint32_t* status;        // device status word
};

// Key-range split of the last, partial wave of work tiles.  With items work tiles on sms
// persistent CTAs, items % sms tiles are left for a final round that would keep most SMs idle;
// when the attention is not causal (all tiles equally long) each of those tail tiles is cut
// into `parts` key ranges that run on otherwise idle SMs; a combine kernel then merges the
// parts' (O, max, sum) of every row with log-sum-exp weights.
constexpr int kMaxSplitParts = 8;
struct SplitPlan {
  int tail = 0;   // work tiles split (the last `tail` in launch order)
  int parts = 1;  // key ranges per split tile (1 = no split)
};
inline SplitPlan prefill_split_plan(long long items, int sms, int n_kblocks, bool causal) {
  SplitPlan sp;
  if (causal || sms < 2 || items <= 0) return sp;
  const long long tail = items % sms;
  if (tail == 0) return sp;
  long long parts = sms / tail;
  if (parts > kMaxSplitParts) parts = kMaxSplitParts;
  if (parts > n_kblocks) parts = n_kblocks;
  if (parts < 2) return sp;
  sp.tail = static_cast<int>(tail);
  sp.parts = static_cast<int>(parts);
  return sp;
}
inline size_t split_round16(size_t x) { return (x + 15) & ~size_t(15); }
// Workspace bytes of a split plan: partial O, then partial (max, sum).
inline size_t prefill_split_bytes(const SplitPlan& sp, int Dv) {
  if (sp.parts < 2) return 0;
  const size_t rows = static_cast<size_t>(sp.tail) * sp.parts * kCtaRows;
  return split_round16(rows * Dv * 4) + split_round16(rows * 2 * 4);
}

struct DecodeParams {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* kv_len;
  void* o;
  float* lse;
  float* ws;               // [B, Hq, n_splits_max, Dv + 2]
  uint32_t* status;        // device status word
  int64_t q_b, q_h, k_b, k_s, k_h, v_b, v_s, v_h, o_b, o_h;
  int B, Hq, Hkv, max_kv, group, n_splits_max;
  float scale2;            // scale * log2(e)
  // paged caches (page_table != null): key row t of sequence b is row t % page_size of physical
  // page page_table[b * pt_b + t / page_size]; k/v then point at pools [n_pages, page_size, Hkv, .]
  // and k_b/k_s (v_b/v_s) are the page and row strides
  const int32_t* page_table;
  int64_t pt_b;
  int page_size, log2_page, max_pages, n_pages;
};

constexpr int kDecodeSplit = 2048;      // keys per phase-1 CTA (1024 measured 7-8% slower)
constexpr int kDecodeWarps = 4;         // consumer warps: 16 keys of every 64-key chunk each
constexpr int kDecodeDv = 128;

struct MaskConvertParams {
  const uint16_t* mask;
  int64_t mask_b, mask_i;
  int B, Sq, Sk, n_kblocks;
  uint4* bits;
  uint8_t* flags;
};

// int8 tensors [B, S, H, Dh] (element strides, 16-byte aligned rows) widened to contiguous
// 16-bit copies of the same codes (every int8 value is exact in f16 and bf16).
struct WidenSeg {
  const int8_t* src;
  int64_t sb, ss, sh;
  int B, S, H, Dh;         // Dh a multiple of 16; B * S * H < 2^31
  void* dst;               // [B, S, H, Dh] contiguous
  int contig;              // the source is contiguous [B, S, H, Dh] too
};
struct WidenParams {
  WidenSeg seg[3];
  int n_seg;
  int to_bf16;             // 1: bf16 copies, 0: f16
};

// Kernel launchers (return cudaError_t of the launch).  The prefill launchers take the tensor
// maps of Q, K, V and O and set *supported = false (and launch nothing) for head dims they were
// not built for.
cudaError_t launch_prefill_f16(int D, int Dv, bool causal, bool has_mask, const CUtensorMap& tq,
                               const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to, const PrefillParams& p, cudaStream_t st,
                               bool* supported);
cudaError_t launch_prefill_bf16(int D, int Dv, bool causal, bool has_mask, const CUtensorMap& tq,
                                const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to, const PrefillParams& p, cudaStream_t st,
                                bool* supported);
cudaError_t launch_prefill_f16_block_scaled(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                           const CUtensorMap& tv, const CUtensorMap& to, const PrefillParams& p, cudaStream_t st,
                                           bool* supported);
cudaError_t launch_prefill_bf16_block_scaled(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                            const CUtensorMap& tv, const CUtensorMap& to, const PrefillParams& p, cudaStream_t st,
                                            bool* supported);
cudaError_t launch_prefill_e4m3(int D, int Dv, bool causal, bool has_mask, const CUtensorMap& tq,
                                const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to, const PrefillParams& p, cudaStream_t st,
                                bool* supported);

cudaError_t launch_decode(int elem, int D, const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                          cudaStream_t st);

// The decode entry points share one validated call description, built without any CUDA call,
// and one launch path; they differ only in where the per-split partials go.
struct DecodeCall {
  DecodeParams p;          // every field but ws and status
  int elem, D, Dv;
  int map_b, map_s;        // tensor-map extents: [map_b, map_s, Hkv, .] (batch x max_kv, or pages x page_size)
  int box_rows;            // rows of one TMA box
};
// Validates a decode call (page_table null: contiguous caches [B, max_kv, Hkv, .], else pools
// [n_pages, page_size, Hkv, .] with max_kv = max_pages * page_size) and fills *call.  Returns 0
// or the public status code (invalid / unsupported) of the first argument that fails.
int decode_check(const void* q, const void* k, const void* v, const int32_t* page_table, const int32_t* kv_len,
                 void* o, float* lse, int B, int Hq, int Hkv, int max_kv, int page_size, int max_pages, int n_pages,
                 int D, int Dv, const int64_t* strides, float scale, int dtype, DecodeCall* call);
// Bytes of per-split partial results of a decode: [B, Hq, n_splits, Dv + 2] fp32, 16-byte rounded.
size_t decode_partials_bytes(int B, int Hq, int max_kv, int Dv);
// Encodes the tensor maps and launches both phases with the partials in ws; 0 or the public
// status code of a CUDA failure.
int decode_launch(DecodeCall& call, float* ws, cudaStream_t st);

// Device address of the current device's status word.
cudaError_t device_status_ptr(uint32_t** out);

// The current device and its SM count; the count is looked up on the first call per device and
// kept, so a launch costs no device query.
constexpr int kMaxDevices = 64;
cudaError_t current_device_sms(int* dev, int* sms);

// One-time opt-in of kernel `kern` to `bytes` of dynamic shared memory on device `dev`; `done`
// (one per kernel) records the devices already set up, one bit each.
template <typename Kernel>
cudaError_t smem_opt_in(Kernel kern, int bytes, int dev, std::atomic<uint64_t>& done) {
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Tensor map of a [B, S, H, Dh] tensor (element strides sb, ss, sh; innermost stride 1) with a
// box of box0 x 1 x box_rows x 1 elements; false if the driver rejects it.
bool encode_bshd(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int esize, int B, int S, int H, int Dh,
                 int64_t sb, int64_t ss, int64_t sh, int box0, int box_rows, CUtensorMapSwizzle sw);
cudaError_t launch_mask_convert(const MaskConvertParams& p, cudaStream_t st);
cudaError_t launch_varlen_prep(const VarlenPrepParams& p, cudaStream_t st);
cudaError_t launch_widen(const WidenParams& p, cudaStream_t st);

}  // namespace sdpa
