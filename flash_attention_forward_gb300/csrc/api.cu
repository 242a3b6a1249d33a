// C ABI of the library (declared in include/sdpa.h): argument validation, tensor-map
// encoding, instance dispatch and the device status word.  No entry point allocates
// device memory; every argument is checked before the first CUDA call.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <atomic>
#include <mutex>

#include "sdpa.h"
#include "internal.h"

namespace sdpa {
namespace {
__device__ uint32_t g_status_word;
}  // namespace

std::atomic<uint32_t*> g_status_ptr[kMaxDevices] = {};
std::atomic<int> g_sm_count[kMaxDevices] = {};

namespace {
std::atomic<int> g_stall_next{0};

// Device address of this device's status word (looked up once per device; a race between two
// first calls resolves the same address twice).
cudaError_t status_ptr(uint32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  uint32_t* ptr = g_status_ptr[dev].load(std::memory_order_acquire);
  if (ptr == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return e;
    ptr = static_cast<uint32_t*>(p);
    g_status_ptr[dev].store(ptr, std::memory_order_release);
  }
  *out = ptr;
  return cudaSuccess;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

cudaError_t device_status_ptr(uint32_t** out) { return status_ptr(out); }

cudaError_t current_device_sms(int* dev, int* sms) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  if (*dev < 0 || *dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int n = g_sm_count[*dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, *dev)) != cudaSuccess) return e;
    g_sm_count[*dev].store(n, std::memory_order_relaxed);
  }
  *sms = n;
  return cudaSuccess;
}

bool encode_bshd(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int esize, int B, int S, int H, int Dh,
                 int64_t sb, int64_t ss, int64_t sh, int box0, int box_rows, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)Dh, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)(sh * esize), (cuuint64_t)(ss * esize), (cuuint64_t)(sb * esize)};
  const cuuint32_t box[4] = {(cuuint32_t)box0, 1u, (cuuint32_t)box_rows, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return fn(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Strides usable by a tensor map / 16-byte vector access: positive multiples of `mult` (a
// stride of a size-1 dimension only needs the multiple).
bool stride_ok(int64_t s, int64_t mult) { return s >= 0 && s % mult == 0 && s < (int64_t(1) << 36); }

size_t round16(size_t x) { return (x + 15) & ~size_t(15); }

size_t mask_ws_bytes(int B, int Sq, int Sk) {
  const size_t nkb = (size_t)((Sk + kBlockK - 1) / kBlockK);
  const size_t rows = (size_t)B * (size_t)Sq;
  return round16(rows * nkb * sizeof(uint4)) + round16(rows * nkb);
}

// Split plan of a prefill launch on the current device (no split if the device query fails).
SplitPlan fwd_split_plan(int B, int Hq, int Sq, int Sk, bool causal) {
  int dev = 0, sms = 0;
  if (current_device_sms(&dev, &sms) != cudaSuccess) {
    cudaGetLastError();  // clear the error so that later calls do not see it
    return SplitPlan{};
  }
  const long long items = (long long)((Sq + kCtaRows - 1) / kCtaRows) * B * Hq;
  return prefill_split_plan(items, sms, (Sk + kBlockK - 1) / kBlockK, causal);
}

// Packed variable-length sequences: sequence b owns query rows cu_q[b] .. cu_q[b + 1] and key
// rows cu_k[b] .. cu_k[b + 1] of [total, H, D] tensors.
struct VarlenArgs {
  const int32_t* cu_q;
  const int32_t* cu_k;
  int total_q, total_k, max_seqlen_q;
};

size_t varlen_ws_bytes(int B) { return round16((size_t)(B + 1) * sizeof(int32_t)); }

// Work tiles a varlen launch is sized for: no sequence is longer than max_seqlen_q, and the
// lengths add up to at most total_q.
long long varlen_max_tiles(int B, int total_q, int max_seqlen_q) {
  const long long by_max = (long long)B * ((max_seqlen_q + kCtaRows - 1) / kCtaRows);
  const long long by_total = ((long long)total_q + (long long)(kCtaRows - 1) * B) / kCtaRows;
  return by_max < by_total ? by_max : by_total;
}

// int8 codes: per-block scales, and the widening of the codes that runs just before the prefill.
struct Int8Args {
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  WidenParams widen;
};

// Shared body of the dense, packed and int8-code entry points (vl != null: B sequences packed as
// described by *vl; Sq, Sk are then the longest query length and total_k.  i8 != null: q, k (and
// v) are the 16-bit copies that i8->widen writes, scaled per block).
int fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
               int Sk, int D, int Dv, const int64_t* strides, float scale, int causal, const void* mask,
               const int64_t* mask_strides, void* workspace, size_t workspace_bytes, int elem, float descale_q,
               float descale_k, float descale_v, sdpa_dtype out_dtype, void* stream,
               const VarlenArgs* vl = nullptr, const Int8Args* i8 = nullptr, int causal_off = 0,
               int64_t lse_ld = 0) {
  // ---- validation (no CUDA call before this block passes)
  if (!q || !k || !v || !o) return SDPA_ERR_INVALID;
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1 || D < 1 || Dv < 1) return SDPA_ERR_INVALID;
  if (Hq % Hkv != 0) return SDPA_ERR_INVALID;
  if (!(std::isfinite(scale) && scale > 0.f)) return SDPA_ERR_INVALID;
  if (!(std::isfinite(descale_q) && descale_q > 0.f && std::isfinite(descale_k) && descale_k > 0.f &&
        std::isfinite(descale_v) && descale_v > 0.f))
    return SDPA_ERR_INVALID;
  const int esize = (elem == kE4M3) ? 1 : 2;
  // head dims built for every input type: (64, 64), (128, 128), (192, 128)
  if (!((D == 64 && Dv == 64) || (D == 128 && Dv == 128) || (D == 192 && Dv == 128))) return SDPA_ERR_UNSUPPORTED;
  if (elem == kE4M3) {
    if (out_dtype != SDPA_BF16) return SDPA_ERR_UNSUPPORTED;
  } else {
    if ((elem == kF16 && out_dtype != SDPA_F16) || (elem == kBF16 && out_dtype != SDPA_BF16))
      return SDPA_ERR_UNSUPPORTED;
  }
  int64_t st[SDPA_FWD_NSTRIDES];
  if (vl) {
    // (row, head) strides per tensor; the batch dimension of the tensor maps has extent 1
    int64_t r[SDPA_FWD_VARLEN_NSTRIDES] = {(int64_t)Hq * D, D, (int64_t)Hkv * D, D,
                                          (int64_t)Hkv * Dv, Dv, (int64_t)Hq * Dv, Dv};
    if (strides) std::memcpy(r, strides, sizeof(r));
    const int64_t rows[4] = {vl->total_q, vl->total_k, vl->total_k, vl->total_q};
    for (int t = 0; t < 4; ++t) {
      st[3 * t] = r[2 * t] * rows[t];
      st[3 * t + 1] = r[2 * t];
      st[3 * t + 2] = r[2 * t + 1];
    }
  } else if (strides) {
    std::memcpy(st, strides, sizeof(st));
  } else {
    const int64_t cs[SDPA_FWD_NSTRIDES] = {(int64_t)Sq * Hq * D,  (int64_t)Hq * D,  D,
                                           (int64_t)Sk * Hkv * D, (int64_t)Hkv * D, D,
                                           (int64_t)Sk * Hkv * Dv, (int64_t)Hkv * Dv, Dv,
                                           (int64_t)Sq * Hq * Dv, (int64_t)Hq * Dv, Dv};
    std::memcpy(st, cs, sizeof(st));
  }
  const int64_t in_mult = 16 / esize;  // 16-byte tensor-map strides
  for (int i = 0; i < 9; ++i)
    if (!stride_ok(st[i], in_mult)) return SDPA_ERR_UNSUPPORTED;
  for (int i = 9; i < 12; ++i)
    if (!stride_ok(st[i], 8)) return SDPA_ERR_UNSUPPORTED;  // 16-byte output vectors
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return SDPA_ERR_UNSUPPORTED;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SDPA_ERR_INVALID;
  const int n_kblocks = (Sk + kBlockK - 1) / kBlockK;
  const int n_cta_tiles = (Sq + kCtaRows - 1) / kCtaRows;
  const long long n_items = vl ? varlen_max_tiles(B, vl->total_q, vl->max_seqlen_q) * Hq
                               : (long long)n_cta_tiles * B * Hq;
  if (n_items * kMaxSplitParts >= (1ll << 31)) return SDPA_ERR_UNSUPPORTED;
  if (i8 && (mask || vl || elem == kE4M3 || D != Dv || D == 192)) return SDPA_ERR_UNSUPPORTED;
  if (vl) {
    if (!vl->cu_q || !vl->cu_k || mask) return SDPA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(vl->cu_q) | reinterpret_cast<uintptr_t>(vl->cu_k)) & 3u) return SDPA_ERR_INVALID;
    if (!workspace || !aligned16(workspace) || workspace_bytes < varlen_ws_bytes(B)) return SDPA_ERR_INVALID;
  }
  int64_t mb = 0, mi = 0;
  if (mask) {
    if (reinterpret_cast<uintptr_t>(mask) & 1u) return SDPA_ERR_INVALID;
    mb = mask_strides ? mask_strides[0] : (int64_t)Sq * Sk;
    mi = mask_strides ? mask_strides[1] : (int64_t)Sk;
    if (mb < 0 || mi < 0) return SDPA_ERR_INVALID;
    if (!workspace || !aligned16(workspace) || workspace_bytes < mask_ws_bytes(B, Sq, Sk)) return SDPA_ERR_INVALID;
  }
  // the key-range split of the tail runs only when the caller's workspace also holds its
  // partial results (sdpa_fwd_workspace_size includes them)
  const size_t mask_bytes = mask ? mask_ws_bytes(B, Sq, Sk) : 0;
  SplitPlan sp = vl ? SplitPlan{} : fwd_split_plan(B, Hq, Sq, Sk, causal != 0);
  const size_t split_bytes = prefill_split_bytes(sp, Dv);
  if (split_bytes == 0 || !workspace || !aligned16(workspace) || workspace_bytes < mask_bytes + split_bytes)
    sp = SplitPlan{};

  // ---- tensor maps
  const CUtensorMapDataType dt = elem == kE4M3   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : elem == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapSwizzle sw_qk = elem == kE4M3 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  alignas(64) CUtensorMap tq, tk, tv, to;
  const int mB = vl ? 1 : B, mSq = vl ? vl->total_q : Sq, mSk = vl ? vl->total_k : Sk;  // tensor-map extents
  if (!encode_bshd(&tq, q, dt, esize, mB, mSq, Hq, D, st[0], st[1], st[2], 64, kBlockQ, sw_qk)) return SDPA_ERR_CUDA;
  if (!encode_bshd(&tk, k, dt, esize, mB, mSk, Hkv, D, st[3], st[4], st[5], 64, kBlockK, sw_qk)) return SDPA_ERR_CUDA;
  const bool v_ok = elem == kE4M3
                        ? encode_bshd(&tv, v, dt, 1, mB, mSk, Hkv, Dv, st[6], st[7], st[8], Dv, kBlockK,
                                      CU_TENSOR_MAP_SWIZZLE_NONE)
                        : encode_bshd(&tv, v, dt, 2, mB, mSk, Hkv, Dv, st[6], st[7], st[8], 64, kBlockK,
                                      CU_TENSOR_MAP_SWIZZLE_128B);
  if (!v_ok) return SDPA_ERR_CUDA;
  // O [B, Sq, Hq, Dv] in the output type, 64-column boxes of 128 rows (the epilogue's TMA stores;
  // rows past Sq are clipped; packed sequences store row by row instead)
  const CUtensorMapDataType odt = out_dtype == SDPA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!encode_bshd(&to, o, odt, 2, mB, mSq, Hq, Dv, st[9], st[10], st[11], 64, kBlockQ, CU_TENSOR_MAP_SWIZZLE_128B))
    return SDPA_ERR_CUDA;

  uint32_t* status = nullptr;
  if (status_ptr(&status) != cudaSuccess) return SDPA_ERR_CUDA;
  cudaStream_t stm = static_cast<cudaStream_t>(stream);

  PrefillParams p{};
  p.o = o;
  p.lse = lse;
  p.o_b = st[9], p.o_s = st[10], p.o_h = st[11];
  p.B = B, p.Hq = Hq, p.Hkv = Hkv, p.Sq = Sq, p.Sk = Sk;
  p.lse_ld = lse_ld > 0 ? lse_ld : Sq;
  p.causal_off = causal_off;
  p.group = Hq / Hkv;
  p.n_cta_tiles = n_cta_tiles;
  p.n_kblocks = n_kblocks;
  const double s_eff = (double)scale * (double)descale_q * (double)descale_k;
  p.scale2 = (float)(s_eff * 1.4426950408889634);
  p.inv_scale = (float)(1.0 / s_eff);
  p.out_scale = descale_v;
  p.status = status;
  p.stall_first_stage = g_stall_next.exchange(0);
  p.n_full = (int)(n_items - sp.tail);
  p.split_tail = sp.tail;
  p.split_parts = sp.parts;
  p.n_units = p.n_full + sp.tail * sp.parts;
  if (sp.parts > 1) {
    char* base = static_cast<char*>(workspace) + mask_bytes;
    const size_t rows = (size_t)sp.tail * sp.parts * kCtaRows;
    p.split_o = reinterpret_cast<float*>(base);
    p.split_ml = reinterpret_cast<float*>(base + round16(rows * Dv * 4));
  }
  if (mask) {
    const size_t rows = (size_t)B * (size_t)Sq;
    uint4* bits = static_cast<uint4*>(workspace);
    uint8_t* flags = reinterpret_cast<uint8_t*>(static_cast<char*>(workspace) + round16(rows * n_kblocks * sizeof(uint4)));
    MaskConvertParams mp{static_cast<const uint16_t*>(mask), mb, mi, B, Sq, Sk, n_kblocks, bits, flags};
    if (launch_mask_convert(mp, stm) != cudaSuccess) return SDPA_ERR_CUDA;
    p.mask_bits = bits;
    p.mask_flags = flags;
    p.mask = static_cast<const uint16_t*>(mask);
    p.mask_b = mb, p.mask_i = mi;
  }
  if (vl) {
    int32_t* prefix = static_cast<int32_t*>(workspace);
    VarlenPrepParams vp{vl->cu_q, vl->cu_k, B, vl->total_q, vl->total_k, (int)(n_items / Hq), prefix, status};
    if (launch_varlen_prep(vp, stm) != cudaSuccess) return SDPA_ERR_CUDA;
    p.varlen = 1;
    p.total_q = vl->total_q;
    p.cu_q = vl->cu_q;
    p.cu_k = vl->cu_k;
    p.tile_prefix = prefix;
  }
  bool supported = false;
  cudaError_t e;
  if (i8) {
    if (launch_widen(i8->widen, stm) != cudaSuccess) return SDPA_ERR_CUDA;
    p.q_scale = i8->q_scale;
    p.k_scale = i8->k_scale;
    p.v_scale = i8->v_scale;
    p.n_qblocks = (Sq + kBlockQ - 1) / kBlockQ;
    e = elem == kBF16 ? launch_prefill_bf16_block_scaled(D, causal != 0, tq, tk, tv, to, p, stm, &supported)
                      : launch_prefill_f16_block_scaled(D, causal != 0, tq, tk, tv, to, p, stm, &supported);
    if (!supported) return SDPA_ERR_UNSUPPORTED;
    return e == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
  }
  if (elem == kE4M3)
    e = launch_prefill_e4m3(D, Dv, causal != 0, mask != nullptr, tq, tk, tv, to, p, stm, &supported);
  else if (elem == kBF16)
    e = launch_prefill_bf16(D, Dv, causal != 0, mask != nullptr, tq, tk, tv, to, p, stm, &supported);
  else
    e = launch_prefill_f16(D, Dv, causal != 0, mask != nullptr, tq, tk, tv, to, p, stm, &supported);
  if (!supported) return SDPA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

}  // namespace

size_t decode_partials_bytes(int B, int Hq, int max_kv, int Dv) {
  const size_t n_splits = (size_t)((max_kv + kDecodeSplit - 1) / kDecodeSplit);
  return round16((size_t)B * Hq * n_splits * (size_t)(Dv + 2) * sizeof(float));
}

int decode_check(const void* q, const void* k, const void* v, const int32_t* page_table, const int32_t* kv_len,
                 void* o, float* lse, int B, int Hq, int Hkv, int max_kv, int page_size, int max_pages, int n_pages,
                 int D, int Dv, const int64_t* strides, float scale, int dtype, DecodeCall* call) {
  const bool paged = page_table != nullptr;
  if (!q || !k || !v || !kv_len || !o) return SDPA_ERR_INVALID;
  if (B < 1 || Hq < 1 || Hkv < 1 || max_kv < 1 || D < 1 || Dv < 1) return SDPA_ERR_INVALID;
  if (Hq % Hkv != 0) return SDPA_ERR_INVALID;
  if (!(std::isfinite(scale) && scale > 0.f)) return SDPA_ERR_INVALID;
  if (paged && (page_size & (page_size - 1))) return SDPA_ERR_INVALID;  // a power of two
  if (dtype != SDPA_F16 && dtype != SDPA_BF16) return SDPA_ERR_UNSUPPORTED;
  // head dims: (128, 128) and the MLA shape (192, 128)
  if (!((D == 128 || D == 192) && Dv == kDecodeDv)) return SDPA_ERR_UNSUPPORTED;
  if (paged && page_size < 16) return SDPA_ERR_UNSUPPORTED;
  const int group = Hq / Hkv;
  if (group > 16) return SDPA_ERR_UNSUPPORTED;  // one 16-row tensor-core tile per KV head
  if (B > 65535 || Hkv > 65535) return SDPA_ERR_UNSUPPORTED;  // launch-grid y and z extents
  // element strides {q_b, q_h, k_b, k_s, k_h, v_b, v_s, v_h, o_b, o_h} (+ page-table row stride)
  int64_t st[SDPA_DECODE_PAGED_NSTRIDES];
  const int rows = paged ? page_size : max_kv;  // rows of one batch entry of the caches
  if (strides) {
    std::memcpy(st, strides, sizeof(int64_t) * (paged ? SDPA_DECODE_PAGED_NSTRIDES : SDPA_DECODE_NSTRIDES));
  } else {
    const int64_t cs[SDPA_DECODE_PAGED_NSTRIDES] = {(int64_t)Hq * D,  D,  (int64_t)rows * Hkv * D, (int64_t)Hkv * D,
                                                    D, (int64_t)rows * Hkv * Dv, (int64_t)Hkv * Dv, Dv,
                                                    (int64_t)Hq * Dv, Dv, max_pages};
    std::memcpy(st, cs, sizeof(st));
  }
  for (int i = 0; i < SDPA_DECODE_NSTRIDES; ++i)
    if (!stride_ok(st[i], 8)) return SDPA_ERR_UNSUPPORTED;  // 16-byte rows for TMA and vector loads
  if (paged && st[10] < max_pages) return SDPA_ERR_INVALID;  // page-table rows hold max_pages entries
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return SDPA_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(kv_len) & 3u) return SDPA_ERR_INVALID;
  if (paged && (reinterpret_cast<uintptr_t>(page_table) & 3u)) return SDPA_ERR_INVALID;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SDPA_ERR_INVALID;

  DecodeParams& p = call->p;
  p = DecodeParams{};
  p.q = q, p.k = k, p.v = v, p.kv_len = kv_len, p.o = o, p.lse = lse;
  p.q_b = st[0], p.q_h = st[1], p.k_b = st[2], p.k_s = st[3], p.k_h = st[4];
  p.v_b = st[5], p.v_s = st[6], p.v_h = st[7], p.o_b = st[8], p.o_h = st[9];
  p.B = B, p.Hq = Hq, p.Hkv = Hkv, p.max_kv = max_kv, p.group = group;
  p.n_splits_max = (max_kv + kDecodeSplit - 1) / kDecodeSplit;
  p.scale2 = (float)((double)scale * 1.4426950408889634);
  if (paged) {
    p.page_table = page_table;
    p.pt_b = st[10];
    p.page_size = page_size;
    p.log2_page = __builtin_ctz((unsigned)page_size);
    p.max_pages = max_pages;
    p.n_pages = n_pages;
  }
  call->elem = dtype == SDPA_BF16 ? kBF16 : kF16;
  call->D = D, call->Dv = Dv;
  call->map_b = paged ? n_pages : B;
  call->map_s = rows;
  call->box_rows = paged && page_size < 64 ? page_size : 64;  // a box never spans two pages
  return SDPA_OK;
}

int decode_launch(DecodeCall& call, float* ws, cudaStream_t st) {
  DecodeParams& p = call.p;
  const CUtensorMapDataType dt = call.elem == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  alignas(64) CUtensorMap tk, tv;
  if (!encode_bshd(&tk, p.k, dt, 2, call.map_b, call.map_s, p.Hkv, call.D, p.k_b, p.k_s, p.k_h, 64, call.box_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_bshd(&tv, p.v, dt, 2, call.map_b, call.map_s, p.Hkv, call.Dv, p.v_b, p.v_s, p.v_h, 64, call.box_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return SDPA_ERR_CUDA;
  uint32_t* status = nullptr;
  if (status_ptr(&status) != cudaSuccess) return SDPA_ERR_CUDA;
  p.ws = ws;
  p.status = status;
  return launch_decode(call.elem, call.D, p, tk, tv, st) == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

}  // namespace sdpa

using namespace sdpa;

extern "C" {

size_t sdpa_fwd_workspace_size(int B, int Hq, int Sq, int Sk, int Dv, int causal, int has_mask) {
  if (B < 1 || Hq < 1 || Sq < 1 || Sk < 1 || Dv < 1) return 0;
  const size_t mask_bytes = has_mask ? mask_ws_bytes(B, Sq, Sk) : 0;
  return mask_bytes + prefill_split_bytes(fwd_split_plan(B, Hq, Sq, Sk, causal != 0), Dv);
}

int sdpa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
             int Sk, int D, int Dv, const int64_t* strides, float scale, int causal, const void* mask,
             const int64_t* mask_strides, void* workspace, size_t workspace_bytes, sdpa_dtype in_dtype,
             sdpa_dtype out_dtype, void* stream) {
  if (in_dtype != SDPA_F16 && in_dtype != SDPA_BF16) return SDPA_ERR_UNSUPPORTED;
  return fwd_common(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, Dv, strides, scale, causal, mask, mask_strides,
                    workspace, workspace_bytes, in_dtype == SDPA_BF16 ? kBF16 : kF16, 1.f, 1.f, 1.f, out_dtype,
                    stream);
}

int sdpa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
                 int Sk, int D, int Dv, const int64_t* strides, float scale, int causal, const void* mask,
                 const int64_t* mask_strides, void* workspace, size_t workspace_bytes, float descale_q,
                 float descale_k, float descale_v, sdpa_dtype out_dtype, void* stream) {
  return fwd_common(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, Dv, strides, scale, causal, mask, mask_strides,
                    workspace, workspace_bytes, kE4M3, descale_q, descale_k, descale_v, out_dtype, stream);
}

size_t sdpa_fwd_varlen_workspace_size(int B) { return B < 1 ? 0 : varlen_ws_bytes(B); }

namespace {
int fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens_q,
               const int32_t* cu_seqlens_k, int B, int Hq, int Hkv, int total_q, int total_k, int max_seqlen_q,
               int D, int Dv, const int64_t* strides, float scale, int causal, void* workspace,
               size_t workspace_bytes, int elem, float descale_q, float descale_k, float descale_v,
               sdpa_dtype out_dtype, void* stream) {
  if (B < 1 || total_q < 1 || total_k < 1 || max_seqlen_q < 1 || max_seqlen_q > total_q) return SDPA_ERR_INVALID;
  const VarlenArgs vl{cu_seqlens_q, cu_seqlens_k, total_q, total_k, max_seqlen_q};
  return fwd_common(q, k, v, o, lse, B, Hq, Hkv, max_seqlen_q, total_k, D, Dv, strides, scale,
                    causal, nullptr, nullptr, workspace, workspace_bytes, elem, descale_q, descale_k, descale_v,
                    out_dtype, stream, &vl);
}
}  // namespace

int sdpa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens_q,
                    const int32_t* cu_seqlens_k, int B, int Hq, int Hkv, int total_q, int total_k, int max_seqlen_q,
                    int D, int Dv, const int64_t* strides, float scale, int causal, void* workspace,
                    size_t workspace_bytes, sdpa_dtype in_dtype, sdpa_dtype out_dtype, void* stream) {
  if (in_dtype != SDPA_F16 && in_dtype != SDPA_BF16) return SDPA_ERR_UNSUPPORTED;
  return fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, total_q, total_k, max_seqlen_q, D, Dv,
                    strides, scale, causal, workspace, workspace_bytes, in_dtype == SDPA_BF16 ? kBF16 : kF16, 1.f,
                    1.f, 1.f, out_dtype, stream);
}

int sdpa_fwd_varlen_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B, int Hq, int Hkv, int total_q,
                        int total_k, int max_seqlen_q, int D, int Dv, const int64_t* strides, float scale, int causal,
                        void* workspace, size_t workspace_bytes, float descale_q, float descale_k, float descale_v,
                        sdpa_dtype out_dtype, void* stream) {
  return fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, total_q, total_k, max_seqlen_q, D, Dv,
                    strides, scale, causal, workspace, workspace_bytes, kE4M3, descale_q, descale_k, descale_v,
                    out_dtype, stream);
}

namespace {
// Bytes of the widened 16-bit copies of the int8 operands (Q, K, and V when it is int8).
size_t int8_widened_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D, bool v_int8) {
  const size_t q = round16((size_t)B * Sq * Hq * D * 2), kv = round16((size_t)B * Sk * Hkv * D * 2);
  return q + kv + (v_int8 ? kv : 0);
}
}  // namespace

size_t sdpa_fwd_int8_workspace_size(int B, int Hq, int Hkv, int Sq, int Sk, int D, int v_int8, int causal) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1 || D < 1) return 0;
  return int8_widened_bytes(B, Hq, Hkv, Sq, Sk, D, v_int8 != 0) +
         prefill_split_bytes(fwd_split_plan(B, Hq, Sq, Sk, causal != 0), D);
}

int sdpa_fwd_int8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
                  int Sk, int D, const int64_t* strides, const float* q_scale, const float* k_scale,
                  const float* v_scale, float scale, int causal, void* workspace, size_t workspace_bytes,
                  sdpa_dtype v_dtype, sdpa_dtype out_dtype, void* stream) {
  if (!q || !k || !v || !o || !q_scale || !k_scale) return SDPA_ERR_INVALID;
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1 || D < 1) return SDPA_ERR_INVALID;
  if (out_dtype != SDPA_F16 && out_dtype != SDPA_BF16) return SDPA_ERR_UNSUPPORTED;
  if (v_dtype != SDPA_I8 && v_dtype != out_dtype) return SDPA_ERR_UNSUPPORTED;
  const bool v_int8 = v_dtype == SDPA_I8;
  if (v_int8 != (v_scale != nullptr)) return SDPA_ERR_INVALID;
  if (D != 64 && D != 128) return SDPA_ERR_UNSUPPORTED;
  if (((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale)) & 3u) ||
      (v_scale && !aligned16(v_scale)))
    return SDPA_ERR_INVALID;
  int64_t st[SDPA_FWD_NSTRIDES];
  if (strides) {
    std::memcpy(st, strides, sizeof(st));
  } else {
    const int64_t cs[SDPA_FWD_NSTRIDES] = {(int64_t)Sq * Hq * D, (int64_t)Hq * D, D, (int64_t)Sk * Hkv * D,
                                           (int64_t)Hkv * D,     D,               (int64_t)Sk * Hkv * D,
                                           (int64_t)Hkv * D,     D,               (int64_t)Sq * Hq * D,
                                           (int64_t)Hq * D,      D};
    std::memcpy(st, cs, sizeof(st));
  }
  // int8 operands: 16-byte rows for the widening loads
  for (int i = 0; i < (v_int8 ? 9 : 6); ++i)
    if (!stride_ok(st[i], 16)) return SDPA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || (v_int8 && !aligned16(v))) return SDPA_ERR_UNSUPPORTED;
  const size_t wide = int8_widened_bytes(B, Hq, Hkv, Sq, Sk, D, v_int8);
  if (!workspace || !aligned16(workspace) || workspace_bytes < wide) return SDPA_ERR_INVALID;

  char* ws = static_cast<char*>(workspace);
  void* q16 = ws;
  void* k16 = ws + round16((size_t)B * Sq * Hq * D * 2);
  void* v16 = v_int8 ? static_cast<char*>(k16) + round16((size_t)B * Sk * Hkv * D * 2) : const_cast<void*>(v);
  Int8Args a{q_scale, k_scale, v_scale, WidenParams{}};
  a.widen.to_bf16 = out_dtype == SDPA_BF16;
  auto seg = [&](const void* src, const int64_t* s3, int S, int H) {
    const bool contig = s3[2] == D && s3[1] == (int64_t)H * D && s3[0] == (int64_t)S * H * D;
    return WidenSeg{static_cast<const int8_t*>(src), s3[0], s3[1], s3[2], B, S, H, D, nullptr, contig ? 1 : 0};
  };
  if ((long long)B * std::max(Sq, Sk) * std::max(Hq, Hkv) >= (1ll << 31)) return SDPA_ERR_UNSUPPORTED;
  a.widen.seg[0] = seg(q, st, Sq, Hq);
  a.widen.seg[0].dst = q16;
  a.widen.seg[1] = seg(k, st + 3, Sk, Hkv);
  a.widen.seg[1].dst = k16;
  if (v_int8) {
    a.widen.seg[2] = seg(v, st + 6, Sk, Hkv);
    a.widen.seg[2].dst = v16;
  }
  a.widen.n_seg = v_int8 ? 3 : 2;
  // the prefill reads the contiguous copies; V keeps the caller's strides when it is 16-bit
  const int64_t st16[SDPA_FWD_NSTRIDES] = {(int64_t)Sq * Hq * D,
                                           (int64_t)Hq * D,
                                           D,
                                           (int64_t)Sk * Hkv * D,
                                           (int64_t)Hkv * D,
                                           D,
                                           v_int8 ? (int64_t)Sk * Hkv * D : st[6],
                                           v_int8 ? (int64_t)Hkv * D : st[7],
                                           v_int8 ? (int64_t)D : st[8],
                                           st[9],
                                           st[10],
                                           st[11]};
  return fwd_common(q16, k16, v16, o, lse, B, Hq, Hkv, Sq, Sk, D, D, st16, scale, causal, nullptr, nullptr,
                    ws + wide, workspace_bytes - wide, out_dtype == SDPA_BF16 ? kBF16 : kF16, 1.f, 1.f, 1.f,
                    out_dtype, stream, nullptr, &a);
}

namespace {
constexpr int kMaxHostChunks = 8;

// Per device: the two copy streams and the events of sdpa_fwd_host, created on first use and
// kept for the life of the process.
struct HostPipe {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev[2 * kMaxHostChunks + 2] = {};
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu;  // held while a call enqueues (the events are shared)

cudaError_t host_pipe(int dev, HostPipe** out) {
  HostPipe& hp = g_pipe[dev];
  if (hp.h2d == nullptr) {
    // build the whole set first: a failure part-way leaves the device's entry empty
    HostPipe fresh;
    cudaError_t e = cudaStreamCreateWithFlags(&fresh.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&fresh.d2h, cudaStreamNonBlocking);
    for (cudaEvent_t& ev : fresh.ev)
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      for (cudaEvent_t ev : fresh.ev)
        if (ev) cudaEventDestroy(ev);
      if (fresh.d2h) cudaStreamDestroy(fresh.d2h);
      if (fresh.h2d) cudaStreamDestroy(fresh.h2d);
      return e;
    }
    hp = fresh;
  }
  *out = &hp;
  return cudaSuccess;
}

struct HostLayout {
  size_t q, k, v, o, lse, total;  // byte offsets of the device copies in the workspace, and their end
};

HostLayout host_layout(int B, int Hq, int Hkv, int Sq, int Sk, int D, int Dv, size_t esize) {
  HostLayout L{};
  L.q = 0;
  L.k = L.q + round16((size_t)B * Sq * Hq * D * esize);
  L.v = L.k + round16((size_t)B * Sk * Hkv * D * esize);
  L.o = L.v + round16((size_t)B * Sk * Hkv * Dv * esize);
  L.lse = L.o + round16((size_t)B * Sq * Hq * Dv * 2);
  L.total = L.lse + round16((size_t)B * Hq * Sq * 4);
  return L;
}

// Query rows per chunk: whole 256-row work tiles, at most kMaxHostChunks chunks.
int host_chunk_rows(int Sq) {
  const int per = (Sq + kMaxHostChunks - 1) / kMaxHostChunks;
  return std::max(kCtaRows, (per + kCtaRows - 1) / kCtaRows * kCtaRows);
}
}  // namespace

size_t sdpa_fwd_host_workspace_size(int B, int Hq, int Hkv, int Sq, int Sk, int D, int Dv, int causal) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1 || D < 1 || Dv < 1) return 0;
  const int rows = host_chunk_rows(Sq);
  return host_layout(B, Hq, Hkv, Sq, Sk, D, Dv, 2).total +
         prefill_split_bytes(fwd_split_plan(B, Hq, std::min(rows, Sq), Sk, causal != 0), Dv);
}

int sdpa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
                  int Sk, int D, int Dv, float scale, int causal, void* workspace, size_t workspace_bytes,
                  sdpa_dtype in_dtype, sdpa_dtype out_dtype, void* stream) {
  // ---- validation (no CUDA call before this block passes)
  if (!q || !k || !v || !o) return SDPA_ERR_INVALID;
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1 || D < 1 || Dv < 1 || Hq % Hkv != 0) return SDPA_ERR_INVALID;
  if (!(std::isfinite(scale) && scale > 0.f)) return SDPA_ERR_INVALID;
  if (in_dtype != SDPA_F16 && in_dtype != SDPA_BF16) return SDPA_ERR_UNSUPPORTED;
  if (out_dtype != in_dtype) return SDPA_ERR_UNSUPPORTED;
  if (!((D == 64 && Dv == 64) || (D == 128 && Dv == 128) || (D == 192 && Dv == 128))) return SDPA_ERR_UNSUPPORTED;
  const HostLayout L = host_layout(B, Hq, Hkv, Sq, Sk, D, Dv, 2);
  if (!workspace || !aligned16(workspace) || workspace_bytes < L.total) return SDPA_ERR_INVALID;
  const int rows = host_chunk_rows(Sq);
  const int n_chunks = (Sq + rows - 1) / rows;
  if ((long long)((rows + kCtaRows - 1) / kCtaRows) * B * Hq * kMaxSplitParts >= (1ll << 31))
    return SDPA_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDPA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe* hp = nullptr;
  if (host_pipe(dev, &hp) != cudaSuccess) return SDPA_ERR_CUDA;
  cudaStream_t stm = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  char *dq = ws + L.q, *dk = ws + L.k, *dv = ws + L.v, *dO = ws + L.o;
  float* dl = reinterpret_cast<float*>(ws + L.lse);
  const size_t qrow = (size_t)Hq * D * 2, krow = (size_t)Hkv * D * 2, vrow = (size_t)Hkv * Dv * 2,
               orow = (size_t)Hq * Dv * 2;
  const int64_t st[SDPA_FWD_NSTRIDES] = {(int64_t)Sq * Hq * D,   (int64_t)Hq * D,  D,
                                         (int64_t)Sk * Hkv * D,  (int64_t)Hkv * D, D,
                                         (int64_t)Sk * Hkv * Dv, (int64_t)Hkv * Dv, Dv,
                                         (int64_t)Sq * Hq * Dv,  (int64_t)Hq * Dv, Dv};
  // B rows of `bytes` starting at row r of a [B, S, ...] tensor whose rows are `row` bytes
  auto copy_rows = [&](void* dst, const void* src, size_t row, int S, int r0, int r1, cudaMemcpyKind kind,
                       cudaStream_t s) {
    const size_t off = (size_t)r0 * row, pitch = (size_t)S * row;
    return cudaMemcpy2DAsync(static_cast<char*>(dst) + off, pitch, static_cast<const char*>(src) + off, pitch,
                             (size_t)(r1 - r0) * row, B, kind, s);
  };
  cudaEvent_t* ev_in = hp->ev;                    // chunk inputs on the device
  cudaEvent_t* ev_out = hp->ev + kMaxHostChunks;  // chunk outputs computed
  cudaEvent_t ev_start = hp->ev[2 * kMaxHostChunks], ev_done = hp->ev[2 * kMaxHostChunks + 1];
  // the device copies may still be in use by earlier work in `stream`
  if (cudaEventRecord(ev_start, stm) != cudaSuccess || cudaStreamWaitEvent(hp->h2d, ev_start, 0) != cudaSuccess)
    return SDPA_ERR_CUDA;
  // K and V go up first, whole (one copy each: every copy command costs the copy engine a few
  // microseconds, and the total time of the upward copies, not their order, sets the pace);
  // then Q chunk by chunk
  if (cudaMemcpyAsync(dk, k, (size_t)B * Sk * krow, cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess ||
      cudaMemcpyAsync(dv, v, (size_t)B * Sk * vrow, cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess)
    return SDPA_ERR_CUDA;
  for (int i = 0; i < n_chunks; ++i) {
    // causal: the last rows first.  Their chunk is the longest to compute, so it now overlaps
    // the later uploads, and the pipeline ends on the cheapest chunk.
    const int c = causal ? n_chunks - 1 - i : i;
    const int r0 = c * rows, r1 = std::min(Sq, r0 + rows);
    // causal (top-left): rows r0..r1-1 see keys below r1; otherwise every key
    const int k_need = causal ? std::min(Sk, r1) : Sk;
    if (copy_rows(dq, q, qrow, Sq, r0, r1, cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess) return SDPA_ERR_CUDA;
    if (cudaEventRecord(ev_in[c], hp->h2d) != cudaSuccess || cudaStreamWaitEvent(stm, ev_in[c], 0) != cudaSuccess)
      return SDPA_ERR_CUDA;
    const int rc = fwd_common(dq + (size_t)r0 * qrow, dk, dv, dO + (size_t)r0 * orow, lse ? dl + r0 : nullptr, B, Hq,
                              Hkv, r1 - r0, std::max(k_need, 1), D, Dv, st, scale, causal, nullptr, nullptr,
                              ws + L.total, workspace_bytes - L.total, in_dtype == SDPA_BF16 ? kBF16 : kF16, 1.f, 1.f,
                              1.f, out_dtype, stream, nullptr, nullptr, causal ? r0 : 0, Sq);
    if (rc != SDPA_OK) return rc;
    if (cudaEventRecord(ev_out[c], stm) != cudaSuccess || cudaStreamWaitEvent(hp->d2h, ev_out[c], 0) != cudaSuccess)
      return SDPA_ERR_CUDA;
    if (copy_rows(o, dO, orow, Sq, r0, r1, cudaMemcpyDeviceToHost, hp->d2h) != cudaSuccess) return SDPA_ERR_CUDA;
  }
  if (lse && cudaMemcpyAsync(lse, dl, (size_t)B * Hq * Sq * 4, cudaMemcpyDeviceToHost, hp->d2h) != cudaSuccess)
    return SDPA_ERR_CUDA;
  if (cudaEventRecord(ev_done, hp->d2h) != cudaSuccess || cudaStreamWaitEvent(stm, ev_done, 0) != cudaSuccess)
    return SDPA_ERR_CUDA;
  return SDPA_OK;
}

size_t sdpa_decode_workspace_size(int B, int Hq, int max_kv, int Dv) {
  if (B < 1 || Hq < 1 || max_kv < 1 || Dv < 1) return 0;
  return decode_partials_bytes(B, Hq, max_kv, Dv);
}

int sdpa_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_len, void* o, float* lse,
                int B, int Hq, int Hkv, int max_kv, int D, int Dv, const int64_t* strides, float scale,
                void* workspace, size_t workspace_bytes, sdpa_dtype dtype, void* stream) {
  DecodeCall call;
  const int rc = decode_check(q, k_cache, v_cache, nullptr, kv_len, o, lse, B, Hq, Hkv, max_kv, 0, 0, 0, D, Dv,
                              strides, scale, dtype, &call);
  if (rc != SDPA_OK) return rc;
  if (!workspace || !aligned16(workspace) || workspace_bytes < decode_partials_bytes(B, Hq, max_kv, Dv))
    return SDPA_ERR_INVALID;
  return decode_launch(call, static_cast<float*>(workspace), static_cast<cudaStream_t>(stream));
}

int sdpa_decode_paged(const void* q, const void* k_pool, const void* v_pool, const int32_t* page_table,
                      const int32_t* kv_len, void* o, float* lse, int B, int Hq, int Hkv, int page_size, int max_pages,
                      int n_pages, int D, int Dv, const int64_t* strides, float scale, void* workspace,
                      size_t workspace_bytes, sdpa_dtype dtype, void* stream) {
  if (!page_table) return SDPA_ERR_INVALID;
  if (page_size < 1 || max_pages < 1 || n_pages < 1) return SDPA_ERR_INVALID;
  const long long max_kv_ll = (long long)max_pages * page_size;
  if (max_kv_ll > (1ll << 30)) return SDPA_ERR_UNSUPPORTED;
  const int max_kv = (int)max_kv_ll;
  DecodeCall call;
  const int rc = decode_check(q, k_pool, v_pool, page_table, kv_len, o, lse, B, Hq, Hkv, max_kv, page_size,
                              max_pages, n_pages, D, Dv, strides, scale, dtype, &call);
  if (rc != SDPA_OK) return rc;
  if (!workspace || !aligned16(workspace) || workspace_bytes < decode_partials_bytes(B, Hq, max_kv, Dv))
    return SDPA_ERR_INVALID;
  return decode_launch(call, static_cast<float*>(workspace), static_cast<cudaStream_t>(stream));
}

int sdpa_check_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SDPA_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)) != cudaSuccess) return SDPA_ERR_CUDA;
  if (word == 0) return SDPA_OK;
  const uint32_t zero = 0;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return SDPA_ERR_CUDA;
  if (word & kStatusTimeout) return SDPA_ERR_TIMEOUT;
  return (word & kStatusBadSeqlens) ? SDPA_ERR_INVALID : SDPA_ERR_CUDA;
}

const char* sdpa_status_string(int status) {
  switch (status) {
    case SDPA_OK: return "SDPA_OK";
    case SDPA_ERR_INVALID: return "SDPA_ERR_INVALID";
    case SDPA_ERR_UNSUPPORTED: return "SDPA_ERR_UNSUPPORTED";
    case SDPA_ERR_CUDA: return "SDPA_ERR_CUDA";
    case SDPA_ERR_TIMEOUT: return "SDPA_ERR_TIMEOUT";
    default: return "SDPA_ERR_UNKNOWN";
  }
}

int sdpa_version(void) { return 100; }

int sdpa_debug_stall_next_call(void) {
  g_stall_next.store(1);
  return SDPA_OK;
}

}  // extern "C"
