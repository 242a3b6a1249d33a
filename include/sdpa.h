/*
 * sdpa.h -- C ABI of the GB300 (sm_103a) scaled-dot-product-attention forward library.
 *
 * What every prefill entry point computes, per batch b, query head h and query row i
 * (page "Xe SDPA Forward Mainloop", sections "Full simplified pseudocode" and
 * "softmax() helper"; GQA head mapping from page "Xe2 ESIMD Flash Attention - SDP
 * Prefill & Decode", section "GQA layout"):
 *
 *     kvh        = h / (Hq / Hkv)
 *     s[j]       = scale * dot(Q[b,i,h,:], K[b,j,kvh,:]) + mask[b,i,j]      (mask optional)
 *     s[j]       = -inf  if causal and j > i                                 (top-left causal)
 *     O[b,i,h,:] = sum_j softmax(s)[j] * V[b,j,kvh,:]
 *     LSE[b,h,i] = ln sum_j exp(s[j])
 *
 * computed block by block with the online softmax (row max m, rescale of the running O
 * and l, exp2 with scale*log2(e) folded in, row sum l).  A row whose keys are all
 * masked (every s[j] = -inf) yields O = 0 and LSE = -inf, never NaN (page "Xe2 ESIMD
 * Flash Attention", section "Correctness testing", names that row as the usual NaN
 * source).  K/V lengths need not be multiples of any block size (same page, section
 * "kv_len alignment").
 *
 * Conventions shared by all entry points
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library never
 *    frees or retains them.  Scalars and stride arrays are HOST values.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL is the
 *    legacy default stream).  The return value reports argument validation and launch
 *    errors only.  Errors detected on the device (a bounded wait that gave up) are
 *    reported by sdpa_check_device_status().
 *  - Element strides are in ELEMENTS, not bytes; the innermost (head-dim) stride is 1.
 *  - Validation happens before any CUDA call; an invalid call launches nothing.
 *  - The library allocates no device memory in these entry points.  Decode and masked
 *    prefill take a caller workspace sized by the *_workspace_size functions.
 *  - sdpa_fwd, sdpa_fwd_fp8, sdpa_fwd_varlen*, sdpa_fwd_int8, sdpa_decode and
 *    sdpa_decode_paged may be recorded into a CUDA graph (stream capture) once a first call on
 *    the device has run outside the capture; sdpa_fwd_host may not.
 */
#ifndef SDPA_GB300_H
#define SDPA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SDPA_OK = 0,
  SDPA_ERR_INVALID = 1,     /* bad argument: null pointer, non-positive size, Hq % Hkv != 0, bad scale */
  SDPA_ERR_UNSUPPORTED = 2, /* valid but not built: head dims, dtypes, alignment, strides */
  SDPA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch, tensor-map encode) */
  SDPA_ERR_TIMEOUT = 4      /* a kernel's bounded wait gave up (see sdpa_check_device_status) */
} sdpa_status;

typedef enum { SDPA_F16 = 0, SDPA_BF16 = 1, SDPA_E4M3 = 2, SDPA_I8 = 3 } sdpa_dtype;

/* Number of int64 entries in the prefill stride array. */
#define SDPA_FWD_NSTRIDES 12
/* Number of int64 entries in the decode stride array. */
#define SDPA_DECODE_NSTRIDES 10
/* Number of int64 entries in the paged-decode stride array. */
#define SDPA_DECODE_PAGED_NSTRIDES 11

/*
 * sdpa_fwd_workspace_size -- bytes of device scratch sdpa_fwd / sdpa_fwd_fp8 use, for the
 * current device (the SM count enters the second part).  Two parts, in this order:
 *  1. with an additive mask (has_mask != 0): the mask condensed into one bit per (row, key)
 *     marking -inf entries plus one flag per (row, 128-key block) marking blocks that hold
 *     finite non-zero values.  Required: a masked call with less workspace is rejected.
 *  2. without causal masking, when the work tiles of 2 x 128 query rows do not divide evenly
 *     over the SMs: partial results of the last, partial round of tiles, whose key range is
 *     split over the otherwise idle SMs (unnormalised fp32 O, row max and row sum per part);
 *     a second kernel in the same stream merges them with log-sum-exp weights.  Optional:
 *     with less workspace the call runs unsplit; results agree within rounding.
 * Zero when neither applies.  Sizes below 1 give 0.
 */
size_t sdpa_fwd_workspace_size(int B, int Hq, int Sq, int Sk, int Dv, int causal, int has_mask);

/*
 * sdpa_fwd -- fused attention prefill, fp16 or bf16 inputs, fp32 softmax state.
 *
 *   q    [B, Sq, Hq, D]      in_dtype         k [B, Sk, Hkv, D]   in_dtype
 *   v    [B, Sk, Hkv, Dv]    in_dtype         o [B, Sq, Hq, Dv]   out_dtype (written)
 *   lse  [B, Hq, Sq] fp32 contiguous, natural log; may be NULL (then not written)
 *   strides: NULL for the contiguous layouts above, else 12 element strides
 *            {q_b, q_s, q_h,  k_b, k_s, k_h,  v_b, v_s, v_h,  o_b, o_s, o_h}
 *   scale:   > 0 and finite (the softmax temperature; 1/sqrt(D) is customary)
 *   causal:  nonzero -> key j visible to query i iff j <= i (top-left aligned)
 *   mask:    NULL, or fp16 additive mask indexed [b, i, j], shared by all heads, added
 *            after scaling; element strides mask_strides = {m_b, m_i} (NULL means
 *            {Sq*Sk, Sk}; m_b may be 0 to broadcast over the batch).  Only 2-byte
 *            alignment is required.
 *   workspace: device scratch, 16-byte aligned, contents on entry irrelevant: at least the
 *            mask part of sdpa_fwd_workspace_size(B, Hq, Sq, Sk, Dv, causal, mask!=0) when
 *            mask != NULL; the full size enables the split of the last round of tiles.
 *            May be NULL when mask is NULL.  Calls that overlap on the GPU need separate
 *            workspaces.
 *   in_dtype: SDPA_F16 or SDPA_BF16.  out_dtype: SDPA_F16 or SDPA_BF16.
 *
 * Supported head dims: (D, Dv) in {(64, 64), (128, 128), (192, 128)} (D = 192 keeps one K/V stage
 * in shared memory next to two 48 KB Q tiles, so its loads do not overlap its MMAs).  q/k/v/o base pointers must be
 * 16-byte aligned and their s/h/b strides multiples of 8 elements (tensor-memory-access
 * descriptor rule); otherwise SDPA_ERR_UNSUPPORTED.  Sizes: B, Hq, Hkv, Sq, Sk >= 1.
 */
int sdpa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
             int Sk, int D, int Dv, const int64_t* strides, float scale, int causal, const void* mask,
             const int64_t* mask_strides, void* workspace, size_t workspace_bytes, sdpa_dtype in_dtype,
             sdpa_dtype out_dtype, void* stream);

/*
 * sdpa_fwd_fp8 -- the same prefill with FP8 e4m3 Q/K/V codes and per-tensor fp32 scales
 * (Q = q_code * descale_q, likewise K and V; host floats).  Q K^T runs on e4m3 tensor
 * cores with fp32 accumulation, the descales folded into the softmax scale; P and V
 * meet in fp16 (every e4m3 value is exact in fp16) with fp32 accumulation; O is
 * multiplied by descale_v in the epilogue.  (page "MlaMmaOp", struct summary: the
 * MLA prefill path streams FP8 e4m3 K/V with D != Dv.)
 *
 * Supported head dims: (D, Dv) in {(64, 64), (128, 128), (192, 128)}.  q/k/v strides must be
 * multiples of 16 elements.  out_dtype: SDPA_BF16.  Other arguments as in sdpa_fwd.
 */
int sdpa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
                 int Sk, int D, int Dv, const int64_t* strides, float scale, int causal, const void* mask,
                 const int64_t* mask_strides, void* workspace, size_t workspace_bytes, float descale_q,
                 float descale_k, float descale_v, sdpa_dtype out_dtype, void* stream);

/* Number of int64 entries in the packed (varlen) prefill stride array. */
#define SDPA_FWD_VARLEN_NSTRIDES 8

/*
 * sdpa_fwd_varlen_workspace_size -- bytes of device scratch sdpa_fwd_varlen /
 * sdpa_fwd_varlen_fp8 need for B sequences: the per-sequence work-tile prefix,
 * round_up((B + 1) * 4, 16).  0 for B < 1.
 */
size_t sdpa_fwd_varlen_workspace_size(int B);

/*
 * sdpa_fwd_varlen -- the prefill of sdpa_fwd over B sequences of different lengths packed
 * back to back (page "Xe SDPA Forward Mainloop", section "SageV1 concrete instance": the
 * run-time variant selects a variable-length template parameter).  Sequence b owns query
 * rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key/value rows cu_seqlens_k[b] ..
 * cu_seqlens_k[b+1]-1; it attends to its own keys only, and causal masking is top-left
 * aligned within each sequence (key j visible to query i iff j <= i, both counted from the
 * sequence's first row).  A sequence with queries but no keys gets O = 0, LSE = -inf.
 *
 *   q    [total_q, Hq, D]     in_dtype         k [total_k, Hkv, D]   in_dtype
 *   v    [total_k, Hkv, Dv]   in_dtype         o [total_q, Hq, Dv]   out_dtype (written
 *                                               for the rows some sequence owns)
 *   lse  [Hq, total_q] fp32 contiguous, natural log; may be NULL
 *   cu_seqlens_q, cu_seqlens_k: DEVICE int32 [B + 1], 4-byte aligned, non-decreasing, first
 *            entry >= 0, last entry <= total_q (total_k).  Read on the device: offsets that
 *            break these rules make the call store nothing and raise a status that
 *            sdpa_check_device_status() reports as SDPA_ERR_INVALID.
 *   max_seqlen_q: >= every cu_seqlens_q[b+1] - cu_seqlens_q[b] and <= total_q (it sizes
 *            the launch; a longer sequence is reported like bad offsets).
 *   strides: NULL for the contiguous layouts above, else 8 element strides
 *            {q_s, q_h,  k_s, k_h,  v_s, v_h,  o_s, o_h} (row and head; head dim stride 1)
 *   workspace: device scratch of sdpa_fwd_varlen_workspace_size(B) bytes, 16-byte aligned;
 *            required.  Calls that overlap on the GPU need separate workspaces.
 *   scale, causal, head dims, dtypes, alignment and stride rules: as in sdpa_fwd.
 * No additive mask; B, Hq, Hkv, total_q, total_k, max_seqlen_q >= 1.  Two kernels run in
 * `stream`: a one-block scan of the per-sequence tile counts, then the prefill.
 */
int sdpa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens_q,
                    const int32_t* cu_seqlens_k, int B, int Hq, int Hkv, int total_q, int total_k, int max_seqlen_q,
                    int D, int Dv, const int64_t* strides, float scale, int causal, void* workspace,
                    size_t workspace_bytes, sdpa_dtype in_dtype, sdpa_dtype out_dtype, void* stream);

/*
 * sdpa_fwd_varlen_fp8 -- sdpa_fwd_varlen with FP8 e4m3 Q/K/V codes and per-tensor scales,
 * computed as in sdpa_fwd_fp8.  out_dtype: SDPA_BF16.
 */
int sdpa_fwd_varlen_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B, int Hq, int Hkv, int total_q,
                        int total_k, int max_seqlen_q, int D, int Dv, const int64_t* strides, float scale, int causal,
                        void* workspace, size_t workspace_bytes, float descale_q, float descale_k, float descale_v,
                        sdpa_dtype out_dtype, void* stream);

/*
 * sdpa_fwd_host_workspace_size -- bytes of device scratch sdpa_fwd_host needs: device copies of
 * Q, K, V, O and LSE (contiguous, each rounded up to 16 bytes), then the optional split partials
 * of one chunk (see sdpa_fwd_workspace_size).  Sizes below 1 give 0.
 */
size_t sdpa_fwd_host_workspace_size(int B, int Hq, int Hkv, int Sq, int Sk, int D, int Dv, int causal);

/*
 * sdpa_fwd_host -- sdpa_fwd on HOST buffers: copies the inputs to the device, computes, and
 * copies O (and LSE) back, overlapping the three.  K and V go up first on a copy stream, then
 * Q in at most 8 chunks of whole 256-row work tiles (causal: the last rows first, so that the
 * most expensive chunk overlaps the remaining uploads); a chunk's prefill runs in `stream` as
 * soon as its rows have landed (over the keys those rows see, causal masking counted from the
 * chunk's global row), and its O rows come back on a second copy stream while later chunks are
 * still copying or computing.  Results equal sdpa_fwd's on the same inputs (causal: bit for bit).
 *
 *   q, k, v, o, lse: HOST pointers, contiguous [B, Sq, Hq, D], [B, Sk, Hkv, D], [B, Sk, Hkv, Dv],
 *            [B, Sq, Hq, Dv], [B, Hq, Sq] fp32 (lse may be NULL).  Page-locked (pinned) memory is
 *            needed for the copies to overlap; pageable memory works but serialises them.
 *   workspace: DEVICE scratch of sdpa_fwd_host_workspace_size(...) bytes, 16-byte aligned.
 *   in_dtype = out_dtype: SDPA_F16 or SDPA_BF16.  Head dims, scale, causal: as in sdpa_fwd.
 * Asynchronous: when the call returns, `stream` has been made to wait for the last copy back,
 * so synchronizing `stream` makes o and lse readable.  The two copy streams and their events
 * are created on the first call on a device (make that call outside stream capture) and kept
 * until the process exits; concurrent calls on one device are serialised while they enqueue
 * and share the copy streams.  On SDPA_ERR_CUDA part of the work may already be enqueued.
 */
int sdpa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
                  int Sk, int D, int Dv, float scale, int causal, void* workspace, size_t workspace_bytes,
                  sdpa_dtype in_dtype, sdpa_dtype out_dtype, void* stream);

/*
 * sdpa_fwd_int8_workspace_size -- bytes of device scratch sdpa_fwd_int8 needs: the 16-bit copies
 * of the int8 operands (Q and K, plus V when v_int8 != 0; B*S*H*D*2 bytes each, rounded up to 16)
 * followed by the optional split partials described under sdpa_fwd_workspace_size.  Sizes below
 * 1 give 0.
 */
size_t sdpa_fwd_int8_workspace_size(int B, int Hq, int Hkv, int Sq, int Sk, int D, int v_int8, int causal);

/*
 * sdpa_fwd_int8 -- prefill with int8 Q/K codes and per-block scales (page "Xe SDPA Forward
 * Mainloop", section "SageV1 concrete instance": the SageV1 prefill takes its Q/K dtype, a P.V
 * dtype, scale pointers and a use_int8_pv switch, and has launchers for head dims 64 and 128).
 * With Q = q_code * q_scale[b, h, i / 128] and K = k_code * k_scale[b, kvh, j / 128]:
 *
 *     s[j] = scale * q_scale[b,h,i/128] * k_scale[b,kvh,j/128] * dot(q_code[b,i,h,:], k_code[b,j,kvh,:])
 *
 * then softmax, O and LSE as in sdpa_fwd.  V is either 16-bit values (v_dtype == out_dtype) or
 * int8 codes (v_dtype == SDPA_I8) with per-channel scales: V[b,j,kvh,c] = v_code * v_scale[b,kvh,c].
 * sm_103a has no int8 tensor-core MMA, so a first kernel copies the codes into 16-bit form (exact)
 * in the workspace and the prefill multiplies them on the 16-bit tensor cores; the integer dot
 * products are exact in the fp32 accumulator (|sum| < 2^24), so the scores equal an int32
 * accumulation times the scales.  P is rounded to out_dtype; the v_scale factor multiplies the
 * accumulated O columns.
 *
 *   q [B, Sq, Hq, D] int8    k [B, Sk, Hkv, D] int8    v [B, Sk, Hkv, D] int8 or out_dtype
 *   o [B, Sq, Hq, D] out_dtype; lse [B, Hq, Sq] fp32 or NULL
 *   strides: NULL or the 12 element strides of sdpa_fwd; int8 strides multiples of 16 elements,
 *            16-bit strides multiples of 8; q, k (and int8 v) 16-byte aligned
 *   q_scale  DEVICE fp32 [B, Hq, ceil(Sq / 128)], contiguous; k_scale DEVICE fp32 [B, Hkv,
 *            ceil(Sk / 128)], contiguous; both 4-byte aligned; positive finite values expected
 *   v_scale  DEVICE fp32 [B, Hkv, D], contiguous, 16-byte aligned, when v_dtype == SDPA_I8; else NULL
 *   workspace: at least the copy part of sdpa_fwd_int8_workspace_size(...), 16-byte aligned
 *   D = Dv in {64, 128}; out_dtype SDPA_F16 or SDPA_BF16 (the copies and P use that type); no
 *   additive mask.  Other arguments as in sdpa_fwd.  Two kernels run in `stream` (the copy, then
 *   the prefill; plus the split merge when it applies).
 */
int sdpa_fwd_int8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
                  int Sk, int D, const int64_t* strides, const float* q_scale, const float* k_scale,
                  const float* v_scale, float scale, int causal, void* workspace, size_t workspace_bytes,
                  sdpa_dtype v_dtype, sdpa_dtype out_dtype, void* stream);

/*
 * sdpa_decode_workspace_size -- bytes of device scratch sdpa_decode needs for per-split
 * partial results (unnormalised O, running max, running sum) of every (b, q-head, split).
 */
size_t sdpa_decode_workspace_size(int B, int Hq, int max_kv, int Dv);

/*
 * sdpa_decode -- two-phase split-KV decode: one query token per (b, query head) against
 * the first kv_len[b] rows of a padded K/V cache.  Phase 1 gives every (b, kv head,
 * split of keys) a partial (O, m, l); phase 2 merges the splits of a (b, q head) with a
 * log-sum-exp combine.  Cache rows at or beyond kv_len[b] never contribute (they may hold
 * anything, NaN included); keys stream in 64-row chunks, so up to 63 such rows may be read,
 * never past max_kv.
 * (page "Xe2 ESIMD Flash Attention", section "Assets": two-phase full-dense decode)
 *
 *   q       [B, Hq, D]                 dtype            o   [B, Hq, Dv]  dtype (written)
 *   k_cache [B, max_kv, Hkv, D]        dtype            lse [B, Hq] fp32 contiguous or NULL
 *   v_cache [B, max_kv, Hkv, Dv]       dtype
 *   kv_len  [B] int32, DEVICE pointer, each in [0, max_kv]; kv_len[b] = 0 gives O = 0,
 *           LSE = -inf.  Values outside [0, max_kv] are clamped into it on the device.
 *   strides: NULL for the layouts above, else 10 element strides
 *            {q_b, q_h,  k_b, k_s, k_h,  v_b, v_s, v_h,  o_b, o_h}
 *   workspace: at least sdpa_decode_workspace_size(B, Hq, max_kv, Dv) bytes, 16-byte
 *           aligned, device memory; its contents on entry do not matter.
 *   dtype:  SDPA_F16 or SDPA_BF16.
 *
 * Supported: (D, Dv) in {(128, 128), (192, 128)} (the second is the MLA head shape of page
 * "MlaMmaOp"); 1 <= Hq/Hkv <= 16 (all query heads of a KV head share one 16-row tensor-core tile,
 * so every K/V byte is read once; section "GQA layout" of the Xe2 page leaves the group size
 * open); B <= 65535 and Hkv <= 65535 (launch-grid limits); pointers 16-byte
 * aligned; s/h/b strides multiples of 8 elements.  Otherwise SDPA_ERR_UNSUPPORTED.
 */
int sdpa_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_len, void* o, float* lse,
                int B, int Hq, int Hkv, int max_kv, int D, int Dv, const int64_t* strides, float scale,
                void* workspace, size_t workspace_bytes, sdpa_dtype dtype, void* stream);

/*
 * sdpa_decode_paged -- sdpa_decode over a paged K/V cache: key row t of sequence b is row
 * t % page_size of physical page page_table[b][t / page_size] of a shared page pool.  The pages
 * leave the layout of a cache to a page table (page "Xe SDPA Forward Mainloop", section
 * "Arguments / params": an optional page table, page size and pages per sequence are runtime
 * arguments of the mainloop); the arithmetic is sdpa_decode's, chunk for chunk, so a paged cache
 * holding the same rows as a contiguous one gives the same result.
 *
 *   k_pool, v_pool [n_pages, page_size, Hkv, D | Dv]  dtype, device
 *   page_table [B, max_pages] int32, DEVICE pointer: physical page of each logical page.  Entries
 *           for pages at or past ceil(kv_len[b] / page_size) are never used for a visible key; any
 *           value there (or outside [0, n_pages)) is harmless: such rows read as zeros or are masked.
 *   kv_len  [B] int32, device; clamped into [0, max_pages * page_size].
 *   page_size: a power of two >= 16.
 *   strides: NULL for the layouts above, else 11 element strides
 *            {q_b, q_h,  k_page, k_row, k_h,  v_page, v_row, v_h,  o_b, o_h,  page_table row}
 *   workspace: at least sdpa_decode_workspace_size(B, Hq, max_pages * page_size, Dv) bytes.
 *   Other arguments, limits and results as in sdpa_decode; a page-table row stride below
 *   max_pages or a page_size that is not a power of two is SDPA_ERR_INVALID, a page_size below
 *   16 SDPA_ERR_UNSUPPORTED.
 */
int sdpa_decode_paged(const void* q, const void* k_pool, const void* v_pool, const int32_t* page_table,
                      const int32_t* kv_len, void* o, float* lse, int B, int Hq, int Hkv, int page_size, int max_pages,
                      int n_pages, int D, int Dv, const int64_t* strides, float scale, void* workspace,
                      size_t workspace_bytes, sdpa_dtype dtype, void* stream);

/*
 * sdpa_decode_noalloc -- sdpa_decode for callers that cannot allocate device memory: runtimes
 * without a device allocator of their own, hosts that hand out device memory only through
 * their own pool and forbid library allocations, and serving loops that must not call
 * cudaMalloc on the hot path (it can synchronize the device).  The pages this library follows
 * have no counterpart for it.
 *
 * Arguments and results are those of sdpa_decode without the workspace: the per-split
 * partials go to a fixed 32 MiB array in the library's own device memory, which every GPU
 * that loads the library holds until the process exits.  A call that would need more
 * (B * Hq * ceil(max_kv / 2048) * (Dv + 2) * 4 bytes > 32 MiB) returns SDPA_ERR_UNSUPPORTED
 * and launches nothing.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before any stream
 * capture.  All calls on a device share the array and it keeps the last call's contents
 * (the decode rewrites every partial it reads, so nothing needs clearing); calls whose
 * kernels overlap on the GPU race on it.  No cudaMalloc, cudaFree or allocating library
 * routine is called.
 */
int sdpa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_len, void* o,
                        float* lse, int B, int Hq, int Hkv, int max_kv, int D, int Dv, const int64_t* strides,
                        float scale, sdpa_dtype dtype, void* stream);

/*
 * sdpa_check_device_status -- synchronizes `stream`, then reports and clears the device
 * status word the kernels raise when a bounded wait inside them gives up (a pipeline
 * stage that never arrived): SDPA_ERR_TIMEOUT in that case, SDPA_ERR_INVALID when a varlen
 * call found bad sequence offsets, SDPA_ERR_CUDA if the synchronization itself failed, else
 * SDPA_OK.  The status word is per device and per
 * process, shared by all streams.
 */
int sdpa_check_device_status(void* stream);

/* Human-readable name of a status code (static string). */
const char* sdpa_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int sdpa_version(void);

/*
 * sdpa_debug_stall_next_call -- test hook for the failure path.  Arms a one-shot flag
 * (process-wide): the next prefill launch (of any sdpa_fwd* entry point) withholds its first K/V stage, so
 * every CTA's bounded waits give up after about one second, the CTAs drain their copies,
 * free tensor memory and exit, and sdpa_check_device_status() then returns
 * SDPA_ERR_TIMEOUT.  The CUDA context stays usable.  Returns SDPA_OK.  Nothing in the
 * library calls it.
 */
int sdpa_debug_stall_next_call(void);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_GB300_H */
