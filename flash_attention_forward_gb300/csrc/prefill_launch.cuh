// Host-side launch of one prefill kernel instance.
#pragma once

#include "prefill.cuh"

namespace sdpa {

template <int ELEM, int D, int DV, bool CAUSAL, bool MASK, int VAR>
cudaError_t launch_prefill_instance(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                                    const PrefillParams& p, cudaStream_t st) {
  using C = PrefillCfg<ELEM, D, DV>;
  auto kern = prefill_kernel<ELEM, D, DV, CAUSAL, MASK, VAR>;
  // persistent: one CTA per SM (shared memory admits no second one), looping over work units
  int dev = 0, sms = 0;
  cudaError_t e = current_device_sms(&dev, &sms);
  if (e != cudaSuccess) return e;
  // the shared-memory opt-in is per device and made once
  static std::atomic<uint64_t> opted{0};
  if ((e = smem_opt_in(kern, C::SMEM, dev, opted)) != cudaSuccess) return e;
  const long long units = p.n_units;
  const unsigned grid = (unsigned)(units < sms ? units : sms);
  // Group KV units so that a group is a whole number of snake round pairs (2 x grid work
  // tiles; the snake balances inside it) and its K/V stays within a 64 MiB share of L2.
  PrefillParams q = p;
  const long long per_unit = (long long)p.n_cta_tiles * p.group;
  const long long two_rounds = 2LL * grid;
  long long a = per_unit, b = two_rounds;
  while (b) { const long long t = a % b; a = b; b = t; }          // gcd(per_unit, 2 x grid)
  const long long aligned = two_rounds / a;
  const long long kv_unit_bytes = (long long)p.Sk * (D * C::ESZ + DV * C::ESZ);
  const long long cap = (64LL << 20) / (kv_unit_bytes > 0 ? kv_unit_bytes : 1);
  long long ug = aligned < cap ? aligned : cap;
  const long long kv_units = (long long)p.B * p.Hkv;
  q.units_per_group = (int)(ug < 1 ? 1 : (ug > kv_units ? kv_units : ug));
  {
    const long long G = p.group, upg = q.units_per_group;
    const long long last_units = kv_units - (kv_units - 1) / upg * upg;  // units of the last group
    q.div_gsize = make_fastdiv((uint32_t)(upg * G * p.n_cta_tiles));
    q.div_band = make_fastdiv((uint32_t)(upg * G));
    q.div_band_last = make_fastdiv((uint32_t)(last_units * G));
    q.div_group = make_fastdiv((uint32_t)G);
    q.div_heads = make_fastdiv((uint32_t)(VAR == kVarlen ? p.Hq : p.Hkv));
  }
  // Programmatic dependent launch where the previous kernel of the stream is this library's own:
  // the masked prefill after mask_convert_kernel (only its softmax reads what that kernel
  // writes, after griddepcontrol.wait), and the split merge after the prefill.
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  if constexpr (MASK) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPrefillThreads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, to, q)) != cudaSuccess) return e;
  } else {
    kern<<<grid, kPrefillThreads, C::SMEM, st>>>(tq, tk, tv, to, q);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (!CAUSAL && VAR != kVarlen && p.split_parts > 1) {
    const long long threads = (long long)p.split_tail * kCtaRows * (DV / 8);
    cudaLaunchConfig_t ccfg = {};
    ccfg.gridDim = dim3((unsigned)((threads + 127) / 128));
    ccfg.blockDim = dim3(128);
    ccfg.stream = st;
    ccfg.attrs = pdl;
    ccfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&ccfg, split_combine_kernel<ELEM == kE4M3 ? kBF16 : ELEM, DV>, q)) != cudaSuccess)
      return e;
  }
  return cudaGetLastError();
}

template <int ELEM, int D, int DV>
cudaError_t launch_prefill_dims(bool causal, bool has_mask, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& to, const PrefillParams& p, cudaStream_t st) {
  if (p.varlen)  // packed sequences: no mask, no split tail
    return causal ? launch_prefill_instance<ELEM, D, DV, true, false, kVarlen>(tq, tk, tv, to, p, st)
                  : launch_prefill_instance<ELEM, D, DV, false, false, kVarlen>(tq, tk, tv, to, p, st);
  if (causal)
    return has_mask ? launch_prefill_instance<ELEM, D, DV, true, true, kDense>(tq, tk, tv, to, p, st)
                    : launch_prefill_instance<ELEM, D, DV, true, false, kDense>(tq, tk, tv, to, p, st);
  return has_mask ? launch_prefill_instance<ELEM, D, DV, false, true, kDense>(tq, tk, tv, to, p, st)
                  : launch_prefill_instance<ELEM, D, DV, false, false, kDense>(tq, tk, tv, to, p, st);
}

// int8 codes widened to 16 bits (Q/K/V already in the 16-bit type), per-block score scales.
template <int ELEM, int D>
cudaError_t launch_prefill_block_scaled(bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                        const CUtensorMap& tv, const CUtensorMap& to, const PrefillParams& p, cudaStream_t st) {
  return causal ? launch_prefill_instance<ELEM, D, D, true, false, kBlockScaled>(tq, tk, tv, to, p, st)
                : launch_prefill_instance<ELEM, D, D, false, false, kBlockScaled>(tq, tk, tv, to, p, st);
}

}  // namespace sdpa
