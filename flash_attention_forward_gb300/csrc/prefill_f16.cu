// Prefill instances for f16 inputs: (D, Dv) in {(64, 64), (128, 128), (192, 128)} x causal x
// (mask, packed sequences or neither), plus the int8-code instances (D = Dv in {64, 128}, per-block
// score scales).
#include "prefill_launch.cuh"

namespace sdpa {

cudaError_t launch_prefill_f16(int D, int Dv, bool causal, bool has_mask, const CUtensorMap& tq,
                               const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to, const PrefillParams& p, cudaStream_t st,
                               bool* supported) {
  *supported = true;
  if (D == 64 && Dv == 64) return launch_prefill_dims<kF16, 64, 64>(causal, has_mask, tq, tk, tv, to, p, st);
  if (D == 128 && Dv == 128) return launch_prefill_dims<kF16, 128, 128>(causal, has_mask, tq, tk, tv, to, p, st);
  if (D == 192 && Dv == 128) return launch_prefill_dims<kF16, 192, 128>(causal, has_mask, tq, tk, tv, to, p, st);
  *supported = false;
  return cudaSuccess;
}

cudaError_t launch_prefill_f16_block_scaled(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                      const CUtensorMap& tv, const CUtensorMap& to, const PrefillParams& p, cudaStream_t st,
                                      bool* supported) {
  *supported = true;
  if (D == 64) return launch_prefill_block_scaled<kF16, 64>(causal, tq, tk, tv, to, p, st);
  if (D == 128) return launch_prefill_block_scaled<kF16, 128>(causal, tq, tk, tv, to, p, st);
  *supported = false;
  return cudaSuccess;
}

}  // namespace sdpa
