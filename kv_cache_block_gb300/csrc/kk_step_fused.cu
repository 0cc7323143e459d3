// The decode step with the decode token's append fused in
// (kk_step_options.k_new): the instantiations of the step kernel that carry
// it (kk_step.cuh), in a translation unit of their own.
#include "kk_step.cuh"

namespace kk {

cudaError_t launch_step_fused(const StepParams& p, cudaStream_t s) {
  if (p.bt.R == 0) return cudaSuccess;
  const bool bf16 = p.kc.dtype == 1;
  switch (p.D) {
    case 32: return bf16 ? launch_typed<bf16_t, 32, true>(p, s) : launch_typed<float, 32, true>(p, s);
    case 64: return bf16 ? launch_typed<bf16_t, 64, true>(p, s) : launch_typed<float, 64, true>(p, s);
    case 128: return bf16 ? launch_typed<bf16_t, 128, true>(p, s) : launch_typed<float, 128, true>(p, s);
    case 256: return bf16 ? launch_typed<bf16_t, 256, true>(p, s) : cudaErrorInvalidValue;  // fp32 rows of 1 KB
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kk
