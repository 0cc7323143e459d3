// One decode step of the Key-Key selector (the kernel is in kk_step.cuh):
// the host-side sizes of its workspace and its launch.
#include "kk_step.cuh"

namespace kk {

int step_hier_level_cap(int D) { return kStage * D / 2; }

int step_split_cap(int max_blocks, int K) {
  const int Kp = K <= 1 ? 1 : 1 << (32 - __builtin_clz(K - 1));
  int cap = std::min(kMergeSlots / Kp, kMaxSplits);
  cap = std::min(cap, max_blocks / kSplitMinBlocks);
  return cap >= 2 ? cap : 0;
}

size_t step_workspace_bytes(int R, int max_blocks, int K) {
  const int cap = step_split_cap(max_blocks, K);
  if (cap == 0 || R <= 0) return 0;
  const int Kp = K <= 1 ? 1 : 1 << (32 - __builtin_clz(K - 1));
  const size_t words = ((size_t)R * sizeof(unsigned long long) + 255) & ~size_t(255);
  return words + (size_t)R * cap * Kp * sizeof(uint64_t);
}

cudaError_t launch_step(const StepParams& p, cudaStream_t s) {
  if (p.bt.R == 0) return cudaSuccess;
  if (p.k_new) return launch_step_fused(p, s);
  const bool bf16 = (p.flags & kStepAnchor) && p.kc.dtype == 1;
#define KK_STEP_CASE(DD) \
  if (p.D == DD) return bf16 ? launch_typed<bf16_t, DD, false>(p, s) : launch_typed<float, DD, false>(p, s);
  KK_STEP_CASE(32)
  KK_STEP_CASE(64)
  KK_STEP_CASE(128)
  KK_STEP_CASE(256)
#undef KK_STEP_CASE
  return cudaErrorInvalidValue;
}

}  // namespace kk
