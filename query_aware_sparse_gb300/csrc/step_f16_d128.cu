// Fused decode step instantiated for fp16 K/V/q with fp16 summaries, head dim 128
// (one file per variant and head dim, so the instantiations compile in parallel).
#include "step_impl.cuh"

namespace quest {

cudaError_t launch_step_f16_d128(const StepArgs& a, const StepPlan& p, cudaStream_t s) {
  return launch_s<__half, 128, false>(a, p, s);
}

void shape_step_f16_d128(int dev, int page_size, int group, int* smem, int* per_sm) {
  shape_s<__half, 128, false>(dev, page_size, group, smem, per_sm);
}

}  // namespace quest
