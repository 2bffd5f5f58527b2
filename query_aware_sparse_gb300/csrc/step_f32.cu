// Fused decode step instantiated for fp32 K/V/q with fp32 summaries.
#include "step_impl.cuh"

namespace quest {

cudaError_t launch_step_f32(const StepArgs& a, const StepPlan& p, cudaStream_t s) {
  return a.head_dim == 128 ? launch_s<float, 128, false>(a, p, s) : launch_s<float, 64, false>(a, p, s);
}

void shape_step_f32(int dev, int head_dim, int page_size, int group, int* smem, int* per_sm) {
  if (head_dim == 128) shape_s<float, 128, false>(dev, page_size, group, smem, per_sm);
  else shape_s<float, 64, false>(dev, page_size, group, smem, per_sm);
}

}  // namespace quest
