// Cluster decode step instantiated for fp16 K/V/q with E4M3 summary codes, head dim 64
// (page sizes 16 and 32, GQA groups 1, 2, 4 and 8; one file per variant and head
// dim, so the instantiations compile in parallel).
#include "cstep_impl.cuh"

namespace quest {

cudaError_t launch_cstep_e4m3_d64(const StepArgs& a, const StepPlan& p, cudaStream_t s) {
  return cstep_launch_sg<__half, 64, true>(a, p, s);
}

int clusters_cstep_e4m3_d64(int dev, int page_size, int group) {
  return cstep_clusters_sg<__half, 64, true>(dev, page_size, group);
}

}  // namespace quest
