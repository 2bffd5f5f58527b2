// Plan and dispatch of the fused decode step (the kernel is in
// step_impl.cuh; the step_<variant>_d<head_dim>.cu files instantiate it per
// element type, summary format and head dim, so they compile in parallel).
// Including the kernel's header instantiates nothing here: its templates
// are only instantiated by the variant files.
#include <cstdlib>

#include "step_impl.cuh"

namespace quest {

namespace {

// The cluster kernel (cstep_impl.cuh) for shapes it is built for: units of
// the batch spread evenly over the clusters the device keeps resident. It
// uses no workspace (the size returned is a token 256 bytes).
StepPlan plan_cstep(int32_t batch, int32_t h_kv, int32_t group, int32_t head_dim,
                    int32_t page_size, int32_t dtype, int32_t summary_fp8) {
  StepPlan p{};
  // groups of 4 and 8 only with fp16 K/V (their attention runs on the warp MMA)
  const bool g_ok = group == 1 || group == 2 || ((group == 4 || group == 8) && dtype == QUEST_F16);
  if (!g_ok || (head_dim != 64 && head_dim != 128) || (page_size != 16 && page_size != 32))
    return p;
  if (summary_fp8 && dtype != QUEST_F16) return p;
  if (getenv("QUEST_STEP_LEGACY")) return p;     // the grid-wide kernel instead (comparisons)
  int dev = 0, maxc = 32;                         // no device (sizing only): a default part
  if (cudaGetDevice(&dev) == cudaSuccess) {
    const bool d128 = head_dim == 128;
    if (dtype == QUEST_F16 && summary_fp8)
      maxc = d128 ? clusters_cstep_e4m3_d128(dev, page_size, group) : clusters_cstep_e4m3_d64(dev, page_size, group);
    else if (dtype == QUEST_F16)
      maxc = d128 ? clusters_cstep_f16_d128(dev, page_size, group) : clusters_cstep_f16_d64(dev, page_size, group);
    else
      maxc = d128 ? clusters_cstep_f32_d128(dev, page_size, group) : clusters_cstep_f32_d64(dev, page_size, group);
  }
  cudaGetLastError();
  if (maxc <= 0) return p;
  const long long units = (long long)batch * h_kv;
  const long long per = (units + maxc - 1) / maxc;
  if (per > kCStepUnitsPerCluster) return p;
  // every resident cluster takes units (their counts differ by at most one;
  // the kernel deals them out longest request first)
  long long nc = units < maxc ? units : maxc;
  if (nc < 1) nc = 1;
  if (const char* e = getenv("QUEST_STEP_CLUSTERS")) {   // cluster count override (experiments)
    const long long want = atoll(e);
    if (want > 0 && want <= maxc && (units + want - 1) / want <= kCStepUnitsPerCluster) nc = want;
  }
  p.ok = true;
  p.cluster = true;
  p.grid = (int32_t)(nc * 4);
  p.workspace_bytes = 256;
  return p;
}

}  // namespace

StepPlan plan_step(int32_t batch, int32_t nnz, int32_t h_kv, int32_t group, int32_t head_dim,
                   int32_t page_size, int32_t dtype, int32_t k, int32_t summary_fp8) {
  {
    StepPlan c = plan_cstep(batch, h_kv, group, head_dim, page_size, dtype, summary_fp8);
    if (c.ok) return c;
  }
  StepPlan p{};
  int smem = 0, per_sm = 0, dev = 0, sms = 148;
  const bool have_dev = cudaGetDevice(&dev) == cudaSuccess &&
                        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
  cudaGetLastError();
  if (have_dev) {
    const bool d128 = head_dim == 128;
    if (dtype == QUEST_F16 && summary_fp8) {
      if (d128) shape_step_e4m3_d128(dev, page_size, group, &smem, &per_sm);
      else shape_step_e4m3_d64(dev, page_size, group, &smem, &per_sm);
    } else if (dtype == QUEST_F16) {
      if (d128) shape_step_f16_d128(dev, page_size, group, &smem, &per_sm);
      else shape_step_f16_d64(dev, page_size, group, &smem, &per_sm);
    } else {
      if (d128) shape_step_f32_d128(dev, page_size, group, &smem, &per_sm);
      else shape_step_f32_d64(dev, page_size, group, &smem, &per_sm);
    }
  } else {
    per_sm = 1;   // no device (sizing only): one CTA per SM of a default part
  }
  const long long units = (long long)batch * h_kv;
  p.smem = smem;
  p.grid = sms * (per_sm > 2 ? 2 : per_sm);
  p.ok = per_sm >= 1 && smem <= 227 * 1024 && p.grid > 0;
  // partial slots per unit: worker CTAs whose round share can overlap one unit
  long long np = 1;
  const int rounds = units < kRounds ? (int)units : kRounds;
  const int workers = p.grid > 0 ? p.grid - select_ctas((int)units, p.grid) : 0;
  for (int q = 0; q < rounds && workers > 0; ++q) {
    const long long k0 = q * units / rounds, k1 = (q + 1) * units / rounds;
    const long long len = (k1 - k0) * k;
    long long n;
    if (k1 - k0 <= workers) {                  // a group of workers per unit
      n = (workers + (k1 - k0) - 1) / (k1 - k0);
    } else {
      const long long minlen = len / workers;
      n = minlen == 0 ? workers : (k + minlen - 1) / minlen + 1;
    }
    np = n > np ? n : np;
  }
  if (np > workers) np = workers > 0 ? workers : 1;
  p.chunk_pages = 0;
  p.n_chunks = (int32_t)np;
  p.counters_bytes = ((size_t)(4 + 2 * units) * sizeof(unsigned) + 255) & ~(size_t)255;
  p.tagged_bytes = ((size_t)h_kv * nnz * sizeof(unsigned long long) + 255) & ~(size_t)255;
  const size_t rows = (size_t)units * group * p.n_chunks;
  p.workspace_bytes = p.counters_bytes + p.tagged_bytes + rows * head_dim * sizeof(float) +
                      rows * 4 * sizeof(float);
  p.workspace_bytes = (p.workspace_bytes + 255) & ~(size_t)255;
  return p;
}

cudaError_t launch_step(const StepArgs& a, const StepPlan& p, cudaStream_t s) {
  const bool d128 = a.head_dim == 128;
  if (p.cluster) {
    if (a.dtype == QUEST_F16 && a.summary_fp8)
      return d128 ? launch_cstep_e4m3_d128(a, p, s) : launch_cstep_e4m3_d64(a, p, s);
    if (a.dtype == QUEST_F16) return d128 ? launch_cstep_f16_d128(a, p, s) : launch_cstep_f16_d64(a, p, s);
    return d128 ? launch_cstep_f32_d128(a, p, s) : launch_cstep_f32_d64(a, p, s);
  }
  if (a.dtype == QUEST_F16 && a.summary_fp8)
    return d128 ? launch_step_e4m3_d128(a, p, s) : launch_step_e4m3_d64(a, p, s);
  if (a.dtype == QUEST_F16) return d128 ? launch_step_f16_d128(a, p, s) : launch_step_f16_d64(a, p, s);
  return d128 ? launch_step_f32_d128(a, p, s) : launch_step_f32_d64(a, p, s);
}

}  // namespace quest
