// Split-K sparse decode attention for callers that cannot allocate device
// memory: the same kernels as quest_sparse_decode_attn, with the split-K
// partials kept in a fixed buffer that lives in this library's own module
// memory instead of in a caller-provided workspace.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

// Largest split-K partial area this entry point can use (4 MiB).
constexpr size_t kNoAllocScratchBytes = 4u << 20;

// The scratch itself: one copy per device that loads the library, held until
// the process exits. Host code must not pass this name to a kernel (on the
// host it is only a stand-in); it passes the address from cudaGetSymbolAddress.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
float* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch on the current device; looked up once per
// device, with that device current, on the first call made on it.
float* scratch_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" QUEST_API quest_status quest_sparse_decode_attn_noalloc(
    const quest_cache* cache, const quest_pages* pages, const void* q, int32_t group,
    const int32_t* sel_logical, const int32_t* sel_phys, int32_t k, float* out, float* lse,
    float sm_scale, void* stream) {
  // the same checks, in the same order, as quest_sparse_decode_attn
  quest_status st = quest::check_cache(cache);
  if (st != QUEST_OK) return st;
  if ((st = quest::check_pages(pages, true)) != QUEST_OK) return st;
  if (!quest::valid_group(group) || k < 1) return QUEST_ERR_INVALID_ARG;
  if (!quest::attn_supported(cache->dtype, cache->head_dim, cache->page_size, group))
    return QUEST_ERR_UNSUPPORTED;
  if (pages->batch == 0) return QUEST_OK;
  if (!q || !sel_logical || !sel_phys || !out || !quest::aligned16(q)) return QUEST_ERR_INVALID_ARG;
  const quest::AttnPlan plan = quest::plan_attn(pages->batch, cache->h_kv, group,
                                                cache->head_dim, cache->page_size, cache->dtype, k);
  if (plan.workspace_bytes > kNoAllocScratchBytes) return QUEST_ERR_WORKSPACE;   // too large
  float* scratch = scratch_ptr();
  if (!scratch) return QUEST_ERR_CUDA;
  quest::AttnArgs a{};
  a.q = q; a.k_pool = cache->k_pool; a.v_pool = cache->v_pool;
  a.sel_logical = sel_logical; a.sel_phys = sel_phys; a.seq_lens = pages->seq_lens;
  a.out = out; a.lse = lse;
  // Every partial row the combine reads is written by the split kernel of the
  // same call, so nothing in the scratch has to start at zero.
  const size_t rows = (size_t)pages->batch * cache->h_kv * group * plan.n_chunks;
  a.part_o = scratch;
  a.part_ml = scratch + rows * cache->head_dim;
  a.batch = pages->batch; a.n_phys = cache->n_phys; a.h_kv = cache->h_kv; a.group = group;
  a.page_size = cache->page_size; a.head_dim = cache->head_dim; a.dtype = cache->dtype;
  a.k = k; a.n_chunks = plan.n_chunks; a.chunk_pages = plan.chunk_pages;
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf((float)cache->head_dim);
  a.scale_log2 = scale * quest::LOG2E;
  a.err = quest::error_word_ptr();
  if (!a.err) return QUEST_ERR_CUDA;
  return quest::launch_attn(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? QUEST_OK
                                                                                  : QUEST_ERR_CUDA;
}
