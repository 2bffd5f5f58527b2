// C ABI of libquest: host-side validation, the device error word and the
// dispatch to the kernel files. No torch types, no allocation.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

// The device error word: one per device that loads the library, living in
// the module's global memory (no allocation). Kernels receive its address.
__device__ unsigned int quest_device_error_word;

namespace {

using quest::AttnPlan;

constexpr int kMaxDevices = 64;
unsigned* g_err_ptr[kMaxDevices] = {};
std::mutex g_err_mu;

// Device address of the error word for the current device (set-up once per
// device, with that device current).
unsigned* err_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, quest_device_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_err_ptr[dev];
}

using quest::aligned16;
using quest::check_cache;
using quest::check_pages;
using quest::valid_group;

unsigned long long* g_trace = nullptr;      // quest_set_trace buffer (device)
int32_t g_trace_ctas = 0;
// quest_test_step_fault: fault mode and wait limit of later calls
std::atomic<int32_t> g_test_fault{0};
std::atomic<uint32_t> g_wait_limit{quest::kStepWaitLimit};

quest_status launched(cudaError_t e) { return e == cudaSuccess ? QUEST_OK : QUEST_ERR_CUDA; }

}  // namespace

extern "C" {

quest_status quest_append_kv(const quest_cache* cache, const quest_pages* pages,
                             const void* k_new, const void* v_new, int32_t n_new,
                             const int32_t* append_indptr,
                             const int32_t* seq_lens_before, void* stream) {
  quest_status st = check_cache(cache);
  if (st != QUEST_OK) return st;
  if ((st = check_pages(pages, false)) != QUEST_OK) return st;
  if (n_new < 0) return QUEST_ERR_INVALID_ARG;
  if (pages->batch == 0 || n_new == 0) return QUEST_OK;
  if (!k_new || !v_new || !append_indptr || !seq_lens_before) return QUEST_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return QUEST_ERR_INVALID_ARG;
  quest::AppendArgs a{};
  a.k_pool = cache->k_pool; a.v_pool = cache->v_pool; a.summary = cache->summary;
  a.k_new = k_new; a.v_new = v_new;
  a.page_indptr = pages->page_indptr; a.page_indices = pages->page_indices;
  a.append_indptr = append_indptr; a.seq_lens_before = seq_lens_before;
  a.batch = pages->batch; a.n_new = n_new; a.n_phys = cache->n_phys; a.h_kv = cache->h_kv;
  a.page_size = cache->page_size; a.head_dim = cache->head_dim; a.dtype = cache->dtype;
  a.summary_fp8 = cache->summary_fp8;
  a.err = err_ptr();
  if (!a.err) return QUEST_ERR_CUDA;
  return launched(quest::launch_append(a, static_cast<cudaStream_t>(stream)));
}

quest_status quest_score_pages(const quest_cache* cache, const quest_pages* pages,
                               const void* q, int32_t group, float* scores,
                               void* stream) {
  quest_status st = check_cache(cache);
  if (st != QUEST_OK) return st;
  if ((st = check_pages(pages, true)) != QUEST_OK) return st;
  if (!valid_group(group)) return QUEST_ERR_UNSUPPORTED;
  if (!quest::score_supported(cache->dtype, cache->head_dim, group)) return QUEST_ERR_UNSUPPORTED;
  if (pages->batch == 0 || pages->nnz == 0) return QUEST_OK;
  if (!q || !scores || !aligned16(q)) return QUEST_ERR_INVALID_ARG;
  quest::ScoreArgs a{};
  a.summary = cache->summary; a.q = q;
  a.page_indptr = pages->page_indptr; a.page_indices = pages->page_indices;
  a.seq_lens = pages->seq_lens; a.scores = scores;
  a.batch = pages->batch; a.nnz = pages->nnz; a.n_phys = cache->n_phys; a.h_kv = cache->h_kv;
  a.group = group; a.page_size = cache->page_size; a.head_dim = cache->head_dim;
  a.dtype = cache->dtype; a.summary_fp8 = cache->summary_fp8;
  a.err = err_ptr();
  if (!a.err) return QUEST_ERR_CUDA;
  return launched(quest::launch_score(a, static_cast<cudaStream_t>(stream)));
}

quest_status quest_score_pages_per_head(const quest_cache* cache, const quest_pages* pages,
                                        const void* q, int32_t group, float* scores,
                                        void* stream) {
  quest_status st = check_cache(cache);
  if (st != QUEST_OK) return st;
  if ((st = check_pages(pages, true)) != QUEST_OK) return st;
  if (!valid_group(group)) return QUEST_ERR_UNSUPPORTED;
  if (!quest::score_supported(cache->dtype, cache->head_dim, group)) return QUEST_ERR_UNSUPPORTED;
  if (pages->batch == 0 || pages->nnz == 0) return QUEST_OK;
  if (!q || !scores || !aligned16(q)) return QUEST_ERR_INVALID_ARG;
  quest::ScoreArgs a{};
  a.summary = cache->summary; a.q = q;
  a.page_indptr = pages->page_indptr; a.page_indices = pages->page_indices;
  a.seq_lens = pages->seq_lens; a.scores = scores; a.per_head = 1;
  a.batch = pages->batch; a.nnz = pages->nnz; a.n_phys = cache->n_phys; a.h_kv = cache->h_kv;
  a.group = group; a.page_size = cache->page_size; a.head_dim = cache->head_dim;
  a.dtype = cache->dtype; a.summary_fp8 = cache->summary_fp8;
  a.err = err_ptr();
  if (!a.err) return QUEST_ERR_CUDA;
  return launched(quest::launch_score(a, static_cast<cudaStream_t>(stream)));
}

quest_status quest_select_topk(const quest_pages* pages, int32_t h_kv,
                               int32_t page_size, const float* scores, int32_t k,
                               int32_t n_sink, int32_t n_local,
                               int32_t* sel_logical, int32_t* sel_phys,
                               int32_t* sel_count, void* stream) {
  quest_status st = check_pages(pages, true);
  if (st != QUEST_OK) return st;
  if (h_kv <= 0 || k < 1) return QUEST_ERR_INVALID_ARG;
  if (n_sink < 0 || n_local < 0 || (int64_t)n_sink + n_local > k) return QUEST_ERR_INVALID_ARG;
  if (page_size != 16 && page_size != 32) return QUEST_ERR_UNSUPPORTED;
  if (pages->batch == 0) return QUEST_OK;
  if ((!scores && pages->nnz > 0) || !sel_logical || !sel_phys || !sel_count)
    return QUEST_ERR_INVALID_ARG;
  quest::SelectArgs a{};
  a.scores = scores;
  a.page_indptr = pages->page_indptr; a.page_indices = pages->page_indices;
  a.seq_lens = pages->seq_lens;
  a.sel_logical = sel_logical; a.sel_phys = sel_phys; a.sel_count = sel_count;
  a.batch = pages->batch; a.nnz = pages->nnz; a.h_kv = h_kv; a.k = k;
  a.page_size = page_size;
  a.n_sink = n_sink; a.n_local = n_local;
  a.err = err_ptr();
  if (!a.err) return QUEST_ERR_CUDA;
  return launched(quest::launch_select(a, static_cast<cudaStream_t>(stream)));
}

size_t quest_attn_workspace_size(int32_t batch, int32_t h_kv, int32_t group,
                                 int32_t head_dim, int32_t page_size, int32_t k) {
  if (batch <= 0 || h_kv <= 0 || k < 1 || !valid_group(group)) return 0;
  // the plan does not depend on the element type beyond shared memory per
  // CTA; take the larger (fp32) footprint so one size serves both types
  AttnPlan p16 = quest::plan_attn(batch, h_kv, group, head_dim, page_size, QUEST_F16, k);
  AttnPlan p32 = quest::plan_attn(batch, h_kv, group, head_dim, page_size, QUEST_F32, k);
  return p16.workspace_bytes > p32.workspace_bytes ? p16.workspace_bytes : p32.workspace_bytes;
}

quest_status quest_sparse_decode_attn(const quest_cache* cache,
                                      const quest_pages* pages, const void* q,
                                      int32_t group, const int32_t* sel_logical,
                                      const int32_t* sel_phys, int32_t k,
                                      float* out, float* lse, float sm_scale,
                                      void* workspace, size_t workspace_bytes,
                                      void* stream) {
  quest_status st = check_cache(cache);
  if (st != QUEST_OK) return st;
  if ((st = check_pages(pages, true)) != QUEST_OK) return st;
  if (!valid_group(group) || k < 1) return QUEST_ERR_INVALID_ARG;
  if (!quest::attn_supported(cache->dtype, cache->head_dim, cache->page_size, group))
    return QUEST_ERR_UNSUPPORTED;
  if (pages->batch == 0) return QUEST_OK;
  if (!q || !sel_logical || !sel_phys || !out || !aligned16(q)) return QUEST_ERR_INVALID_ARG;
  AttnPlan plan = quest::plan_attn(pages->batch, cache->h_kv, group, cache->head_dim,
                                   cache->page_size, cache->dtype, k);
  if (!workspace || workspace_bytes < plan.workspace_bytes || !aligned16(workspace))
    return QUEST_ERR_WORKSPACE;
  quest::AttnArgs a{};
  a.q = q; a.k_pool = cache->k_pool; a.v_pool = cache->v_pool;
  a.sel_logical = sel_logical; a.sel_phys = sel_phys; a.seq_lens = pages->seq_lens;
  a.out = out; a.lse = lse;
  const size_t rows = (size_t)pages->batch * cache->h_kv * group * plan.n_chunks;
  a.part_o = static_cast<float*>(workspace);
  a.part_ml = a.part_o + rows * cache->head_dim;
  a.batch = pages->batch; a.n_phys = cache->n_phys; a.h_kv = cache->h_kv; a.group = group;
  a.page_size = cache->page_size; a.head_dim = cache->head_dim; a.dtype = cache->dtype;
  a.k = k; a.n_chunks = plan.n_chunks; a.chunk_pages = plan.chunk_pages;
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf((float)cache->head_dim);
  a.scale_log2 = scale * quest::LOG2E;
  a.err = err_ptr();
  if (!a.err) return QUEST_ERR_CUDA;
  return launched(quest::launch_attn(a, static_cast<cudaStream_t>(stream)));
}

size_t quest_union_workspace_size(int32_t batch, int32_t h_kv, int32_t group, int32_t head_dim,
                                  int32_t page_size, int32_t dtype, int32_t k) {
  if (batch <= 0 || h_kv <= 0 || k < 1 || !valid_group(group)) return 0;
  if (!quest::attn_supported(dtype, head_dim, page_size, group)) return 0;
  const int64_t ku = (int64_t)group * k;
  if (ku > INT32_MAX) return 0;
  AttnPlan plan = quest::plan_attn(batch, h_kv, group, head_dim, page_size, dtype, (int32_t)ku);
  const size_t phys = ((size_t)batch * h_kv * ku * sizeof(int32_t) + 255) & ~(size_t)255;
  return phys + plan.workspace_bytes;
}

quest_status quest_union_decode_attn(const quest_cache* cache, const quest_pages* pages,
                                     const void* q, int32_t group, const int32_t* sel_logical,
                                     int32_t k, float* out, float* lse, float sm_scale,
                                     int32_t* union_logical, uint8_t* union_mask,
                                     int32_t* union_count, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  quest_status st = check_cache(cache);
  if (st != QUEST_OK) return st;
  if ((st = check_pages(pages, true)) != QUEST_OK) return st;
  if (!valid_group(group) || k < 1) return QUEST_ERR_INVALID_ARG;
  if (!quest::attn_supported(cache->dtype, cache->head_dim, cache->page_size, group))
    return QUEST_ERR_UNSUPPORTED;
  if ((int64_t)group * k > INT32_MAX) return QUEST_ERR_INVALID_ARG;
  if (pages->batch == 0) return QUEST_OK;
  if (!q || !sel_logical || !out || !union_logical || !union_mask || !union_count ||
      !aligned16(q))
    return QUEST_ERR_INVALID_ARG;
  const int32_t ku = group * k;
  AttnPlan plan = quest::plan_attn(pages->batch, cache->h_kv, group, cache->head_dim,
                                   cache->page_size, cache->dtype, ku);
  const size_t phys_bytes = ((size_t)pages->batch * cache->h_kv * ku * sizeof(int32_t) + 255) &
                            ~(size_t)255;
  if (!workspace || workspace_bytes < phys_bytes + plan.workspace_bytes || !aligned16(workspace))
    return QUEST_ERR_WORKSPACE;
  unsigned* err = err_ptr();
  if (!err) return QUEST_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* u_phys = static_cast<int32_t*>(workspace);
  quest::UnionArgs u{};
  u.sel_logical = sel_logical;
  u.page_indptr = pages->page_indptr; u.page_indices = pages->page_indices;
  u.seq_lens = pages->seq_lens;
  u.u_logical = union_logical; u.u_phys = u_phys; u.u_mask = union_mask; u.u_count = union_count;
  u.batch = pages->batch; u.h_kv = cache->h_kv; u.group = group; u.k = k;
  u.page_size = cache->page_size;
  u.max_pages = pages->nnz < quest::kUnionMaxPages ? pages->nnz : quest::kUnionMaxPages;
  u.err = err;
  cudaError_t e = quest::launch_union(u, s);
  if (e != cudaSuccess) return QUEST_ERR_CUDA;
  quest::AttnArgs a{};
  a.q = q; a.k_pool = cache->k_pool; a.v_pool = cache->v_pool;
  a.sel_logical = union_logical; a.sel_phys = u_phys; a.sel_mask = union_mask;
  a.seq_lens = pages->seq_lens;
  a.out = out; a.lse = lse;
  const size_t rows = (size_t)pages->batch * cache->h_kv * group * plan.n_chunks;
  a.part_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + phys_bytes);
  a.part_ml = a.part_o + rows * cache->head_dim;
  a.batch = pages->batch; a.n_phys = cache->n_phys; a.h_kv = cache->h_kv; a.group = group;
  a.page_size = cache->page_size; a.head_dim = cache->head_dim; a.dtype = cache->dtype;
  a.k = ku; a.n_chunks = plan.n_chunks; a.chunk_pages = plan.chunk_pages;
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf((float)cache->head_dim);
  a.scale_log2 = scale * quest::LOG2E;
  a.err = err;
  return launched(quest::launch_attn(a, s));
}

size_t quest_decode_workspace_size(int32_t batch, int32_t nnz, int32_t h_kv, int32_t group,
                                   int32_t head_dim, int32_t page_size, int32_t dtype,
                                   int32_t k) {
  if (batch <= 0 || nnz < 0 || h_kv <= 0 || k < 1 || !valid_group(group)) return 0;
  if ((dtype != QUEST_F16 && dtype != QUEST_F32) || (head_dim != 64 && head_dim != 128) ||
      (page_size != 16 && page_size != 32))
    return 0;
  // the E4M3-summary variant of the kernel may plan another grid: size for both
  quest::StepPlan p = quest::plan_step(batch, nnz, h_kv, group, head_dim, page_size, dtype, k, 0);
  size_t need = p.ok ? p.workspace_bytes : 0;
  if (dtype == QUEST_F16) {
    quest::StepPlan p8 = quest::plan_step(batch, nnz, h_kv, group, head_dim, page_size, dtype, k, 1);
    if (p8.ok && p8.workspace_bytes > need) need = p8.workspace_bytes;
  }
  return need;
}

int32_t quest_decode_step_kernel(int32_t batch, int32_t h_kv, int32_t group, int32_t head_dim,
                                 int32_t page_size, int32_t dtype, int32_t k, int32_t summary_fp8) {
  if (batch <= 0 || h_kv <= 0 || k < 1 || !valid_group(group)) return 0;
  if ((dtype != QUEST_F16 && dtype != QUEST_F32) || (head_dim != 64 && head_dim != 128) ||
      (page_size != 16 && page_size != 32) || (summary_fp8 != 0 && summary_fp8 != 1) ||
      (summary_fp8 && dtype != QUEST_F16))
    return 0;
  quest::StepPlan p = quest::plan_step(batch, 0, h_kv, group, head_dim, page_size, dtype, k,
                                       summary_fp8);
  return p.ok ? (p.cluster ? 2 : 1) : 0;
}

quest_status quest_decode_step(const quest_cache* cache, const quest_pages* pages,
                               const void* k_new, const void* v_new, const void* q,
                               int32_t group, int32_t k, int32_t n_sink, int32_t n_local,
                               float* scores,
                               int32_t* sel_logical, int32_t* sel_phys, int32_t* sel_count,
                               float* out, float* lse, float sm_scale, void* workspace,
                               size_t workspace_bytes, void* stream) {
  quest_status st = check_cache(cache);
  if (st != QUEST_OK) return st;
  if ((st = check_pages(pages, true)) != QUEST_OK) return st;
  if (!valid_group(group)) return QUEST_ERR_UNSUPPORTED;
  if (k < 1) return QUEST_ERR_INVALID_ARG;
  if (n_sink < 0 || n_local < 0 || (int64_t)n_sink + n_local > k) return QUEST_ERR_INVALID_ARG;
  if (pages->batch == 0) return QUEST_OK;
  if (!q || !scores || !sel_logical || !sel_phys || !sel_count || !out || !aligned16(q))
    return QUEST_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return QUEST_ERR_INVALID_ARG;
  if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return QUEST_ERR_INVALID_ARG;
  quest::StepPlan plan = quest::plan_step(pages->batch, pages->nnz, cache->h_kv, group,
                                          cache->head_dim, cache->page_size, cache->dtype, k,
                                          cache->summary_fp8);
  if (!plan.ok) return QUEST_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < plan.workspace_bytes || !aligned16(workspace))
    return QUEST_ERR_WORKSPACE;
  quest::StepArgs a{};
  a.k_pool = cache->k_pool; a.v_pool = cache->v_pool; a.summary = cache->summary;
  a.k_new = k_new; a.v_new = v_new; a.q = q;
  a.page_indptr = pages->page_indptr; a.page_indices = pages->page_indices;
  a.seq_lens = pages->seq_lens;
  a.scores = scores; a.sel_logical = sel_logical; a.sel_phys = sel_phys; a.sel_count = sel_count;
  a.out = out; a.lse = lse;
  a.counters = static_cast<unsigned*>(workspace);
  a.tagged = reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) +
                                                   plan.counters_bytes);
  const size_t rows = (size_t)pages->batch * cache->h_kv * group * plan.n_chunks;
  a.part_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.counters_bytes +
                                      plan.tagged_bytes);
  a.part_ml = a.part_o + rows * cache->head_dim;
  a.batch = pages->batch; a.nnz = pages->nnz; a.n_phys = cache->n_phys; a.h_kv = cache->h_kv;
  a.group = group; a.page_size = cache->page_size; a.head_dim = cache->head_dim;
  a.dtype = cache->dtype; a.k = k; a.n_chunks = plan.n_chunks; a.chunk_pages = plan.chunk_pages;
  a.summary_fp8 = cache->summary_fp8;
  a.n_sink = n_sink; a.n_local = n_local;
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf((float)cache->head_dim);
  a.scale_log2 = scale * quest::LOG2E;
  a.trace = (g_trace && plan.grid <= g_trace_ctas) ? g_trace : nullptr;
  a.err = err_ptr();
  if (!a.err) return QUEST_ERR_CUDA;
  a.wait_limit = g_wait_limit.load();
  a.test_fault = g_test_fault.load() == 1 ? 1 : 0;
  return launched(quest::launch_step(a, plan, static_cast<cudaStream_t>(stream)));
}

size_t quest_diag_workspace_size(int32_t h_kv, int32_t group, int32_t nnz, int32_t page_size) {
  if (h_kv <= 0 || nnz < 0 || !valid_group(group) || (page_size != 16 && page_size != 32)) return 0;
  return quest::diag_workspace_bytes(h_kv, group, nnz, page_size);
}

quest_status quest_recall_diagnostics(const quest_cache* cache, const quest_pages* pages,
                                      const void* q, int32_t group, const int32_t* sel_logical,
                                      int32_t k, int32_t top_r, float sm_scale, float* slack,
                                      float* eps, float* topr, float* vmax, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  quest_status st = check_cache(cache);
  if (st != QUEST_OK) return st;
  if ((st = check_pages(pages, true)) != QUEST_OK) return st;
  if (!valid_group(group) || cache->summary_fp8) return QUEST_ERR_UNSUPPORTED;
  if (k < 1 || top_r < 1) return QUEST_ERR_INVALID_ARG;
  if (pages->batch == 0) return QUEST_OK;
  if (!q || !sel_logical || !slack || !eps || !topr || !vmax || !aligned16(q))
    return QUEST_ERR_INVALID_ARG;
  const size_t need = quest::diag_workspace_bytes(cache->h_kv, group, pages->nnz, cache->page_size);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return QUEST_ERR_WORKSPACE;
  quest::DiagArgs a{};
  a.k_pool = cache->k_pool; a.v_pool = cache->v_pool; a.summary = cache->summary; a.q = q;
  a.page_indptr = pages->page_indptr; a.page_indices = pages->page_indices;
  a.seq_lens = pages->seq_lens; a.sel_logical = sel_logical;
  a.slack = slack; a.eps = eps; a.topr = topr; a.vmax = vmax;
  a.batch = pages->batch; a.nnz = pages->nnz; a.n_phys = cache->n_phys; a.h_kv = cache->h_kv;
  a.group = group; a.page_size = cache->page_size; a.head_dim = cache->head_dim;
  a.dtype = cache->dtype; a.k = k; a.top_r = top_r;
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf((float)cache->head_dim);
  a.scale_log2 = scale * quest::LOG2E;
  quest::diag_carve(a, workspace);
  a.err = err_ptr();
  if (!a.err) return QUEST_ERR_CUDA;
  return launched(quest::launch_diag(a, static_cast<cudaStream_t>(stream)));
}

int32_t quest_set_trace(void* device_buffer, int32_t max_ctas, int32_t batch, int32_t h_kv,
                        int32_t group, int32_t head_dim, int32_t page_size, int32_t dtype,
                        int32_t k) {
  g_trace = static_cast<unsigned long long*>(device_buffer);
  g_trace_ctas = device_buffer ? max_ctas : 0;
  if (batch <= 0 || h_kv <= 0 || k < 1 || !valid_group(group)) return 0;
  quest::StepPlan p = quest::plan_step(batch, 0, h_kv, group, head_dim, page_size, dtype, k, 0);
  return p.ok ? p.grid : 0;
}

int32_t quest_get_device_error(void* stream) {
  unsigned* p = err_ptr();
  if (!p) return -1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  const unsigned zero = 0;
  if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return -1;
  return (int32_t)v;
}

const char* quest_status_string(int32_t status) {
  switch (status) {
    case QUEST_OK: return "QUEST_OK";
    case QUEST_ERR_INVALID_ARG: return "QUEST_ERR_INVALID_ARG: null pointer, bad size or misaligned pointer";
    case QUEST_ERR_UNSUPPORTED: return "QUEST_ERR_UNSUPPORTED: dtype, head_dim, page_size or group not supported";
    case QUEST_ERR_WORKSPACE: return "QUEST_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case QUEST_ERR_CUDA: return "QUEST_ERR_CUDA: a CUDA call or kernel launch failed";
  }
  return "unknown quest_status";
}

int32_t quest_test_step_fault(int32_t mode, int32_t wait_limit) {
  if (mode < 0 || mode > 2 || wait_limit < 0) return QUEST_ERR_INVALID_ARG;
  g_test_fault = mode;
  g_wait_limit = wait_limit > 0 ? (uint32_t)wait_limit : quest::kStepWaitLimit;
  return QUEST_OK;
}

}  // extern "C"

namespace quest {
unsigned* error_word_ptr() { return err_ptr(); }
int32_t test_fault_mode() { return g_test_fault.load(); }
uint32_t wait_limit() { return g_wait_limit.load(); }
}  // namespace quest
