// Host-side launch interfaces between the C-ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include <atomic>
#include <stdint.h>

#include "../../include/quest.h"

namespace quest {

// Argument checks shared by the entry points (quest_api.cu, noalloc.cu).
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline quest_status check_cache(const quest_cache* c) {
  if (!c || !c->k_pool || !c->v_pool || !c->summary) return QUEST_ERR_INVALID_ARG;
  if (c->n_phys <= 0 || c->h_kv <= 0) return QUEST_ERR_INVALID_ARG;
  if (c->dtype != QUEST_F16 && c->dtype != QUEST_F32) return QUEST_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return QUEST_ERR_UNSUPPORTED;
  if (c->page_size != 16 && c->page_size != 32) return QUEST_ERR_UNSUPPORTED;
  if (c->summary_fp8 != 0 && c->summary_fp8 != 1) return QUEST_ERR_INVALID_ARG;
  if (c->summary_fp8 && c->dtype != QUEST_F16) return QUEST_ERR_UNSUPPORTED;
  if (!aligned16(c->k_pool) || !aligned16(c->v_pool) || !aligned16(c->summary))
    return QUEST_ERR_INVALID_ARG;
  return QUEST_OK;
}

inline quest_status check_pages(const quest_pages* p, bool need_seq_lens) {
  if (!p || p->batch < 0 || p->nnz < 0) return QUEST_ERR_INVALID_ARG;
  if (p->batch == 0) return QUEST_OK;
  if (!p->page_indptr || (p->nnz > 0 && !p->page_indices)) return QUEST_ERR_INVALID_ARG;
  if (need_seq_lens && !p->seq_lens) return QUEST_ERR_INVALID_ARG;
  return QUEST_OK;
}

inline bool valid_group(int32_t g) { return g == 1 || g == 2 || g == 4 || g == 8; }

// quest_test_step_fault's state: the fault mode (0 none, 1 a wait of the
// cluster step runs out, 2 a wait of the attention split kernel runs out)
// and the tries of every bounded in-kernel wait.
int32_t test_fault_mode();
uint32_t wait_limit();

struct AppendArgs {
  void* k_pool; void* v_pool; void* summary;
  const void* k_new; const void* v_new;
  const int32_t* page_indptr; const int32_t* page_indices;
  const int32_t* append_indptr; const int32_t* seq_lens_before;
  int32_t batch, n_new, n_phys, h_kv, page_size, head_dim, dtype;
  int32_t summary_fp8;                        // summary holds E4M3 codes
  unsigned* err;
};

struct ScoreArgs {
  const void* summary; const void* q;
  const int32_t* page_indptr; const int32_t* page_indices; const int32_t* seq_lens;
  float* scores;                              // [h_kv, nnz], or [h_kv * group, nnz] per head
  int32_t per_head;                           // one row per query head, no group max
  int32_t batch, nnz, n_phys, h_kv, group, page_size, head_dim, dtype;
  int32_t summary_fp8;                        // summary holds E4M3 codes
  unsigned* err;
};

struct SelectArgs {
  const float* scores;
  const int32_t* page_indptr; const int32_t* page_indices; const int32_t* seq_lens;
  int32_t* sel_logical; int32_t* sel_phys; int32_t* sel_count;
  int32_t batch, nnz, h_kv, k, page_size;
  int32_t n_sink, n_local;                    // pages always kept (hybrid budget)
  unsigned* err;
};

struct AttnArgs {
  const void* q; const void* k_pool; const void* v_pool;
  const int32_t* sel_logical; const int32_t* sel_phys; const int32_t* seq_lens;
  const uint8_t* sel_mask;   // [batch, h_kv, k] heads of the group per slot, or null (all)
  float* out; float* lse;
  float* part_o;     // [batch, h_q, n_chunks, head_dim]
  float* part_ml;    // [batch, h_q, n_chunks, 2]  (running max in log2 units, sum)
  int32_t batch, n_phys, h_kv, group, page_size, head_dim, dtype, k;
  int32_t n_chunks, chunk_pages;
  float scale_log2;  // sm_scale * log2(e)
  unsigned* err;
  uint32_t wait_limit;   // tries of each bounded wait (set by launch_attn)
  int32_t test_fault;    // 2: a copy slot of CTA 0 never completes (tests; set by launch_attn)
};

// Fused decode step: append (optional, one token per request) + score +
// select + attention + combine in one persistent launch.
struct StepArgs {
  void* k_pool; void* v_pool; void* summary;
  const void* k_new; const void* v_new;      // [batch, h_kv, head_dim] or null
  const void* q;
  const int32_t* page_indptr; const int32_t* page_indices; const int32_t* seq_lens;
  float* scores;                              // [h_kv, nnz]
  int32_t* sel_logical; int32_t* sel_phys; int32_t* sel_count;
  float* out; float* lse;
  unsigned* counters;                         // [4 + 2 * units], see step.cu
  unsigned long long* tagged;                 // [h_kv, nnz] score bits | call tag << 32
  float* part_o; float* part_ml;              // [units, group, n_chunks, head_dim | 4 (max, sum, tag, 0)]
  int32_t batch, nnz, n_phys, h_kv, group, page_size, head_dim, dtype, k;
  int32_t summary_fp8;                        // summary holds E4M3 codes
  int32_t n_sink, n_local;                    // pages always kept (hybrid budget)
  int32_t n_chunks, chunk_pages;
  float scale_log2;
  unsigned long long* trace;                  // [grid, 16] phase stamps, or null
  unsigned* err;
  uint32_t wait_limit;                        // tries of every bounded wait (cluster step)
  int32_t test_fault;                         // 0; 1 = a slot whose copy never arrives (tests)
};

// Recall diagnostics (quest_recall_diagnostics): per query head, against
// dense attention over each request's valid tokens.
struct DiagArgs {
  const void* k_pool; const void* v_pool; const void* summary; const void* q;
  const int32_t* page_indptr; const int32_t* page_indices; const int32_t* seq_lens;
  const int32_t* sel_logical;                 // [batch, h_kv, k]
  float* slack;                               // [h_q, nnz]
  float* eps; float* topr;                    // [batch, h_q]
  float* vmax;                                // [batch, h_kv]
  float* logits;                              // workspace [h_q, nnz * page_size]
  float2* stats;                              // workspace [h_q, nnz] (base-2 max, sum)
  float* vnorm;                               // workspace [h_kv, nnz]
  int32_t batch, nnz, n_phys, h_kv, group, page_size, head_dim, dtype, k, top_r;
  float scale_log2;
  unsigned* err;
};

cudaError_t launch_diag(const DiagArgs& a, cudaStream_t s);
size_t diag_workspace_bytes(int32_t h_kv, int32_t group, int32_t nnz, int32_t page_size);
void diag_carve(DiagArgs& a, void* workspace);

struct StepPlan {
  bool ok;
  bool cluster;                               // the cluster kernel (cstep_impl.cuh)
  int32_t grid, n_chunks, chunk_pages, smem;
  size_t counters_bytes, tagged_bytes, workspace_bytes;
};

cudaError_t launch_step(const StepArgs& a, const StepPlan& p, cudaStream_t s);
StepPlan plan_step(int32_t batch, int32_t nnz, int32_t h_kv, int32_t group, int32_t head_dim,
                   int32_t page_size, int32_t dtype, int32_t k, int32_t summary_fp8);
// Per-variant, per-head-dim instantiations of the fused step
// (step_<variant>_d<head_dim>.cu): launch, and shared memory / resident CTAs
// per SM.
#define QUEST_STEP_VARIANT(name)                                                          \
  cudaError_t launch_step_##name##_d64(const StepArgs& a, const StepPlan& p, cudaStream_t s);  \
  cudaError_t launch_step_##name##_d128(const StepArgs& a, const StepPlan& p, cudaStream_t s); \
  void shape_step_##name##_d64(int dev, int page_size, int group, int* smem, int* per_sm);     \
  void shape_step_##name##_d128(int dev, int page_size, int group, int* smem, int* per_sm);
QUEST_STEP_VARIANT(f32)
QUEST_STEP_VARIANT(f16)
QUEST_STEP_VARIANT(e4m3)
#undef QUEST_STEP_VARIANT
// The same for the cluster kernel (cstep_<variant>_d<head_dim>.cu): launch,
// and clusters of it the current device keeps resident (<= 0: the shape is
// not built or does not fit).
#define QUEST_CSTEP_VARIANT(name)                                                           \
  cudaError_t launch_cstep_##name##_d64(const StepArgs& a, const StepPlan& p, cudaStream_t s);  \
  cudaError_t launch_cstep_##name##_d128(const StepArgs& a, const StepPlan& p, cudaStream_t s); \
  int clusters_cstep_##name##_d64(int dev, int page_size, int group);                        \
  int clusters_cstep_##name##_d128(int dev, int page_size, int group);
QUEST_CSTEP_VARIANT(f32)
QUEST_CSTEP_VARIANT(f16)
QUEST_CSTEP_VARIANT(e4m3)
#undef QUEST_CSTEP_VARIANT
constexpr int32_t kCStepUnitsPerCluster = 64;   // units one cluster of the cluster kernel takes
constexpr uint32_t kStepWaitLimit = 1u << 21;    // tries (up to ~1 us each) of a bounded wait

// Split-K plan of the attention for a problem size on the current device.
struct AttnPlan {
  int32_t n_chunks;
  int32_t chunk_pages;
  size_t workspace_bytes;
};

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);
cudaError_t launch_score(const ScoreArgs& a, cudaStream_t s);
cudaError_t launch_select(const SelectArgs& a, cudaStream_t s);
cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s);

// GQA page union (quest_union_decode_attn): per (request, KV head) the pages
// chosen by any of the group's query heads, in page order, with the bit set
// of the heads that chose each.
struct UnionArgs {
  const int32_t* sel_logical;                 // [batch, h_kv * group, k]
  const int32_t* page_indptr; const int32_t* page_indices; const int32_t* seq_lens;
  int32_t* u_logical; int32_t* u_phys;        // [batch, h_kv, group * k], -1 padded
  uint8_t* u_mask;                            // [batch, h_kv, group * k]
  int32_t* u_count;                           // [batch, h_kv]
  int32_t batch, h_kv, group, k, page_size;
  int32_t max_pages;                          // shared-memory bytes: pages of one request covered
  unsigned* err;
};
constexpr int32_t kUnionMaxPages = 65536;     // cap of max_pages (64 KiB of page bytes)
cudaError_t launch_union(const UnionArgs& a, cudaStream_t s);
AttnPlan plan_attn(int32_t batch, int32_t h_kv, int32_t group, int32_t head_dim,
                   int32_t page_size, int32_t dtype, int32_t k);

bool attn_supported(int32_t dtype, int32_t head_dim, int32_t page_size, int32_t group);

// Device address of the error word for the current device (null on failure).
unsigned* error_word_ptr();
bool score_supported(int32_t dtype, int32_t head_dim, int32_t group);

}  // namespace quest
