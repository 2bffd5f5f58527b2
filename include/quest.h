/*
 * quest.h — C ABI of libquest: Quest-style query-aware page selection over a
 * paged KV cache for long-context decode, on one NVIDIA GB300 (sm_103a).
 *
 * Sources. "Quest page" is the PaperTrace chapter
 * "3.1.1 · Quest：用 min/max 上界筛选 KV 页"; "PageWeaver notes" is the
 * reading-notes page "PageWeaver: KV-Guided Query Unions for Sparse
 * Attention". Each entry point below names the passage that defines it.
 *
 * General contract
 *  - Every pointer argument marked "device" must point to device memory of the
 *    current CUDA device; the caller allocates and owns all of it (pools,
 *    summaries, page tables, outputs, workspace). The library allocates no
 *    memory. Its device state lives in its own module memory: a 4-byte error
 *    word per device, and the fixed 4 MiB buffer of
 *    quest_sparse_decode_attn_noalloc (see there).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream). A QUEST_OK return means the work was enqueued.
 *  - Host-side validation runs first; on any error nothing is enqueued and a
 *    negative quest_status is returned. A failed launch returns QUEST_ERR_CUDA.
 *  - Problems only visible on the device (a page index outside the pool, a
 *    selected page with no valid token, an exhausted wait) never trap: the
 *    offending item is skipped and a bit is OR-ed into the device error word,
 *    which quest_get_device_error() returns and clears.
 *  - Element types: QUEST_F32 or QUEST_F16 for K, V, summaries and q (all the
 *    same type), or with fp16 K/V/q, E4M3 summaries (quest_cache.summary_fp8);
 *    outputs are fp32. head_dim in {64, 128}; page_size in {16, 32}; GQA group
 *    in {1, 2, 4, 8}.
 *  - Data pointers (pools, summary, q, k_new, v_new) must be 16-byte aligned.
 */
#ifndef QUEST_H
#define QUEST_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QUEST_API __attribute__((visibility("default")))
#else
#define QUEST_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QUEST_OK = 0,
  QUEST_ERR_INVALID_ARG = -1,  /* null pointer, bad size, misalignment        */
  QUEST_ERR_UNSUPPORTED = -2,  /* dtype / head_dim / page_size / group not built */
  QUEST_ERR_WORKSPACE = -3,    /* workspace missing or smaller than required   */
  QUEST_ERR_CUDA = -4          /* a CUDA runtime call or launch failed         */
} quest_status;

typedef enum { QUEST_F32 = 0, QUEST_F16 = 1 } quest_dtype;

/* Bits of the device error word. */
#define QUEST_DEVERR_PAGE_RANGE   0x1u  /* physical page id outside [0, n_phys)      */
#define QUEST_DEVERR_TABLE_RANGE  0x2u  /* append/selection beyond the page table    */
#define QUEST_DEVERR_EMPTY_PAGE   0x4u  /* selected page holds no valid token        */
#define QUEST_DEVERR_WAIT_TIMEOUT 0x8u  /* an in-kernel wait hit its iteration limit */
#define QUEST_DEVERR_FP8_RANGE    0x10u /* a key beyond +-448 under an E4M3 summary  */

/*
 * One layer's paged cache (Quest page §1.2: the summary has logical shape
 * [L, P, H_kv, 2, d_h] and is bound to the physical page; one struct = one L).
 *   k_pool, v_pool : device, [n_phys, h_kv, page_size, head_dim], dtype
 *   summary        : device, [n_phys, h_kv, 2, head_dim], dtype;
 *                    [..., 0, :] = per-dimension min m, [..., 1, :] = max M
 *   summary_fp8    : 0 = the summary above. 1 = the summary is uint8 E4M3
 *                    codes of the same shape instead (Quest page §3, the
 *                    paragraph on the summary dtype): the OCP 8-bit float
 *                    without infinities (bias 7, 3 mantissa bits, largest
 *                    finite 448), m rounded toward -inf and M toward +inf, so
 *                    the box still contains every key of the page and U_p
 *                    stays an upper bound; a rounded zero is stored as +0.
 *                    Appends fold new keys straight into the codes (rounding
 *                    commutes with min/max, so the result equals rounding the
 *                    exact summary); scoring reads the codes. Half the
 *                    summary bytes of fp16. Needs dtype QUEST_F16. A key
 *                    beyond +-448 cannot be bounded: its code saturates and
 *                    QUEST_DEVERR_FP8_RANGE is set. quest_recall_diagnostics
 *                    does not take E4M3 summaries (QUEST_ERR_UNSUPPORTED).
 */
typedef struct quest_cache {
  void* k_pool;
  void* v_pool;
  void* summary;
  int32_t n_phys;
  int32_t h_kv;
  int32_t page_size;
  int32_t head_dim;
  int32_t dtype;       /* quest_dtype */
  int32_t summary_fp8; /* 0: summary in dtype; 1: E4M3 codes, directed rounding */
} quest_cache;

/*
 * Ragged page table of a batch of requests (Quest page §2.1: requests are
 * described by an indptr over pages; the page table maps logical pages to
 * physical pages of the pool, Quest page Fig. 1).
 *   page_indptr  : device int32 [batch + 1], page_indptr[0] = 0
 *   page_indices : device int32 [nnz]; entry page_indptr[r] + p is the
 *                  physical page holding logical page p of request r
 *   seq_lens     : device int32 [batch], valid tokens of each request. Only
 *                  the first ceil(seq_lens[r] / page_size) logical pages of a
 *                  request hold tokens; later table entries are reserved pages.
 *   nnz          : host copy of page_indptr[batch]
 */
typedef struct quest_pages {
  const int32_t* page_indptr;
  const int32_t* page_indices;
  const int32_t* seq_lens;
  int32_t batch;
  int32_t nnz;
} quest_pages;

/*
 * quest_append_kv — cache append with incremental summary update
 * (Quest page §1.2 eq (8) and §3 eq (14); page recycling in §3).
 *
 * Token i of request r, append_indptr[r] <= i < append_indptr[r+1], is
 * written at position pos = seq_lens_before[r] + (i - append_indptr[r]):
 * logical page pos / page_size, slot pos % page_size. For each touched
 * (page, KV head, dim): if slot 0 of the page is written by this call the
 * summary restarts from the new keys (m = M = the first new key, then eq (8)),
 * otherwise the new keys are folded into the stored m and M with eq (8).
 * min/max order -0 below +0. Full pages that receive no token are not touched.
 *   k_new, v_new      : device [n_new, h_kv, head_dim], dtype
 *   n_new             : host, total new tokens (= append_indptr[batch])
 *   append_indptr     : device int32 [batch + 1]
 *   seq_lens_before   : device int32 [batch]
 * pages->seq_lens is not read (the caller updates lengths itself). The page
 * table must already map every page the new tokens land in; a token beyond it
 * is skipped with QUEST_DEVERR_TABLE_RANGE. Calls that overlap on the GPU and
 * touch the same page race.
 */
QUEST_API quest_status quest_append_kv(const quest_cache* cache, const quest_pages* pages,
                             const void* k_new, const void* v_new, int32_t n_new,
                             const int32_t* append_indptr,
                             const int32_t* seq_lens_before, void* stream);

/*
 * quest_score_pages — page upper bounds (Quest page §1.1 eq (2)-(3)).
 *
 * scores[g * nnz + e] for table entry e of request r and KV head g is
 *   U = sum_j max(q_{h,j} m_j, q_{h,j} M_j)
 * for the query head h = g (group == 1); with group > 1 the G query heads
 * g*G .. g*G+G-1 share one page set and U is their maximum (Quest page §2.1,
 * group-max aggregation). Unscaled dot-product bounds, fp32 arithmetic.
 * Reserved entries (logical page >= ceil(seq_lens[r] / page_size)) get -inf.
 *   q      : device [batch, h_kv * group, head_dim], dtype
 *   scores : device fp32 [h_kv, nnz]
 */
QUEST_API quest_status quest_score_pages(const quest_cache* cache, const quest_pages* pages,
                               const void* q, int32_t group, float* scores,
                               void* stream);

/*
 * quest_score_pages_per_head — the page bounds of quest_score_pages with one
 * row per query head and no aggregation over the group (Quest page §2.1, the
 * GQA paragraph: each query head may pick its own pages, the shared KV head
 * then reads the union of the picks; quest_union_decode_attn).
 *   scores : device fp32 [h_kv * group, nnz]; row h holds U_{h,p} against the
 *            summary of KV head h / group; reserved entries get -inf.
 * Select each head's pages with quest_select_topk(pages, h_kv * group, ...)
 * on these rows (sel_logical [batch, h_kv * group, k]).
 */
QUEST_API quest_status quest_score_pages_per_head(const quest_cache* cache,
                                                  const quest_pages* pages, const void* q,
                                                  int32_t group, float* scores, void* stream);

/*
 * quest_select_topk — fixed-budget Top-K pages (Quest page Fig. 1, §1.1 and
 * §2: K pages, token budget K * page_size).
 *
 * For each (request r, KV head g) with P_r = ceil(seq_lens[r] / page_size)
 * scored pages: the min(k, P_r) pages with the largest scores, ties broken
 * by the lower logical page index (-0 equals +0). Emitted in ascending
 * logical page order; unused slots hold -1.
 * Hybrid budget (local window + sink + Quest; Quest page §2.2 and §3.2,
 * C = C_local u C_sink u C_quest): the first n_sink and the last n_local of
 * the P_r valid pages are always kept (their union, the tail page being the
 * last local page), and the rest of the k pages are the Top-K of the other
 * pages by the rule above. n_sink = n_local = 0 is plain Quest.
 *   page_size   : tokens per page (gives P_r from seq_lens); 16 or 32
 *   scores      : device fp32 [h_kv, nnz] as written by quest_score_pages
 *   n_sink, n_local : forced pages, >= 0 each, n_sink + n_local <= k
 *                 (else QUEST_ERR_INVALID_ARG)
 *   sel_logical : device int32 [batch, h_kv, k] logical page ids
 *   sel_phys    : device int32 [batch, h_kv, k] physical page ids (page table)
 *   sel_count   : device int32 [batch, h_kv] = min(k, P_r)
 */
QUEST_API quest_status quest_select_topk(const quest_pages* pages, int32_t h_kv,
                               int32_t page_size, const float* scores, int32_t k,
                               int32_t n_sink, int32_t n_local,
                               int32_t* sel_logical, int32_t* sel_phys,
                               int32_t* sel_count, void* stream);

/*
 * quest_sparse_decode_attn — attention over the selected pages only, read in
 * place from the pool (Quest page Fig. 1 and §2.1; token set and 1/sqrt(d)
 * scale as in PageWeaver notes §2 eq (1)-(2)).
 *
 * For query head h of request r with KV head g = h / group, the candidate
 * tokens are the valid tokens of the pages listed in sel_logical[r, g, :]
 * (physical ids in sel_phys; -1 entries skipped; the tail page contributes
 * seq_lens[r] - p * page_size tokens). out = softmax(q k^T * sm_scale) V over
 * those tokens only, lse = log of the softmax denominator (natural log, of the
 * scaled logits). An empty set gives out = 0 and lse = -inf. Split-K: chunks
 * of pages produce partial (o, max, sum) in `workspace`, merged by
 * log-sum-exp in a second pass (Quest page §2.1). The ids of one (r, g) list
 * must be distinct.
 *   q          : device [batch, h_kv * group, head_dim], dtype
 *   sel_*      : device int32 [batch, h_kv, k]
 *   out        : device fp32 [batch, h_kv * group, head_dim]
 *   lse        : device fp32 [batch, h_kv * group], or NULL
 *   sm_scale   : <= 0 selects 1 / sqrt(head_dim)
 *   workspace  : device, >= quest_attn_workspace_size(...) bytes, 16-B aligned
 */
QUEST_API quest_status quest_sparse_decode_attn(const quest_cache* cache,
                                      const quest_pages* pages, const void* q,
                                      int32_t group, const int32_t* sel_logical,
                                      const int32_t* sel_phys, int32_t k,
                                      float* out, float* lse, float sm_scale,
                                      void* workspace, size_t workspace_bytes,
                                      void* stream);

/*
 * quest_sparse_decode_attn_noalloc — the same attention as
 * quest_sparse_decode_attn (same kernels, same arguments and results) without
 * a workspace argument. The paper has no counterpart to this call; it exists
 * for callers that cannot allocate device memory: a plug-in that only receives
 * input and output pointers from its host program, or a serving loop that must
 * not call cudaMalloc (which can synchronise the device) once it is running.
 * The split-K partials go to a fixed 4 MiB buffer inside the library's own
 * module memory (one per device that loads the library, kept until the
 * process exits); the call allocates nothing. A problem whose partials, as
 * planned for the cache's element type on the current device, need more than
 * 4 MiB is rejected with QUEST_ERR_WORKSPACE before anything is launched.
 * quest_attn_workspace_size(...) is the larger of the two element types'
 * plans, so a problem it sizes at 4 MiB or less is always accepted; above
 * that, the cache's own element type decides. The first call on a device
 * looks up the buffer's device address (cudaGetSymbolAddress, with that device
 * current); make that first call before any stream capture. Every call shares
 * the one buffer and leaves its contents behind; no part of it needs to start
 * at zero, but calls that overlap on the GPU (other streams, other threads)
 * race on it.
 */
QUEST_API quest_status quest_sparse_decode_attn_noalloc(const quest_cache* cache,
                                                        const quest_pages* pages,
                                                        const void* q, int32_t group,
                                                        const int32_t* sel_logical,
                                                        const int32_t* sel_phys, int32_t k,
                                                        float* out, float* lse,
                                                        float sm_scale, void* stream);

/* Workspace bytes quest_sparse_decode_attn needs for these sizes on the
 * current device (the split-K chunking depends on its SM count). */
QUEST_API size_t quest_attn_workspace_size(int32_t batch, int32_t h_kv, int32_t group,
                                 int32_t head_dim, int32_t page_size,
                                 int32_t k);

/*
 * quest_union_decode_attn — GQA attention with a page set per query head
 * (Quest page §2.1, the MHA / GQA / head-sharing paragraphs): per (request,
 * KV head) the union of the pages the group's heads chose is formed, each
 * page of it is read once, and query head h weighs only the valid tokens of
 * its own pages (softmax over its own candidate set; an empty set gives o = 0,
 * lse = -inf). Split-K over the union, then the log-sum-exp merge.
 *   sel_logical   : device int32 [batch, h_kv * group, k] per-head logical
 *                   pages (-1 = empty slot), e.g. quest_select_topk on the
 *                   rows of quest_score_pages_per_head
 *   out, lse      : device fp32 [batch, h_kv * group, head_dim], [batch,
 *                   h_kv * group] (lse may be NULL); sm_scale <= 0 selects
 *                   1 / sqrt(head_dim)
 *   union_logical : device int32 [batch, h_kv, group * k] (written): the union
 *                   in increasing page order, -1 padded
 *   union_mask    : device uint8 [batch, h_kv, group * k] (written): bit i set
 *                   when head i of the group chose the page
 *   union_count   : device int32 [batch, h_kv] (written): pages in the union
 *   workspace     : device, >= quest_union_workspace_size(...) bytes, 16-B
 *                   aligned
 * A selected page with no valid token is skipped (QUEST_DEVERR_EMPTY_PAGE);
 * requests of more than 65536 pages (or more than pages->nnz) are cut there
 * (QUEST_DEVERR_TABLE_RANGE).
 */
QUEST_API quest_status quest_union_decode_attn(const quest_cache* cache, const quest_pages* pages,
                                               const void* q, int32_t group,
                                               const int32_t* sel_logical, int32_t k, float* out,
                                               float* lse, float sm_scale, int32_t* union_logical,
                                               uint8_t* union_mask, int32_t* union_count,
                                               void* workspace, size_t workspace_bytes,
                                               void* stream);

/* Workspace bytes quest_union_decode_attn needs (0 for unsupported shapes). */
QUEST_API size_t quest_union_workspace_size(int32_t batch, int32_t h_kv, int32_t group,
                                            int32_t head_dim, int32_t page_size, int32_t dtype,
                                            int32_t k);

/*
 * quest_decode_step — one decode step of one layer in a single fused launch:
 * the append of one new token per request (optional), page scoring, Top-K
 * selection and sparse attention with its log-sum-exp merge (the four calls
 * above, Quest page Fig. 1 and §1.2/§2.1, in one kernel). Results equal those of quest_append_kv (one token per request at
 * position seq_lens[r] - 1) followed by quest_score_pages, quest_select_topk
 * and quest_sparse_decode_attn on the same arguments.
 *   pages->seq_lens : lengths INCLUDING the new token
 *   k_new, v_new    : device [batch, h_kv, head_dim] dtype, or both NULL
 *                     (no append: the cache already holds every token)
 *   q, group, k, n_sink, n_local : as quest_score_pages / quest_select_topk
 *   scores          : device fp32 [h_kv, nnz] (written)
 *   sel_logical, sel_phys, sel_count : as quest_select_topk (written)
 *   out, lse        : as quest_sparse_decode_attn (lse may be NULL)
 *   sm_scale        : <= 0 selects 1 / sqrt(head_dim)
 *   workspace       : device, >= quest_decode_workspace_size(...) bytes,
 *                     16-B aligned, ZERO-FILLED before its first use; a call
 *                     that completes leaves its counters at zero again (after
 *                     a QUEST_DEVERR_WAIT_TIMEOUT, zero it again). Calls that
 *                     share a workspace must not overlap on the GPU.
 * Two kernels serve it (quest_decode_step_kernel tells which one a shape
 * gets): a kernel on clusters of four CTAs, one cluster per group of
 * (request, KV head) units, with the units' keys and partials exchanged in
 * distributed shared memory (no workspace use beyond the size check); and a
 * persistent cooperative kernel (one or two CTAs per SM, hand-offs through
 * the workspace) for the shapes the first one does not take. Returns
 * QUEST_ERR_UNSUPPORTED for shapes neither fits.
 */
QUEST_API quest_status quest_decode_step(const quest_cache* cache, const quest_pages* pages,
                                         const void* k_new, const void* v_new,
                                         const void* q, int32_t group, int32_t k,
                                         int32_t n_sink, int32_t n_local,
                                         float* scores, int32_t* sel_logical,
                                         int32_t* sel_phys, int32_t* sel_count,
                                         float* out, float* lse, float sm_scale,
                                         void* workspace, size_t workspace_bytes,
                                         void* stream);

/* Workspace bytes quest_decode_step needs on the current device for a page
 * table of nnz entries (0 if the shape is unsupported). */
QUEST_API size_t quest_decode_workspace_size(int32_t batch, int32_t nnz, int32_t h_kv, int32_t group,
                                             int32_t head_dim, int32_t page_size,
                                             int32_t dtype, int32_t k);

/* Which kernel quest_decode_step launches for these sizes on the current
 * device: 2 the cluster kernel (cstep_kernel), 1 the cooperative grid-wide
 * kernel (step_kernel), 0 the shape is unsupported. summary_fp8 as in
 * quest_cache. */
QUEST_API int32_t quest_decode_step_kernel(int32_t batch, int32_t h_kv, int32_t group,
                                           int32_t head_dim, int32_t page_size, int32_t dtype,
                                           int32_t k, int32_t summary_fp8);

/*
 * quest_recall_diagnostics — how well a selection covers dense attention, per
 * query head (Quest page §1.1: the recall paragraph and eq (6)-(7); §3.1 page
 * slack), computed on the GPU from the cache itself. Query head h is judged
 * by the pages chosen for its KV head h / group; every quantity runs over the
 * request's valid tokens (pages->seq_lens).
 *   q           : device [batch, h_kv * group, head_dim], dtype
 *   sel_logical : device int32 [batch, h_kv, k] logical page ids, -1 = empty
 *                 slot (as quest_select_topk writes them)
 *   top_r       : >= 1; the row's min(top_r, seq_len) largest dense logits
 *                 (ties to the lower position) are the top-R tokens
 *   sm_scale    : <= 0 selects 1 / sqrt(head_dim) (used by eps only)
 *   slack       : device fp32 [h_kv * group, nnz]: g_p(q_h) = U_p(q_h) - the
 *                 largest q_h.k over the page's valid keys (unscaled; U_p from
 *                 the stored summary, per query head, no group max); NaN for
 *                 table entries past a request's ceil(seq_len / page_size)
 *   eps         : device fp32 [batch, h_kv * group]: dense softmax mass of the
 *                 tokens outside the selected pages
 *   topr        : device fp32 [batch, h_kv * group]: the share of the top-R
 *                 tokens that lie on selected pages
 *   vmax        : device fp32 [batch, h_kv]: max_t ||v_t||_2 (eq (7))
 *   workspace   : device, >= quest_diag_workspace_size(...) bytes, 16-B aligned
 * Rows of more than 65536 pages are cut to their first 65536 pages. A dense
 * pass over every valid key and value: a diagnostic, off the decode path.
 */
QUEST_API quest_status quest_recall_diagnostics(const quest_cache* cache, const quest_pages* pages,
                                                const void* q, int32_t group,
                                                const int32_t* sel_logical, int32_t k,
                                                int32_t top_r, float sm_scale, float* slack,
                                                float* eps, float* topr, float* vmax,
                                                void* workspace, size_t workspace_bytes,
                                                void* stream);

/* Workspace bytes quest_recall_diagnostics needs (0 for unsupported sizes). */
QUEST_API size_t quest_diag_workspace_size(int32_t h_kv, int32_t group, int32_t nnz,
                                           int32_t page_size);

/* Phase trace of quest_decode_step (profiling aid, off by default): with a
 * device buffer of at least 16 * max_ctas uint64 set, each later call whose
 * grid has at most max_ctas CTAs writes, per CTA, 16 %globaltimer stamps (ns;
 * a stamp a CTA does not reach stays as it was).
 * Cluster kernel: [0] start, [1] the previous kernel on the stream waited
 * for, [5] every CTA's keys of the first unit in, [10] its Top-K done, [11]
 * its physical ids looked up, [6] its selection published, [4] the first
 * attention tile of warp 0 done, [7] the last unit merged (owning CTA), [9]
 * exit.
 * Grid-wide kernel: [0] start, [1] scoring done, [2] selection done, [3..5]
 * attention start / pages done / merged, [6..7] first select started / last
 * select done (CTAs that select), [9] exit; [10..15] on CTAs that only
 * select: polled / done of their 1st..3rd select; on the others: descriptors
 * loaded, first page done, partials merged, final merges.
 * NULL turns it off. Returns the grid size the current device uses for these
 * shapes (0 if the shape is unsupported). */
QUEST_API int32_t quest_set_trace(void* device_buffer, int32_t max_ctas, int32_t batch,
                                  int32_t h_kv, int32_t group, int32_t head_dim,
                                  int32_t page_size, int32_t dtype, int32_t k);

/* Test hook of the kernels' failure handling (no counterpart on the pages).
 * mode 0: normal operation. mode 1: in later quest_decode_step calls that
 * take the cluster kernel, warp 0 of the first CTA of each cluster first
 * waits on a barrier nothing arrives on. mode 2: in later
 * quest_sparse_decode_attn(_noalloc) and quest_union_decode_attn calls, the
 * first copy slot of warp 0 of the first CTA expects 16 bytes more than its
 * copies bring. Either way that wait runs out: the kernel sets
 * QUEST_DEVERR_WAIT_TIMEOUT, issues no further copies, waits (bounded) for
 * those in flight and returns, its outputs unspecified; the device stays
 * usable. wait_limit: tries of every bounded in-kernel wait of those calls
 * (each up to about 1 us); 0 restores the default (about 2 s). Process-wide
 * host state; returns QUEST_ERR_INVALID_ARG for other values. */
QUEST_API int32_t quest_test_step_fault(int32_t mode, int32_t wait_limit);

/* Synchronises `stream`, returns the device error word of the current device
 * (QUEST_DEVERR_* bits) and clears it. Returns -1 if a CUDA call fails. */
QUEST_API int32_t quest_get_device_error(void* stream);

/* Static, NUL-terminated description of a status code. */
QUEST_API const char* quest_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* QUEST_H */
