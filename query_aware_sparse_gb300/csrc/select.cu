// a3: fixed-budget Top-K pages per (request, KV head) (Quest page Fig. 1,
// §1.1 and §2: K pages for a token budget of K * S tokens). Ties go to the
// lower logical page index; winners are emitted in ascending page order.
// Hybrid budget (Quest page §2.2, §3.2): the first n_sink and last n_local
// valid pages are always kept and Quest fills the rest of the K pages.
// One CTA per (request, KV head) runs the block-wide select of topk.cuh.
#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace quest {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelSmemKeys = 16384;   // scores cached in shared memory up to this P

__global__ void __launch_bounds__(kSelThreads)
select_kernel(const SelectArgs a) {
  extern __shared__ uint32_t s_keys[];
  __shared__ TopkSmem<kSelThreads> sm;
  const int r = blockIdx.x / a.h_kv;
  const int g = blockIdx.x % a.h_kv;
  const int lo = a.page_indptr[r];
  const int table_pages = a.page_indptr[r + 1] - lo;
  int P = (a.seq_lens[r] + a.page_size - 1) / a.page_size;
  if (P > table_pages) {
    if (threadIdx.x == 0) report(a.err, QUEST_DEVERR_TABLE_RANGE);
    P = table_pages;
  }
  const size_t out = ((size_t)r * a.h_kv + g) * a.k;
  const int32_t* idx = a.page_indices + lo;
  // forced pages: [0, f_lo) and [f_hi, P)
  const int f_lo = min(a.n_sink, P), f_hi = max(f_lo, P - a.n_local);
  block_topk<kSelThreads>(a.scores + (size_t)g * a.nnz + lo, P, a.k, s_keys, kSelSmemKeys, sm,
                          a.sel_logical + out, a.sel_phys + out,
                          a.sel_count + (size_t)r * a.h_kv + g,
                          [idx](int i) { return idx[i]; },
                          [f_lo, f_hi](int i) { return i < f_lo || i >= f_hi; },
                          f_lo + (P - f_hi));
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, cudaStream_t s) {
  if (a.batch == 0 || a.h_kv == 0) return cudaSuccess;
  const size_t smem = kSelSmemKeys * sizeof(uint32_t);
  int dev = 0;
  cudaGetDevice(&dev);
  static std::atomic<bool> attr_done[64];   // per device
  if (dev < 0 || dev >= 64 || !attr_done[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev].store(true, std::memory_order_release);
  }
  select_kernel<<<(unsigned)a.batch * a.h_kv, kSelThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace quest
