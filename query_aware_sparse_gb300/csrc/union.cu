// GQA page union (Quest page §2.1, the MHA / GQA / head-sharing paragraphs):
// every query head of a group picks its own Top-K pages; the group's shared
// KV head then reads the union of those picks once, and each page carries
// the bit set of the heads that picked it so that each head's attention still
// covers its own pages only.
//
// One CTA per (request, KV head). The group's G * k selected ids are OR-ed
// into a byte per page (bit i = head i of the group) held in shared memory,
// four pages to a word. A block-wide scan over the words then writes the
// pages with a non-zero byte in increasing page order, with their physical
// ids and head bits; the rest of the G * k slots get -1. At most G * k
// distinct pages can be chosen, so the output never overflows.
#include "common.cuh"
#include "internal.h"

namespace quest {
namespace {

constexpr int kUnionThreads = 256;
constexpr int kUnionWarps = kUnionThreads / 32;

__global__ void __launch_bounds__(kUnionThreads)
union_kernel(const UnionArgs a) {
  extern __shared__ uint32_t owners[];               // [ceil(P / 4)]
  __shared__ int warp_tot[kUnionWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int unit = blockIdx.x;                        // r * h_kv + g
  const int g = unit % a.h_kv, r = unit / a.h_kv;
  const int G = a.group, KU = G * a.k;
  const int lo = __ldg(a.page_indptr + r);
  const int tp = __ldg(a.page_indptr + r + 1) - lo;
  const int S = a.page_size;
  int P = (__ldg(a.seq_lens + r) + S - 1) / S;
  if (P > tp || P > a.max_pages) {
    if (tid == 0) report(a.err, QUEST_DEVERR_TABLE_RANGE);
    P = min(tp, a.max_pages);
  }
  const int nw = (P + 3) / 4;
  for (int i = tid; i < nw; i += kUnionThreads) owners[i] = 0u;
  __syncthreads();
  // slot j of the group's rows belongs to head j / k of the group
  const int32_t* sel = a.sel_logical + (size_t)unit * KU;
  for (int j = tid; j < KU; j += kUnionThreads) {
    const int lp = __ldg(sel + j);
    if (lp < 0) continue;
    if (lp >= P) {                                    // no valid token there
      report(a.err, QUEST_DEVERR_EMPTY_PAGE);
      continue;
    }
    atomicOr(&owners[lp >> 2], (1u << (j / a.k)) << (8 * (lp & 3)));
  }
  __syncthreads();
  // compaction in page order: thread t owns a contiguous run of words
  const int per = (nw + kUnionThreads - 1) / kUnionThreads;
  const int w0 = min(nw, tid * per), w1 = min(nw, w0 + per);
  int cnt = 0;
  for (int i = w0; i < w1; ++i) {
    const uint32_t x = owners[i];
    cnt += ((x & 0xffu) != 0) + ((x & 0xff00u) != 0) + ((x & 0xff0000u) != 0) + ((x >> 24) != 0);
  }
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kUnionWarps; ++w) {
    base += w < warp ? warp_tot[w] : 0;
    total += warp_tot[w];
  }
  int pos = base + incl - cnt;
  const size_t ob = (size_t)unit * KU;
  for (int i = w0; i < w1; ++i) {
    const uint32_t x = owners[i];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t m = (x >> (8 * b)) & 0xffu;
      if (m) {
        const int lp = i * 4 + b;
        a.u_logical[ob + pos] = lp;
        a.u_phys[ob + pos] = __ldg(a.page_indices + lo + lp);
        a.u_mask[ob + pos] = (uint8_t)m;
        ++pos;
      }
    }
  }
  for (int j = total + tid; j < KU; j += kUnionThreads) {
    a.u_logical[ob + j] = -1;
    a.u_phys[ob + j] = -1;
    a.u_mask[ob + j] = 0;
  }
  if (tid == 0) a.u_count[unit] = total;
}

}  // namespace

cudaError_t launch_union(const UnionArgs& a, cudaStream_t s) {
  if (a.batch == 0 || a.h_kv == 0) return cudaSuccess;
  const int smem = ((a.max_pages + 3) / 4) * 4;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem);
    if (e != cudaSuccess) return e;
  }
  union_kernel<<<(unsigned)a.batch * a.h_kv, kUnionThreads, smem > 0 ? smem : 4, s>>>(a);
  return cudaGetLastError();
}

}  // namespace quest
