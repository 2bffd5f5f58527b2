// a3: fixed-budget Top-K pages per (request, KV head) (Quest page Fig. 1,
// §1.1 and §2: K pages for a token budget of K * S tokens). Ties go to the
// lower logical page index; winners are emitted in ascending page order.
//
// One CTA per (request, KV head). Scores become order-preserving 32-bit keys
// (-0 folded onto +0 so that they tie); an MSB-first radix select (four 8-bit
// digits, shared-memory histograms with warp-aggregated atomics) finds the
// K-th largest key T and how many keys equal to T are still needed; a
// block-wide scan in page order then emits every key > T plus the first
// `need` keys == T. No sort, no global workspace.
#include "common.cuh"
#include "internal.h"

namespace quest {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelSmemKeys = 16384;   // scores cached in shared memory up to this P

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t x = __float_as_uint(f == 0.f ? 0.f : f);   // -0 -> +0
  return x ^ ((x & 0x80000000u) ? 0xffffffffu : 0x80000000u);
}

// Block-wide exclusive scan of a 64-bit value (sums of two packed counters).
__device__ __forceinline__ unsigned long long block_excl_scan(unsigned long long v,
                                                              unsigned long long* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned long long t = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = lane < kSelWarps ? s_warp[lane] : 0ull;
    unsigned long long wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      unsigned long long t = __shfl_up_sync(FULL, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < kSelWarps) s_warp[lane] = wi - w;   // exclusive warp offsets
  }
  __syncthreads();
  return s_warp[warp] + incl - v;
}

__global__ void __launch_bounds__(kSelThreads)
select_kernel(const SelectArgs a) {
  extern __shared__ uint32_t s_keys[];
  __shared__ uint32_t s_hist[256];
  __shared__ uint32_t s_digit, s_krem;
  __shared__ unsigned long long s_warp[kSelWarps];

  const int r = blockIdx.x / a.h_kv;
  const int g = blockIdx.x % a.h_kv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.k;
  const int lo = a.page_indptr[r];
  const int table_pages = a.page_indptr[r + 1] - lo;
  int P = (a.seq_lens[r] + a.page_size - 1) / a.page_size;
  if (P > table_pages) {
    if (tid == 0) report(a.err, QUEST_DEVERR_TABLE_RANGE);
    P = table_pages;
  }
  const size_t out = ((size_t)r * a.h_kv + g) * K;

  if (P <= K) {    // every scored page is selected
    for (int i = tid; i < K; i += kSelThreads) {
      a.sel_logical[out + i] = i < P ? i : -1;
      a.sel_phys[out + i] = i < P ? a.page_indices[lo + i] : -1;
    }
    if (tid == 0) a.sel_count[(size_t)r * a.h_kv + g] = P;
    return;
  }

  const float* sc = a.scores + (size_t)g * a.nnz + lo;
  const bool cached = P <= kSelSmemKeys;
  if (cached)
    for (int i = tid; i < P; i += kSelThreads) s_keys[i] = score_key(__ldg(sc + i));
  auto key_at = [&](int i) -> uint32_t { return cached ? s_keys[i] : score_key(__ldg(sc + i)); };

  // Radix select of the K-th largest key.
  uint32_t prefix = 0, krem = K;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const uint32_t hi_mask = pass == 0 ? 0u : (0xffffffffu << (shift + 8));
    for (int i = tid; i < 256; i += kSelThreads) s_hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < P; base += kSelThreads) {
      const int i = base + tid;
      uint32_t dig = 256;
      if (i < P) {
        const uint32_t key = key_at(i);
        if ((key & hi_mask) == prefix) dig = (key >> shift) & 255u;
      }
      const unsigned peers = __match_any_sync(FULL, dig);
      if (dig < 256 && (__ffs(peers) - 1) == lane) atomicAdd(&s_hist[dig], __popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t h[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) { h[j] = s_hist[lane * 8 + j]; tot += h[j]; }
      uint32_t incl = tot;            // sum over lanes >= lane
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t t = __shfl_down_sync(FULL, incl, o);
        if (lane + o < 32) incl += t;
      }
      uint32_t cum = incl - tot;      // keys in higher digits
#pragma unroll
      for (int j = 7; j >= 0; --j) {
        if (cum < krem && krem <= cum + h[j]) { s_digit = lane * 8 + j; s_krem = krem - cum; }
        cum += h[j];
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    krem = s_krem;
  }
  const uint32_t T = prefix;
  const uint32_t need = krem;   // keys equal to T still to take (>= 1)

  // Stable compaction in page order: keys > T, plus the first `need` == T.
  const int per = (P + kSelThreads - 1) / kSelThreads;
  const int c0 = min(P, tid * per), c1 = min(P, c0 + per);
  uint32_t gt = 0, eq = 0;
  for (int i = c0; i < c1; ++i) {
    const uint32_t key = key_at(i);
    gt += key > T;
    eq += key == T;
  }
  const unsigned long long ex =
      block_excl_scan(((unsigned long long)gt << 32) | eq, s_warp);
  uint32_t gt_b = (uint32_t)(ex >> 32), eq_b = (uint32_t)ex;
  for (int i = c0; i < c1; ++i) {
    const uint32_t key = key_at(i);
    int pos = -1;
    if (key > T) {
      pos = gt_b + min(eq_b, need);
      ++gt_b;
    } else if (key == T) {
      if (eq_b < need) pos = gt_b + eq_b;
      ++eq_b;
    }
    if (pos >= 0 && pos < K) {
      a.sel_logical[out + pos] = i;
      a.sel_phys[out + pos] = a.page_indices[lo + i];
    }
  }
  if (tid == 0) a.sel_count[(size_t)r * a.h_kv + g] = K;
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, cudaStream_t s) {
  if (a.batch == 0 || a.h_kv == 0) return cudaSuccess;
  const size_t smem = kSelSmemKeys * sizeof(uint32_t);
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_done[64] = {};   // per device; racing setters write the same value
  if (dev >= 64 || !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_done[dev] = true;
  }
  select_kernel<<<(unsigned)a.batch * a.h_kv, kSelThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace quest
