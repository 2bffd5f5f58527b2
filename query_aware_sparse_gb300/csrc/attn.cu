// a4 + a5: attention over the selected pages only, read in place from the
// paged pool (Quest page Fig. 1 and §2.1; token set and 1/sqrt(d) scale of
// PageWeaver notes §2 eq (1)-(2)), split over chunks of pages, then merged
// by log-sum-exp (Quest page §2.1: one row-global max and sum, never a
// per-page softmax average).
//
// Split-K kernel: one CTA per (request, KV head, chunk of pages), NW warps.
// Each warp owns a ring of NST shared-memory slots; its lane 0 streams the
// warp's pages in with 1-D bulk async copies (cp.async.bulk, completion on
// an mbarrier): one (page, head) K block and V block are each S*d contiguous
// elements of the pool. The CTA merges its warps and writes one partial
// (o, max, sum) per query head; the combine kernel merges the chunks.
// Decode attention is a matrix-vector product per query head; groups of 1
// and 2 stay on FMA. Groups of 4 and 8 with fp16 K/V run QK^T and PV on the
// warp MMA (attn_mma_kernel): each warp streams its pages with 16-byte
// cp.async copies into XOR-swizzled 16-token tiles read by ldmatrix.
// With a slot mask (the GQA page union) each page carries the heads that
// chose it, and the other heads of the group give it no weight.
#include "attn_dev.cuh"
#include "attn_mma.cuh"
#include "common.cuh"
#include "internal.h"

namespace quest {
namespace {

constexpr int kNW = 4;        // warps per CTA
constexpr int kNST = 2;       // bulk-copy slots per warp
constexpr int kMaxWarpPages = 32;

template <typename T, int D, int S, int G>
struct AttnShape {
  using W = WarpAttn<T, D, S, G>;
  static constexpr int STAGE_BYTES = kNW * kNST * 2 * W::BLOCK_BYTES;
  static constexpr int BAR_OFF = STAGE_BYTES;
  static constexpr int LOGIT_OFF = BAR_OFF + kNW * kNST * 8;
  static constexpr int DESC_OFF = LOGIT_OFF + kNW * W::NV * 4;
  static constexpr int SMEM = DESC_OFF + kNW * kMaxWarpPages * 8;
  static_assert(kNW * G * (D + 2) * 4 <= STAGE_BYTES, "merge buffer must fit in the stage area");
};

template <typename T, int D, int S, int G, bool MASK>
__global__ void __launch_bounds__(kNW * 32)
attn_split_kernel(const AttnArgs a) {
  using Sh = AttnShape<T, D, S, G>;
  using W = typename Sh::W;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::BAR_OFF);
  float* logits_all = reinterpret_cast<float*>(smem + Sh::LOGIT_OFF);
  int2* desc_all = reinterpret_cast<int2*>(smem + Sh::DESC_OFF);
  const uint64_t pol = evict_first_policy();   // K/V pages are read once

  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c = blockIdx.x % a.n_chunks;
  const int unit = blockIdx.x / a.n_chunks;     // r * h_kv + g
  const int g = unit % a.h_kv, r = unit / a.h_kv;
  const int h_q = a.h_kv * G;
  const int L = a.seq_lens[r];
  const size_t sel_base = (size_t)unit * a.k;

  uint64_t* my_bars = bars + w * kNST;
  float* lg = logits_all + w * W::NV;
  int2* desc = desc_all + w * kMaxWarpPages;
  T* my_stage = reinterpret_cast<T*>(smem) + (size_t)w * kNST * 2 * S * D;

  // This warp's pages: j = c*cp + w + NW*i, i < nmine.
  const int jc0 = c * a.chunk_pages;
  const int jc1 = min(a.k, jc0 + a.chunk_pages);
  const int j0 = jc0 + w;
  const int nmine = j0 < jc1 ? (jc1 - j0 + kNW - 1) / kNW : 0;
  int my_pp = -1, my_valid = 0, my_heads = 0xff;
  if (lane < nmine) {
    const int j = j0 + lane * kNW;
    const int lp = __ldg(a.sel_logical + sel_base + j);
    const int pp = __ldg(a.sel_phys + sel_base + j);
    if constexpr (MASK) my_heads = a.sel_mask[sel_base + j];   // heads that chose the page
    if (lp >= 0 && my_heads != 0) {
      const int valid = min(S, L - lp * S);
      if (valid <= 0) report(a.err, QUEST_DEVERR_EMPTY_PAGE);
      else if (pp < 0 || pp >= a.n_phys) report(a.err, QUEST_DEVERR_PAGE_RANGE);
      else { my_pp = pp; my_valid = valid; }
    }
  }
  const unsigned vmask = __ballot_sync(FULL, my_valid > 0);
  const int nv = __popc(vmask);
  if (my_valid > 0)
    desc[__popc(vmask & ((1u << lane) - 1))] = make_int2(my_pp, my_valid | (my_heads << 8));
  if (lane == 0) {
    for (int s = 0; s < kNST; ++s) mbar_init(my_bars + s, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const size_t head_block = (size_t)S * D;                 // elements per (page, head)
  const T* kbase = static_cast<const T*>(a.k_pool) + (size_t)g * head_block;
  const T* vbase = static_cast<const T*>(a.v_pool) + (size_t)g * head_block;
  const size_t page_stride = (size_t)a.h_kv * head_block;

  // the failure-handling test: warp 0 of CTA 0 expects 16 bytes more in its
  // first slot than the copies bring, so that slot's wait runs out
  const uint32_t extra = (a.test_fault == 2 && blockIdx.x == 0 && w == 0) ? 16u : 0u;
  auto issue = [&](int n) {
    const int slot = n % kNST;
    const int pp = desc[n].x;
    T* dst = my_stage + (size_t)slot * 2 * head_block;
    mbar_expect_tx(my_bars + slot, 2 * W::BLOCK_BYTES + (n == 0 ? extra : 0u));
    bulk_g2s_hint(dst, kbase + (size_t)pp * page_stride, W::BLOCK_BYTES, my_bars + slot, pol);
    bulk_g2s_hint(dst + head_block, vbase + (size_t)pp * page_stride, W::BLOCK_BYTES, my_bars + slot, pol);
  };
  if (lane == 0)
    for (int n = 0; n < min(kNST, nv); ++n) issue(n);

  W st;
  st.init(static_cast<const T*>(a.q) + ((size_t)r * h_q + g * G) * D, a.scale_log2, lane);

  // a wait that runs out ends this warp's pages: no more copies are issued,
  // the other slots' copies in flight are waited for (bounded), and the CTA
  // writes an empty partial instead of merging through the stage area
  bool dead = false;
  for (int n = 0; n < nv; ++n) {
    const int slot = n % kNST;
    if (!warp_wait_bounded(my_bars + slot, (n / kNST) & 1, a.wait_limit)) {
      if (lane == 0) report(a.err, QUEST_DEVERR_WAIT_TIMEOUT);
      dead = true;
      for (int m = n + 1; m < min(n + kNST, nv); ++m)
        warp_wait_bounded(my_bars + m % kNST, (m / kNST) & 1, a.wait_limit);
      break;
    }
    const T* Kb = my_stage + (size_t)slot * 2 * head_block;
    if constexpr (MASK)
      st.page(Kb, Kb + head_block, desc[n].y & 0xff, lg, lane, (unsigned)desc[n].y >> 8);
    else
      st.page(Kb, Kb + head_block, desc[n].y & 0xff, lg, lane);
    __syncwarp();
    if (lane == 0 && n + kNST < nv) {
      fence_proxy_async_smem();
      issue(n + kNST);
    }
  }

  const size_t row0 = ((size_t)r * h_q + g * G) * a.n_chunks + c;
  if (__syncthreads_or(dead)) {
    for (int gi = w; gi < G; gi += kNW) {
      for (int col = lane; col < D; col += 32) a.part_o[(row0 + (size_t)gi * a.n_chunks) * D + col] = 0.f;
      if (lane == 0) {
        a.part_ml[(row0 + (size_t)gi * a.n_chunks) * 2 + 0] = -INFINITY;
        a.part_ml[(row0 + (size_t)gi * a.n_chunks) * 2 + 1] = 0.f;
      }
    }
    return;
  }
  // Merge the warps of this CTA (stage area reused once every warp is done).
  float* mo = reinterpret_cast<float*>(smem);                 // [NW][G][D]
  float* ml = mo + kNW * G * D;                               // [NW][G][2]
  st.stash(mo, ml, w, lane);
  __syncthreads();
  merge_warps<D, G, kNW, kNW * 32>(
      mo, ml,
      [&](int gi, int col, float o) { a.part_o[(row0 + (size_t)gi * a.n_chunks) * D + col] = o; },
      [&](int gi, float mx, float l) {
        a.part_ml[(row0 + (size_t)gi * a.n_chunks) * 2 + 0] = mx;
        a.part_ml[(row0 + (size_t)gi * a.n_chunks) * 2 + 1] = l;
      });
}

// Groups of 4 and 8, fp16: the same split as attn_split_kernel (head masks too)
// with QK^T and PV on the warp MMA. Each warp keeps two pages in flight in
// its own slots (a page's K and V as one cp.async group).
template <int D, int S>
struct AttnMmaShape {
  static constexpr int RB = D * 2;                          // bytes of a K or V row
  static constexpr int BLK = S * RB;                        // a (page, head) K or V block
  static constexpr int SLOT = 2 * BLK;                      // K then V
  static constexpr int STAGE_BYTES = kNW * kNST * SLOT;
  static constexpr int PS_OFF = STAGE_BYTES;                // [kNW][256 B] P tiles
  static constexpr int DESC_OFF = PS_OFF + kNW * 256;
  static constexpr int SMEM = DESC_OFF + kNW * kMaxWarpPages * 8;
  static_assert(S % 16 == 0, "whole 16-token tiles");
};

template <int D, int S, int G, bool MASK>
__global__ void __launch_bounds__(kNW * 32)
attn_mma_kernel(const AttnArgs a) {
  using Sh = AttnMmaShape<D, S>;
  using W = WarpAttnMmaS<D, G>;
  static_assert(kNW * G * (D + 2) * 4 <= Sh::STAGE_BYTES, "merge buffer must fit in the stage area");
  extern __shared__ __align__(128) unsigned char smem[];
  int2* desc_all = reinterpret_cast<int2*>(smem + Sh::DESC_OFF);

  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c = blockIdx.x % a.n_chunks;
  const int unit = blockIdx.x / a.n_chunks;     // r * h_kv + g
  const int g = unit % a.h_kv, r = unit / a.h_kv;
  const int h_q = a.h_kv * G;
  const int L = a.seq_lens[r];
  const size_t sel_base = (size_t)unit * a.k;
  int2* desc = desc_all + w * kMaxWarpPages;
  unsigned char* stage = smem + (size_t)w * kNST * Sh::SLOT;
  __half* ps = reinterpret_cast<__half*>(smem + Sh::PS_OFF + w * 256);

  // this warp's pages: j = c*cp + w + NW*i, i < nmine (as attn_split_kernel)
  const int jc0 = c * a.chunk_pages;
  const int jc1 = min(a.k, jc0 + a.chunk_pages);
  const int j0 = jc0 + w;
  const int nmine = j0 < jc1 ? (jc1 - j0 + kNW - 1) / kNW : 0;
  int my_pp = -1, my_valid = 0, my_heads = 0xff;
  if (lane < nmine) {
    const int j = j0 + lane * kNW;
    const int lp = __ldg(a.sel_logical + sel_base + j);
    const int pp = __ldg(a.sel_phys + sel_base + j);
    if constexpr (MASK) my_heads = a.sel_mask[sel_base + j];   // heads that chose the page
    if (lp >= 0 && my_heads != 0) {
      const int valid = min(S, L - lp * S);
      if (valid <= 0) report(a.err, QUEST_DEVERR_EMPTY_PAGE);
      else if (pp < 0 || pp >= a.n_phys) report(a.err, QUEST_DEVERR_PAGE_RANGE);
      else { my_pp = pp; my_valid = valid; }
    }
  }
  const unsigned vmask = __ballot_sync(FULL, my_valid > 0);
  const int nv = __popc(vmask);
  if (my_valid > 0)
    desc[__popc(vmask & ((1u << lane) - 1))] = make_int2(my_pp, my_valid | (my_heads << 8));
  __syncwarp();

  auto issue = [&](int n) {                     // page n's K and V into slot n % kNST
    const int pp = desc[n].x;
    unsigned char* dst = stage + (n % kNST) * Sh::SLOT;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const unsigned char* src = static_cast<const unsigned char*>(half ? a.v_pool : a.k_pool) +
                                 ((size_t)pp * a.h_kv + g) * Sh::BLK;
#pragma unroll
      for (int k = 0; k < Sh::BLK / 512; ++k) {
        const int pc = k * 32 + lane;               // 16-byte piece of the block
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                     :: "r"(smem_u32(dst + half * Sh::BLK + W::sw(pc / (Sh::RB / 16), pc % (Sh::RB / 16)))),
                        "l"(src + (size_t)pc * 16) : "memory");
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
#pragma unroll
  for (int n = 0; n < kNST - 1; ++n) {
    if (n < nv) issue(n);
    else asm volatile("cp.async.commit_group;" ::: "memory");
  }

  W st;
  st.init(static_cast<const __half*>(a.q) + ((size_t)r * h_q + g * G) * D, a.scale_log2, lane);
  static_assert(kNST == 2, "one page streams while the other is folded");
  for (int n = 0; n < nv; ++n) {
    if (n + 1 < nv) issue(n + 1);
    else asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncwarp();
    const uint32_t kb = smem_u32(stage + (n % kNST) * Sh::SLOT), vb = kb + Sh::BLK;
    const int valid = desc[n].y & 0xff;
    const unsigned hm = (unsigned)desc[n].y >> 8;
    for (int t = 0; t * 16 < valid; ++t) {
      st.qk(kb + t * 16 * Sh::RB, valid - t * 16, ps, lane, hm);
      st.av(vb + t * 16 * Sh::RB, valid - t * 16, ps, lane);
    }
    __syncwarp();                                   // slot n % kNST may be refilled
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");

  // Merge the warps of this CTA (stage area reused once every warp is done).
  __syncthreads();
  float* mo = reinterpret_cast<float*>(smem);                 // [NW][G][D]
  float* ml = mo + kNW * G * D;                               // [NW][G][2]
  st.stash(mo, ml, w, lane);
  __syncthreads();
  const size_t row0 = ((size_t)r * h_q + g * G) * a.n_chunks + c;
  merge_warps<D, G, kNW, kNW * 32>(
      mo, ml,
      [&](int gi, int col, float o) { a.part_o[(row0 + (size_t)gi * a.n_chunks) * D + col] = o; },
      [&](int gi, float mx, float l) {
        a.part_ml[(row0 + (size_t)gi * a.n_chunks) * 2 + 0] = mx;
        a.part_ml[(row0 + (size_t)gi * a.n_chunks) * 2 + 1] = l;
      });
}

// One warp per (request, query head): LSE merge of the chunk partials. The
// chunk maxima are read lane-parallel; the weighted sum issues its loads
// independently of each other.
template <int D>
__global__ void __launch_bounds__(128)
attn_combine_kernel(const AttnArgs a) {
  constexpr int VD = D / 32;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);       // r * h_q + h
  const int h_q = a.h_kv * a.group;
  if (row >= a.batch * h_q) return;
  const float* pml = a.part_ml + (size_t)row * a.n_chunks * 2;
  const float* po = a.part_o + (size_t)row * a.n_chunks * D;
  float mx = -INFINITY;
  for (int c = lane; c < a.n_chunks; c += 32) mx = fmaxf(mx, pml[c * 2]);
  mx = warp_max(mx);
  float o[VD];
#pragma unroll
  for (int v = 0; v < VD; ++v) o[v] = 0.f;
  float l = 0.f;
  if (mx != -INFINITY) {
    for (int c0 = 0; c0 < a.n_chunks; c0 += 32) {
      const int c = c0 + lane;
      float wc = 0.f, lc = 0.f;
      if (c < a.n_chunks) {
        const float mc = pml[c * 2];
        wc = mc == -INFINITY ? 0.f : exp2f(mc - mx);
        lc = pml[c * 2 + 1];
      }
      l += warp_sum(wc * lc);
      const int nc = min(32, a.n_chunks - c0);
#pragma unroll 4
      for (int i = 0; i < nc; ++i) {
        const float wi = __shfl_sync(FULL, wc, i);
#pragma unroll
        for (int v = 0; v < VD; ++v)
          o[v] = fmaf(wi, po[(size_t)(c0 + i) * D + lane * VD + v], o[v]);
      }
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int v = 0; v < VD; ++v) a.out[(size_t)row * D + lane * VD + v] = o[v] * inv;
  if (a.lse && lane == 0) a.lse[row] = l > 0.f ? (mx + log2f(l)) * LN2 : -INFINITY;
}

template <typename T, int D, int S, int G, bool MASK>
cudaError_t launch_split(const AttnArgs& a, cudaStream_t s) {
  if constexpr (sizeof(T) == 2 && G >= 4) {
    if (a.test_fault != 2) {                        // (the failure test takes the bulk-copy path)
      using Sm = AttnMmaShape<D, S>;
      auto kern = attn_mma_kernel<D, S, G, MASK>;
      int dev = 0;
      cudaGetDevice(&dev);
      static std::atomic<bool> done[64];
      if (dev < 0 || dev >= 64 || !done[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sm::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
      }
      kern<<<(unsigned)a.batch * a.h_kv * a.n_chunks, kNW * 32, Sm::SMEM, s>>>(a);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      const unsigned rows = (unsigned)a.batch * a.h_kv * a.group;
      attn_combine_kernel<D><<<(rows + 3) / 4, 128, 0, s>>>(a);
      return cudaGetLastError();
    }
  }
  using Sh = AttnShape<T, D, S, G>;
  auto kern = attn_split_kernel<T, D, S, G, MASK>;
  int dev = 0;
  cudaGetDevice(&dev);
  static std::atomic<bool> attr_done[64];   // per device and instantiation
  if (dev < 0 || dev >= 64 || !attr_done[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev].store(true, std::memory_order_release);
  }
  const unsigned grid = (unsigned)a.batch * a.h_kv * a.n_chunks;
  kern<<<grid, kNW * 32, Sh::SMEM, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned rows = (unsigned)a.batch * a.h_kv * a.group;
  attn_combine_kernel<D><<<(rows + 3) / 4, 128, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T, int D, int S>
cudaError_t launch_g(const AttnArgs& a, cudaStream_t s) {
  // head masks (GQA page union) only for G > 1: with one head a union page
  // always belongs to it
  const bool m = a.sel_mask != nullptr;
  switch (a.group) {
    case 1: return launch_split<T, D, S, 1, false>(a, s);
    case 2: return m ? launch_split<T, D, S, 2, true>(a, s) : launch_split<T, D, S, 2, false>(a, s);
    case 4: return m ? launch_split<T, D, S, 4, true>(a, s) : launch_split<T, D, S, 4, false>(a, s);
    case 8: return m ? launch_split<T, D, S, 8, true>(a, s) : launch_split<T, D, S, 8, false>(a, s);
  }
  return cudaErrorInvalidValue;
}

template <typename T, int D>
cudaError_t launch_s(const AttnArgs& a, cudaStream_t s) {
  return a.page_size == 16 ? launch_g<T, D, 16>(a, s) : launch_g<T, D, 32>(a, s);
}

int smem_for(int dtype, int head_dim, int page_size, int group) {
  const int esz = dtype == QUEST_F16 ? 2 : 4;
  const int block = page_size * head_dim * esz;
  const int tt = (group * page_size <= 64) ? page_size : 64 / group;
  return kNW * kNST * 2 * block + kNW * kNST * 8 + kNW * group * tt * 4 + kNW * kMaxWarpPages * 8;
}

}  // namespace

bool attn_supported(int32_t dtype, int32_t head_dim, int32_t page_size, int32_t group) {
  return (dtype == QUEST_F16 || dtype == QUEST_F32) && (head_dim == 64 || head_dim == 128) &&
         (page_size == 16 || page_size == 32) &&
         (group == 1 || group == 2 || group == 4 || group == 8) &&
         smem_for(dtype, head_dim, page_size, group) <= 227 * 1024;   // per-CTA limit
}

AttnPlan plan_attn(int32_t batch, int32_t h_kv, int32_t group, int32_t head_dim,
                   int32_t page_size, int32_t dtype, int32_t k) {
  int dev = 0, sms = 148, smem_sm = 228 * 1024;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  }
  cudaGetLastError();
  const int smem = smem_for(dtype, head_dim, page_size, group) + 1024;   // + per-CTA reserve
  const int per_sm = smem_sm / smem > 0 ? smem_sm / smem : 1;
  const long long target = (long long)sms * per_sm;
  const long long total = (long long)batch * h_kv * k;
  long long cp = (total + target * kNW - 1) / (target * kNW) * kNW;       // pages per chunk
  if (cp < kNW) cp = kNW;
  if (cp > kNW * kMaxWarpPages) cp = kNW * kMaxWarpPages;
  AttnPlan p;
  p.chunk_pages = (int32_t)cp;
  p.n_chunks = (int32_t)((k + cp - 1) / cp);
  const size_t rows = (size_t)batch * h_kv * group * p.n_chunks;
  p.workspace_bytes = rows * head_dim * sizeof(float) + rows * 2 * sizeof(float);
  p.workspace_bytes = (p.workspace_bytes + 255) & ~(size_t)255;
  return p;
}

cudaError_t launch_attn(const AttnArgs& args, cudaStream_t s) {
  if (args.batch == 0 || args.h_kv == 0) return cudaSuccess;
  AttnArgs a = args;
  a.wait_limit = wait_limit();
  a.test_fault = test_fault_mode() == 2 ? 2 : 0;
  if (a.dtype == QUEST_F16)
    return a.head_dim == 128 ? launch_s<__half, 128>(a, s) : launch_s<__half, 64>(a, s);
  return a.head_dim == 128 ? launch_s<float, 128>(a, s) : launch_s<float, 64>(a, s);
}

}  // namespace quest
