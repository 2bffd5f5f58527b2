// a2: page upper bounds U_p(q) = sum_j max(q_j m_j, q_j M_j)
// (Quest page §1.1 eq (2)-(3)); GQA groups share one score, the maximum over
// the group's query heads (Quest page §2.1), or with `per_head` one row per
// query head (the per-head selection of the same section's GQA paragraph).
//
// HBM-bound stream of the [n_phys, h_kv, 2, d] summary. A (page, KV head)
// summary is 2*d contiguous elements; LPP lanes cover one page with 16-byte
// loads (min half and max half of the same dims in the same lane), so one
// warp instruction moves 32 x 16 B and the G query heads of the group reuse
// the registers. Each lane keeps UNROLL pages of loads in flight. With E4M3
// summaries (fp16 queries) a lane reads the codes of the same 8 dims as
// 8-byte loads of m and of M: half the bytes over the same lanes.
#include "common.cuh"
#include "internal.h"

namespace quest {
namespace {

constexpr int kScoreThreads = 256;
constexpr int kScoreUnroll = 4;

template <typename T, int D>
struct ScoreShape {
  static constexpr int VEC = Elem<T>::kVec;          // elements per lane-load
  static constexpr int LPP = D / VEC;                // lanes per page
  static constexpr int PPW = 32 / LPP;               // pages per warp step
  static constexpr int WARPS = kScoreThreads / 32;
  static constexpr int TILE = WARPS * PPW * kScoreUnroll;  // pages per CTA
};

__device__ __forceinline__ int find_request(const int32_t* indptr, int lo, int hi, int e) {
  // largest r in [lo, hi] with indptr[r] <= e
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(indptr + mid) <= e) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <typename T, int D, int G>
__device__ __forceinline__ void load_q(const ScoreArgs& a, int r, int g, int sub, uint4 (&q)[G]) {
  constexpr int VEC = Elem<T>::kVec;
  const T* qp = static_cast<const T*>(a.q) +
                ((size_t)r * a.h_kv * G + (size_t)g * G) * D + sub * VEC;
#pragma unroll
  for (int gi = 0; gi < G; ++gi) q[gi] = ld_nc_v4(qp + (size_t)gi * D);
}

template <typename T, int D, int G, bool F8, bool PH>
__global__ void __launch_bounds__(kScoreThreads)
score_kernel(const ScoreArgs a) {
  static_assert(!F8 || sizeof(T) == 2, "E4M3 summaries take fp16 queries");
  using Sh = ScoreShape<T, D>;
  constexpr int VEC = Sh::VEC, LPP = Sh::LPP, PPW = Sh::PPW;
  __shared__ int s_rfirst, s_rlast;

  const int g = blockIdx.y;
  const uint64_t pol = evict_first_policy();   // summaries are read once
  const int e_begin = blockIdx.x * Sh::TILE;
  const int e_end = min(a.nnz, e_begin + Sh::TILE);
  if (threadIdx.x == 0) {
    s_rfirst = find_request(a.page_indptr, 0, a.batch - 1, e_begin);
    s_rlast = find_request(a.page_indptr, 0, a.batch - 1, e_end - 1);
  }
  __syncthreads();
  const int rfirst = s_rfirst, rlast = s_rlast;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int sub = lane % LPP;       // which 16-byte column of the page
  const int pw = lane / LPP;        // which page of the warp step

  uint4 q[G];
  int cur_r = rfirst;
  load_q<T, D, G>(a, cur_r, g, sub, q);
  // fp16 MHA: the query as fp32 and its sign masks, converted once per
  // request instead of once per page (llama_layer 9.46 -> 9.20 us). Not for
  // groups: G = 4 needs 107 registers that way, two CTAs per SM instead of
  // three, and the latency-bound stream slowed down (gqa_batch 91 -> 109 us).
  constexpr bool PRE = sizeof(T) == 2 && !F8 && G == 1;
  float qf[PRE ? G : 1][8];
  uint32_t qm[PRE ? G : 1][4];
  auto convert_q = [&]() {
    if constexpr (PRE) {
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        const uint32_t w[4] = {q[gi].x, q[gi].y, q[gi].z, q[gi].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          qm[gi][j] = ((~w[j] & 0x80008000u) >> 15) * 0xffffu;   // halves with q >= 0
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
          qf[gi][2 * j] = f.x;
          qf[gi][2 * j + 1] = f.y;
        }
      }
    }
  };
  convert_q();

  // Page e handled by (warp, u, pw): consecutive warps take consecutive runs.
  uint4 vm[kScoreUnroll], vM[kScoreUnroll];
  int er[kScoreUnroll];
  bool live[kScoreUnroll];
#pragma unroll
  for (int u = 0; u < kScoreUnroll; ++u) {
    const int e = e_begin + (warp * kScoreUnroll + u) * PPW + pw;
    int r = rfirst;
    live[u] = false;
    if (e < e_end) {
      if (rfirst != rlast) r = find_request(a.page_indptr, rfirst, rlast, e);
      const int lp = e - __ldg(a.page_indptr + r);
      const int valid_pages = (__ldg(a.seq_lens + r) + a.page_size - 1) / a.page_size;
      const int pp = __ldg(a.page_indices + e);
      if (lp < valid_pages) {
        if (pp >= 0 && pp < a.n_phys) {
          if constexpr (F8) {
            const uint8_t* sp = static_cast<const uint8_t*>(a.summary) +
                                ((size_t)pp * a.h_kv + g) * 2 * D + sub * VEC;
            const uint2 cm = ld_stream_v2_hint(sp, pol), cM = ld_stream_v2_hint(sp + D, pol);
            vm[u] = make_uint4(cm.x, cm.y, 0u, 0u);
            vM[u] = make_uint4(cM.x, cM.y, 0u, 0u);
          } else {
            const T* sp = static_cast<const T*>(a.summary) +
                          ((size_t)pp * a.h_kv + g) * 2 * D + sub * VEC;
            vm[u] = ld_stream_v4_hint(sp, pol);
            vM[u] = ld_stream_v4_hint(sp + D, pol);
          }
          live[u] = true;
        } else if (sub == 0) {
          report(a.err, QUEST_DEVERR_PAGE_RANGE);
        }
      }
    }
    er[u] = r;
  }

#pragma unroll
  for (int u = 0; u < kScoreUnroll; ++u) {
    const int e = e_begin + (warp * kScoreUnroll + u) * PPW + pw;
    if (er[u] != cur_r) {       // page of another request: its own query
      cur_r = er[u];
      load_q<T, D, G>(a, cur_r, g, sub, q);
      convert_q();
    }
    float best = -INFINITY;
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      float s = 0.f;
      if (live[u]) {
        if constexpr (F8) {
          s = bound8_e4m3(q[gi], make_uint2(vm[u].x, vm[u].y), make_uint2(vM[u].x, vM[u].y));
        } else if constexpr (PRE) {   // sum_j q_j * (q_j >= 0 ? M_j : m_j)
          const uint32_t mw[4] = {vm[u].x, vm[u].y, vm[u].z, vm[u].w};
          const uint32_t Mw[4] = {vM[u].x, vM[u].y, vM[u].z, vM[u].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t xw = (Mw[j] & qm[gi][j]) | (mw[j] & ~qm[gi][j]);
            const float2 xf = __half22float2(*reinterpret_cast<const __half2*>(&xw));
            s = fmaf(qf[gi][2 * j], xf.x, s);
            s = fmaf(qf[gi][2 * j + 1], xf.y, s);
          }
        } else {
          s = bound16<T>(q[gi], vm[u], vM[u]);
        }
      }
#pragma unroll
      for (int o = 1; o < LPP; o <<= 1) s += __shfl_xor_sync(FULL, s, o);
      best = fmaxf(best, s);
      if (PH && sub == 0 && e < e_end)             // one row per query head
        a.scores[((size_t)g * G + gi) * a.nnz + e] = live[u] ? s : -INFINITY;
    }
    if (!PH && sub == 0 && e < e_end)
      a.scores[(size_t)g * a.nnz + e] = live[u] ? best : -INFINITY;
  }
}

template <typename T, int D, bool F8>
cudaError_t launch_td(const ScoreArgs& a, cudaStream_t s) {
  using Sh = ScoreShape<T, D>;
  dim3 grid((a.nnz + Sh::TILE - 1) / Sh::TILE, a.h_kv);
  // per-head rows only differ from the group max for G > 1
  const bool ph = a.per_head != 0;
  switch (a.group) {
    case 1: score_kernel<T, D, 1, F8, false><<<grid, kScoreThreads, 0, s>>>(a); break;
    case 2:
      if (ph) score_kernel<T, D, 2, F8, true><<<grid, kScoreThreads, 0, s>>>(a);
      else score_kernel<T, D, 2, F8, false><<<grid, kScoreThreads, 0, s>>>(a);
      break;
    case 4:
      if (ph) score_kernel<T, D, 4, F8, true><<<grid, kScoreThreads, 0, s>>>(a);
      else score_kernel<T, D, 4, F8, false><<<grid, kScoreThreads, 0, s>>>(a);
      break;
    case 8:
      if (ph) score_kernel<T, D, 8, F8, true><<<grid, kScoreThreads, 0, s>>>(a);
      else score_kernel<T, D, 8, F8, false><<<grid, kScoreThreads, 0, s>>>(a);
      break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

bool score_supported(int32_t dtype, int32_t head_dim, int32_t group) {
  return (dtype == QUEST_F16 || dtype == QUEST_F32) && (head_dim == 64 || head_dim == 128) &&
         (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_score(const ScoreArgs& a, cudaStream_t s) {
  if (a.nnz == 0 || a.batch == 0) return cudaSuccess;
  if (a.dtype == QUEST_F16 && a.summary_fp8)
    return a.head_dim == 128 ? launch_td<__half, 128, true>(a, s) : launch_td<__half, 64, true>(a, s);
  if (a.dtype == QUEST_F16)
    return a.head_dim == 128 ? launch_td<__half, 128, false>(a, s) : launch_td<__half, 64, false>(a, s);
  return a.head_dim == 128 ? launch_td<float, 128, false>(a, s) : launch_td<float, 64, false>(a, s);
}

}  // namespace quest
