// f4: recall diagnostics of a selection against dense attention, per query
// head (Quest page §1.1: the recall paragraph, eq (6)-(7); §3.1 page slack).
//
// Pass 1 (one warp per (page, KV head) item, CTAs over chunks of the page
// table x KV heads): for each valid token t of the page and each query head h
// of the group, the dense logit s = q_h . k_t; per head the page's largest
// logit, the page bound U_p(q_h) from the stored summary (the slack g_p is
// their difference), the page's softmax statistics in base 2 (max and sum of
// 2^(s * sm_scale * log2 e - max)); the token logits themselves (for the
// top-R tokens); and the largest ||v_t||^2 of the page.
// Pass 2 (one CTA per (request, query head)): excluded mass eps = the pages
// outside the selection's share of the softmax normaliser, the top-R tokens
// of the row by the block Top-K of topk.cuh (ties to the lower position) and
// how many of them lie on selected pages, and V_max over the request.
// A dense pass over every valid key and value: a diagnostic, off the decode
// path.
#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace quest {
namespace {

constexpr int kDiagThreads = 256;
constexpr int kDiagNW = kDiagThreads / 32;
constexpr int kDiagPages = 32;        // page-table entries per CTA of pass 1
constexpr int kDiagMaxG = 8;
constexpr int kDiagBitWords = 2048;   // selected-page bitmap of pass 2: up to 65536 pages

__device__ __forceinline__ int diag_find_req(const int32_t* indptr, int lo, int hi, int e) {
  while (lo < hi) {                   // largest r in [lo, hi] with indptr[r] <= e
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(indptr + mid) <= e) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// one lane's VD consecutive elements of a row, loaded as one vector
template <typename T, int VD>
struct alignas(VD * sizeof(T)) DiagRow { T v[VD]; };

template <typename T, int VD>
__device__ __forceinline__ void load_dims(const T* p, float (&o)[VD]) {
#pragma unroll
  for (int v = 0; v < VD; ++v) o[v] = Elem<T>::to_f(p[v]);
}

template <typename T, int D, int S>
__global__ void __launch_bounds__(kDiagThreads)
diag_pages_kernel(const DiagArgs a) {
  constexpr int VD = D / 32;          // dims per lane
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = blockIdx.y, G = a.group;
  const int h_q = a.h_kv * G;
  const size_t row_tok = (size_t)a.nnz * S;   // token-logit row of one query head
  const int e_begin = blockIdx.x * kDiagPages;
  const int e_end = min(a.nnz, e_begin + kDiagPages);
  float qf[kDiagMaxG][VD];
  int q_r = -1;
  for (int e = e_begin + warp; e < e_end; e += kDiagNW) {
    const int r = diag_find_req(a.page_indptr, 0, a.batch - 1, e);
    const int lp = e - __ldg(a.page_indptr + r);
    const int L = __ldg(a.seq_lens + r);
    const int P = (L + S - 1) / S;
    const int pp = __ldg(a.page_indices + e);
    const bool live = lp < P && pp >= 0 && pp < a.n_phys;
    if (lp < P && !live && lane == 0) report(a.err, QUEST_DEVERR_PAGE_RANGE);
    if (!live) {                      // no page here: NaN slack, empty statistics
      if (lane < G) {
        const int h = g * G + lane;
        a.slack[(size_t)h * a.nnz + e] = __int_as_float(0x7fc00000);
        a.stats[(size_t)h * a.nnz + e] = make_float2(-INFINITY, 0.f);
      }
      if (lane == 0) a.vnorm[(size_t)g * a.nnz + e] = 0.f;
      for (int i = lane; i < G * S; i += 32)
        a.logits[(size_t)(g * G + i / S) * row_tok + (size_t)e * S + i % S] = -INFINITY;
      continue;
    }
    if (r != q_r) {                   // the group's queries, this lane's dims
#pragma unroll
      for (int h = 0; h < kDiagMaxG; ++h)
        if (h < G)
          load_dims<T, VD>(static_cast<const T*>(a.q) + ((size_t)r * h_q + (size_t)g * G + h) * D + lane * VD,
                           qf[h]);
      q_r = r;
    }
    const int valid = min(S, L - lp * S);
    // page bound U_p(q_h) = sum_j max(q_j m_j, q_j M_j) from the stored summary
    const T* sp = static_cast<const T*>(a.summary) + ((size_t)pp * a.h_kv + g) * 2 * D + lane * VD;
    float mn[VD], mx[VD];
    load_dims<T, VD>(sp, mn);
    load_dims<T, VD>(sp + D, mx);
    float U[kDiagMaxG], smax[kDiagMaxG], m2[kDiagMaxG], l2[kDiagMaxG];
#pragma unroll
    for (int h = 0; h < kDiagMaxG; ++h) {
      float u = 0.f;
#pragma unroll
      for (int v = 0; v < VD; ++v) u += fmaxf(qf[h][v] * mn[v], qf[h][v] * mx[v]);
      U[h] = h < G ? warp_sum(u) : 0.f;
      smax[h] = -INFINITY; m2[h] = -INFINITY; l2[h] = 0.f;
    }
    const T* kb = static_cast<const T*>(a.k_pool) + ((size_t)pp * a.h_kv + g) * S * D + lane * VD;
    const T* vb = static_cast<const T*>(a.v_pool) + ((size_t)pp * a.h_kv + g) * S * D + lane * VD;
    float vn2 = 0.f;
    // rows in batches of TB tokens: all loads of a batch are in flight at once
    using Row = DiagRow<T, VD>;
    constexpr int TB = sizeof(Row) >= 16 ? 8 : 16;
    for (int t0 = 0; t0 < S; t0 += TB) {
      Row kr[TB], vr[TB];
#pragma unroll
      for (int i = 0; i < TB; ++i) {
        if (t0 + i < valid) {
          kr[i] = *reinterpret_cast<const Row*>(kb + (size_t)(t0 + i) * D);
          vr[i] = *reinterpret_cast<const Row*>(vb + (size_t)(t0 + i) * D);
        }
      }
#pragma unroll
      for (int i = 0; i < TB; ++i) {
        const int t = t0 + i;
        float* lrow = a.logits + (size_t)e * S + t;
        if (t >= valid) {
          if (lane < G) lrow[(size_t)(g * G + lane) * row_tok] = -INFINITY;
          continue;
        }
        float vs = 0.f;
#pragma unroll
        for (int v = 0; v < VD; ++v) {
          const float x = Elem<T>::to_f(vr[i].v[v]);
          vs = fmaf(x, x, vs);
        }
        vn2 = fmaxf(vn2, warp_sum(vs));
#pragma unroll
        for (int h = 0; h < kDiagMaxG; ++h) {
          if (h >= G) break;
          float s = 0.f;
#pragma unroll
          for (int v = 0; v < VD; ++v) s = fmaf(qf[h][v], Elem<T>::to_f(kr[i].v[v]), s);
          s = warp_sum(s);
          smax[h] = fmaxf(smax[h], s);
          const float x = s * a.scale_log2;
          const float mnew = fmaxf(m2[h], x);
          l2[h] = l2[h] * exp2f(m2[h] - mnew) + exp2f(x - mnew);
          m2[h] = mnew;
          if (lane == h) lrow[(size_t)(g * G + h) * row_tok] = s;
        }
      }
    }
#pragma unroll
    for (int h = 0; h < kDiagMaxG; ++h) {
      if (h < G && lane == h) {
        a.slack[(size_t)(g * G + h) * a.nnz + e] = U[h] - smax[h];
        a.stats[(size_t)(g * G + h) * a.nnz + e] = make_float2(m2[h], l2[h]);
      }
    }
    if (lane == 0) a.vnorm[(size_t)g * a.nnz + e] = sqrtf(vn2);
  }
}

template <int NT>
__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = is_max ? warp_max(v) : warp_sum(v);
  __syncthreads();                    // red[] free
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
  return r;
}

template <int S>
__global__ void __launch_bounds__(kDiagThreads)
diag_reduce_kernel(const DiagArgs a) {
  __shared__ uint32_t bits[kDiagBitWords];
  __shared__ TopkSmem<kDiagThreads> tsm;
  __shared__ float red[kDiagNW];
  __shared__ unsigned s_hits;
  const int tid = threadIdx.x;
  const int h_q = a.h_kv * a.group;
  const int r = blockIdx.x / h_q, h = blockIdx.x % h_q, g = h / a.group;
  const int lo = __ldg(a.page_indptr + r);
  const int tp = __ldg(a.page_indptr + r + 1) - lo;
  int L = __ldg(a.seq_lens + r);
  int P = (L + S - 1) / S;
  if (P > tp) {
    if (tid == 0) report(a.err, QUEST_DEVERR_TABLE_RANGE);
    P = tp;
    L = min(L, P * S);
  }
  P = min(P, kDiagBitWords * 32);
  L = min(L, P * S);
  for (int i = tid; i < (P + 31) / 32; i += kDiagThreads) bits[i] = 0u;
  if (tid == 0) s_hits = 0u;
  __syncthreads();
  const int32_t* sel = a.sel_logical + ((size_t)r * a.h_kv + g) * a.k;
  for (int j = tid; j < a.k; j += kDiagThreads) {
    const int lp = __ldg(sel + j);
    if (lp >= 0 && lp < P) atomicOr(&bits[lp >> 5], 1u << (lp & 31));
  }
  __syncthreads();
  auto selected = [&](int lp) { return (bits[lp >> 5] >> (lp & 31)) & 1u; };

  // eps: the unselected pages' share of the softmax normaliser
  const float2* st = a.stats + (size_t)h * a.nnz + lo;
  float mloc = -INFINITY;
  for (int i = tid; i < P; i += kDiagThreads) mloc = fmaxf(mloc, st[i].x);
  const float M = block_reduce<kDiagThreads>(mloc, red, true);
  float tot = 0.f, ex = 0.f;
  for (int i = tid; i < P; i += kDiagThreads) {
    const float2 v = st[i];
    const float w = v.y > 0.f ? v.y * exp2f(v.x - M) : 0.f;
    tot += w;
    if (!selected(i)) ex += w;
  }
  tot = block_reduce<kDiagThreads>(tot, red, false);
  ex = block_reduce<kDiagThreads>(ex, red, false);

  // top-R tokens of the row (block Top-K, ties to the lower position)
  const int R = min(a.top_r, L);
  const float* row = a.logits + (size_t)h * a.nnz * S + (size_t)lo * S;
  for (int i = tid; i < kTopkBins; i += kDiagThreads) tsm.hist[i] = 0u;
  __syncthreads();
  block_topk_keys<kDiagThreads>(L, R, [row](int i) { return score_key(__ldcg(row + i)); }, tsm,
                                [&](int, int i) { if (selected(i / S)) atomicAdd(&s_hits, 1u); });
  // V_max over the request (first head of the group)
  float vloc = 0.f;
  if (h % a.group == 0)
    for (int i = tid; i < P; i += kDiagThreads) vloc = fmaxf(vloc, a.vnorm[(size_t)g * a.nnz + lo + i]);
  const float vm = block_reduce<kDiagThreads>(vloc, red, true);
  if (tid == 0) {
    a.eps[(size_t)r * h_q + h] = tot > 0.f ? ex / tot : 0.f;
    a.topr[(size_t)r * h_q + h] = R > 0 ? (float)s_hits / (float)R : 0.f;
    if (h % a.group == 0) a.vmax[(size_t)r * a.h_kv + g] = vm;
  }
}

template <typename T, int D>
cudaError_t launch_d(const DiagArgs& a, cudaStream_t s) {
  const dim3 g1((a.nnz + kDiagPages - 1) / kDiagPages, a.h_kv);
  const unsigned g2 = (unsigned)a.batch * a.h_kv * a.group;
  if (a.page_size == 16) {
    if (a.nnz > 0) diag_pages_kernel<T, D, 16><<<g1, kDiagThreads, 0, s>>>(a);
    diag_reduce_kernel<16><<<g2, kDiagThreads, 0, s>>>(a);
  } else {
    if (a.nnz > 0) diag_pages_kernel<T, D, 32><<<g1, kDiagThreads, 0, s>>>(a);
    diag_reduce_kernel<32><<<g2, kDiagThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

size_t diag_workspace_bytes(int32_t h_kv, int32_t group, int32_t nnz, int32_t page_size) {
  const size_t hq = (size_t)h_kv * group, n = (size_t)nnz;
  auto up = [](size_t b) { return (b + 255) & ~(size_t)255; };
  return up(hq * n * page_size * sizeof(float)) + up(hq * n * sizeof(float2)) +
         up((size_t)h_kv * n * sizeof(float));
}

void diag_carve(DiagArgs& a, void* ws) {
  auto up = [](size_t b) { return (b + 255) & ~(size_t)255; };
  const size_t hq = (size_t)a.h_kv * a.group, n = (size_t)a.nnz;
  char* p = static_cast<char*>(ws);
  a.logits = reinterpret_cast<float*>(p);
  p += up(hq * n * a.page_size * sizeof(float));
  a.stats = reinterpret_cast<float2*>(p);
  p += up(hq * n * sizeof(float2));
  a.vnorm = reinterpret_cast<float*>(p);
}

cudaError_t launch_diag(const DiagArgs& a, cudaStream_t s) {
  if (a.batch == 0 || a.h_kv == 0) return cudaSuccess;
  if (a.dtype == QUEST_F16)
    return a.head_dim == 128 ? launch_d<__half, 128>(a, s) : launch_d<__half, 64>(a, s);
  return a.head_dim == 128 ? launch_d<float, 128>(a, s) : launch_d<float, 64>(a, s);
}

}  // namespace quest
