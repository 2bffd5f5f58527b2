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
#include <cstdlib>

#include "attn_mma.cuh"
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

// GQA groups of 4 and 8 with fp16 queries: the bound as a contraction on the
// warp MMA, U = [m | M] . [q- ; q+] over the 2d summary elements (q- =
// min(q, 0), q+ = max(q, 0); m16n8k16, fp16 in, fp32 accumulate), the group's
// heads as the A rows and 8 pages as an n-tile. A persistent grid of two
// CTAs per SM; each warp streams its run of chunks of 8 table entries
// through a 3-deep ring of 16-byte cp.async copies into XOR-swizzled rows
// (conflict-free fragment reads). A chunk that spans requests runs the MMA
// once per request (each has its own query).
constexpr int kMmaWarps = 8;
constexpr int kMmaRing = 3;

template <int D, bool F8>
struct MmaScoreShape {
  static constexpr int ESS = F8 ? 1 : 2;         // bytes of a summary element
  static constexpr int SUMB = 2 * D * ESS;       // summary of one (page, KV head)
  static constexpr int CHB = 8 * SUMB;           // a chunk
  static constexpr int NCPY = CHB / 512;         // 16-byte pieces per lane
  static constexpr int KT = 2 * D / 16;          // k-steps
  static constexpr int SMEM = kMmaWarps * kMmaRing * CHB;
};

__device__ __forceinline__ void sc_cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void sc_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void sc_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }
template <int SUMB>
__device__ __forceinline__ int sc_sw(int p, int byte) {   // row p, 16-byte unit XOR (p mod 8)
  return p * SUMB + ((((byte >> 4) ^ (p & 7)) << 4) | (byte & 15));
}

template <int D, int G, bool F8, bool PH>
__global__ void __launch_bounds__(kMmaWarps * 32, 2)
score_mma_kernel(const ScoreArgs a) {
  using Sh = MmaScoreShape<D, F8>;
  constexpr int KT = Sh::KT, SUMB = Sh::SUMB, CHB = Sh::CHB;
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tq = lane & 3;
  unsigned char* ring = smem + (size_t)warp * kMmaRing * CHB;
  // chunks of 8 table entries of one KV head, head-major; warp w of the grid
  // takes the contiguous run [c_lo, c_hi) of them (persistent: the copies of
  // a run stream without a break)
  const int nchk = (a.nnz + 7) / 8;
  const long long total = (long long)nchk * a.h_kv;
  const long long gw = (long long)blockIdx.x * kMmaWarps + warp, nw = (long long)gridDim.x * kMmaWarps;
  const long long c_lo = total * gw / nw, c_hi = total * (gw + 1) / nw;
  const int n = (int)(c_hi - c_lo);
  // lane j < 8: entry j of the chunk: its request (found by walking forward
  // from the previous chunk's) and its physical page (-1: a reserved entry
  // past the request's valid pages, or past the table)
  int walk_g = -1, walk_r = 0;
  auto info = [&](int k, int& pp, int& rr) {
    pp = -1;
    rr = -1;
    const long long c = c_lo + k;
    const int g = (int)(c / nchk), e = (int)(c % nchk) * 8 + (lane & 7);
    if (lane < 8 && e < a.nnz) {
      if (g != walk_g) {                           // a run's first chunk of a head: search
        walk_g = g;
        walk_r = find_request(a.page_indptr, 0, a.batch - 1, e);
      }
      while (walk_r + 1 < a.batch && __ldg(a.page_indptr + walk_r + 1) <= e) ++walk_r;
      const int r = walk_r;
      const int lp = e - __ldg(a.page_indptr + r);
      const int valid_pages = (__ldg(a.seq_lens + r) + a.page_size - 1) / a.page_size;
      rr = r;
      if (lp < valid_pages) {
        const int p = __ldg(a.page_indices + e);
        if (p >= 0 && p < a.n_phys) pp = p;
        else report(a.err, QUEST_DEVERR_PAGE_RANGE);
      }
    }
  };
  auto issue = [&](int k, int pp) {
    const int g = (int)((c_lo + k) / nchk);
    unsigned char* dst = ring + (k % kMmaRing) * CHB;
#pragma unroll
    for (int q = 0; q < Sh::NCPY; ++q) {
      const int byte = q * 512 + lane * 16;
      const int j = byte / SUMB;
      const int phj = __shfl_sync(FULL, pp, j);
      if (phj >= 0)
        sc_cp_async16(dst + sc_sw<SUMB>(j, byte % SUMB),
                      static_cast<const unsigned char*>(a.summary) +
                          ((size_t)phj * a.h_kv + g) * SUMB + byte % SUMB);
    }
    sc_commit();
  };
  static_assert(kMmaRing == 3, "the chunk info rotates through three registers");
  int p0 = -1, r0 = -1, p1 = -1, r1 = -1, p2 = -1, r2 = -1;
  if (n > 0) { info(0, p0, r0); issue(0, p0); } else { sc_commit(); }
  if (n > 1) { info(1, p1, r1); issue(1, p1); } else { sc_commit(); }
  int cur_r = -1, cur_g = -1;
  uint32_t qa[KT], qb[KT];
  for (int k = 0; k < n; ++k) {
    if (k + 2 < n) {
      info(k + 2, p2, r2);
      issue(k + 2, p2);
    } else {
      sc_commit();
    }
    sc_wait<kMmaRing - 1>();
    __syncwarp();
    const long long c = c_lo + k;
    const int g = (int)(c / nchk), e0 = (int)(c % nchk) * 8;
    const unsigned char* sb = ring + (k % kMmaRing) * CHB;
    // this lane's columns: entries 2tq and 2tq + 1 of the chunk
    const int rA = __shfl_sync(FULL, r0, 2 * tq), rB = __shfl_sync(FULL, r0, 2 * tq + 1);
    float s0 = -INFINITY, s1 = -INFINITY;          // group max of those two
    float h0 = -INFINITY, h1 = -INFINITY;          // per head (PH): head gid's values
    unsigned todo = __ballot_sync(FULL, lane < 8 && r0 >= 0) & 0xffu;
    while (todo) {
      const int rq = __shfl_sync(FULL, r0, __ffs(todo) - 1);
      todo &= ~(__ballot_sync(FULL, lane < 8 && r0 == rq) & 0xffu);
      if (rq != cur_r || g != cur_g) {             // A fragments of this request's queries
        cur_r = rq;
        cur_g = g;
        const bool hv = gid < G;
        const __half* qh = static_cast<const __half*>(a.q) +
                           ((size_t)rq * a.h_kv * G + (size_t)g * G + (hv ? gid : 0)) * D;
        const __half2 z2 = __float2half2_rn(0.f);
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
          uint2 w = *reinterpret_cast<const uint2*>(qh + 16 * j + 4 * tq);
          if (!hv) w = make_uint2(0u, 0u);
          const __half2 x = *reinterpret_cast<const __half2*>(&w.x), y = *reinterpret_cast<const __half2*>(&w.y);
          const __half2 xn = __hmin2(x, z2), yn = __hmin2(y, z2), xp = __hmax2(x, z2), yp = __hmax2(y, z2);
          qa[j] = *reinterpret_cast<const uint32_t*>(&xn);
          qb[j] = *reinterpret_cast<const uint32_t*>(&yn);
          qa[j + D / 16] = *reinterpret_cast<const uint32_t*>(&xp);
          qb[j + D / 16] = *reinterpret_cast<const uint32_t*>(&yp);
        }
      }
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        uint32_t b0, b1;
        if constexpr (F8) {                         // 4 codes, decoded to fp16 pairs (exact)
          const uint32_t cw = *reinterpret_cast<const uint32_t*>(sb + sc_sw<SUMB>(gid, 16 * kk + 4 * tq));
          asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(b0) : "h"((uint16_t)cw));
          asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(b1) : "h"((uint16_t)(cw >> 16)));
        } else {
          const uint2 cw = *reinterpret_cast<const uint2*>(sb + sc_sw<SUMB>(gid, 32 * kk + 8 * tq));
          b0 = cw.x;
          b1 = cw.y;
        }
        if (kk & 1) mma_f16_16816(c1, qa[kk], 0u, qb[kk], 0u, b0, b1);
        else mma_f16_16816(c0, qa[kk], 0u, qb[kk], 0u, b0, b1);
      }
      // row gid (head gid if < G), columns 2tq, 2tq + 1
      float v0 = gid < G ? c0[0] + c1[0] : -INFINITY;
      float v1 = gid < G ? c0[1] + c1[1] : -INFINITY;
      if constexpr (PH) {
        if (rA == rq) h0 = v0;
        if (rB == rq) h1 = v1;
      } else {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          v0 = fmaxf(v0, __shfl_xor_sync(FULL, v0, o));
          v1 = fmaxf(v1, __shfl_xor_sync(FULL, v1, o));
        }
        if (rA == rq) s0 = v0;
        if (rB == rq) s1 = v1;
      }
    }
    // scores: reserved or unreadable entries get -inf
    const int ppA = __shfl_sync(FULL, p0, 2 * tq), ppB = __shfl_sync(FULL, p0, 2 * tq + 1);
    const int eA = e0 + 2 * tq, eB = eA + 1;
    if constexpr (PH) {
      if (gid < G) {
        float* row = a.scores + ((size_t)g * G + gid) * a.nnz;
        if (eA < a.nnz) row[eA] = ppA >= 0 ? h0 : -INFINITY;
        if (eB < a.nnz) row[eB] = ppB >= 0 ? h1 : -INFINITY;
      }
    } else if (gid == 0) {
      float* row = a.scores + (size_t)g * a.nnz;
      if (eA < a.nnz) row[eA] = ppA >= 0 ? s0 : -INFINITY;
      if (eB < a.nnz) row[eB] = ppB >= 0 ? s1 : -INFINITY;
    }
    __syncwarp();                                   // slot k % ring may be refilled
    p0 = p1; r0 = r1; p1 = p2; r1 = r2;
  }
  sc_wait<0>();
}

template <int D, bool F8>
cudaError_t launch_mma(const ScoreArgs& a, cudaStream_t s) {
  using Sh = MmaScoreShape<D, F8>;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long chunks = (long long)((a.nnz + 7) / 8) * a.h_kv;
  const long long want = (chunks + kMmaWarps - 1) / kMmaWarps;     // a chunk per warp at least
  dim3 grid((unsigned)(want < 2LL * sms ? want : 2LL * sms));       // two CTAs per SM
  const bool ph = a.per_head != 0;
  auto go = [&](auto kern) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, kMmaWarps * 32, Sh::SMEM, s>>>(a);
    return cudaGetLastError();
  };
  if (a.group == 4) return ph ? go(score_mma_kernel<D, 4, F8, true>) : go(score_mma_kernel<D, 4, F8, false>);
  return ph ? go(score_mma_kernel<D, 8, F8, true>) : go(score_mma_kernel<D, 8, F8, false>);
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
  if (a.dtype == QUEST_F16 && (a.group == 4 || a.group == 8) && !getenv("QUEST_SCORE_FMA")) {
    if (a.summary_fp8)
      return a.head_dim == 128 ? launch_mma<128, true>(a, s) : launch_mma<64, true>(a, s);
    return a.head_dim == 128 ? launch_mma<128, false>(a, s) : launch_mma<64, false>(a, s);
  }
  if (a.dtype == QUEST_F16 && a.summary_fp8)
    return a.head_dim == 128 ? launch_td<__half, 128, true>(a, s) : launch_td<__half, 64, true>(a, s);
  if (a.dtype == QUEST_F16)
    return a.head_dim == 128 ? launch_td<__half, 128, false>(a, s) : launch_td<__half, 64, false>(a, s);
  return a.head_dim == 128 ? launch_td<float, 128, false>(a, s) : launch_td<float, 64, false>(a, s);
}

}  // namespace quest
