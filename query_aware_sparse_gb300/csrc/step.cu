// Fused decode step of one layer, one persistent launch:
//   a1 append of the new token (eq (8)) folded into the scoring of its page,
//   a2 page upper bounds U_p (Quest page §1.1 eq (2)-(3); GQA group max §2.1),
//   a3 Top-K pages per (request, KV head) (Quest page Fig. 1, §2),
//   a4 attention over the selected pages (Quest page Fig. 1, §2.1), and
//   a5 the log-sum-exp merge of its split-K partials (Quest page §2.1).
//
// Work order. The first NSEL CTAs are select workers; the others score a
// fixed slice of the page table for each KV head in turn (head-major), so
// head g is fully scored after about (g+1)/h_kv of the scoring time. Each
// scoring CTA adds its slice's page count to the unit's counter after every
// head; the select workers take the (request, KV head) units in head order,
// wait (bounded) until a unit's count is complete, run the block-wide select
// and publish a ready flag, so the selects of early heads overlap the
// scoring of later ones. All CTAs then claim attention items (unit, chunk of
// pages) from a queue in head order; an item waits (bounded) for its unit's
// flag, streams its pages in with bulk async copies and writes a partial; the
// CTA that finishes a unit's last chunk merges the partials into the output.
//
// The launch is cooperative, so every CTA is resident and the waits (select
// workers on scoring CTAs, attention items on select workers) always end.
// Cross-CTA hand-offs use release/acquire (fence + atomic, L2 loads); a
// proxy fence orders them before the bulk copies read the pool. Counters in
// the workspace are returned to zero by the last CTA that uses them.
#include "attn_dev.cuh"
#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace quest {
namespace {

constexpr int kNT = 256;              // threads per CTA
constexpr int kNW = kNT / 32;
constexpr int kNSS = 8;               // score ring stages (cp.async groups)
constexpr int kKeysCap = 8192;        // selector keys cached in shared memory
constexpr int kMaxSelectCtas = 16;    // select workers (no scoring)

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_all() {
  asm volatile("fence.proxy.async;" ::: "memory");
}

template <typename T, int D, int S, int G>
struct StepShape {
  using W = WarpAttn<T, D, S, G>;
  static constexpr int VEC = Elem<T>::kVec;
  static constexpr int LPP = D / VEC;                 // lanes per page when scoring
  static constexpr int PB = kNT / LPP;                // pages per score round
  static constexpr int NST = W::BLOCK_BYTES <= 4096 ? 2 : 1;   // attention pages per warp
  static constexpr int CP = kNW * NST;                // pages per attention item
  static constexpr int RING = kNSS * kNT * 32;        // m and M, 16 B each
  static constexpr int META = kNSS * kNT * 16;
  static constexpr int STAGES = kNW * NST * 2 * W::BLOCK_BYTES;
  static constexpr int MERGE = kNW * G * (D + 2) * 4;
  static constexpr int U0 = RING + META > STAGES ? RING + META : STAGES;
  static constexpr int UNION = U0 > MERGE ? U0 : MERGE;
  static constexpr int KEYS_OFF = UNION;
  static constexpr int BAR_OFF = KEYS_OFF + kKeysCap * 4;
  static constexpr int LOGIT_OFF = BAR_OFF + kNW * NST * 8;
  static constexpr int DESC_OFF = LOGIT_OFF + kNW * W::NV * 4;
  static constexpr int SMEM = DESC_OFF + kNW * NST * 8;
};

__device__ __forceinline__ int find_req(const int32_t* indptr, int lo, int hi, int e) {
  while (lo < hi) {                         // largest r in [lo, hi] with indptr[r] <= e
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(indptr + mid) <= e) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <typename T, int D, int S, int G>
__global__ void __launch_bounds__(kNT, 1)
step_kernel(const StepArgs a) {
  using Sh = StepShape<T, D, S, G>;
  using W = typename Sh::W;
  using KO = KeyOps<T>;
  constexpr int VEC = Sh::VEC, LPP = Sh::LPP, PB = Sh::PB, NST = Sh::NST, CP = Sh::CP;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ TopkSmem<kNT> tsm;
  __shared__ int s_rf, s_rl, s_item, s_last, s_ok;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nblk = gridDim.x, b = blockIdx.x;
  const int U = a.batch * a.h_kv;
  const int h_q = a.h_kv * G;
  unsigned* done = a.counters;              // [U] valid pages scored this call
  unsigned* ready = a.counters + U;         // [U] selection published
  unsigned* att_done = a.counters + 2 * U;  // [U] attention chunks finished
  unsigned* q_attn = a.counters + 3 * U;    // attention item queue head
  unsigned* exit_cnt = q_attn + 1;          // CTAs finished

  uint4* ring = reinterpret_cast<uint4*>(smem);                       // [NSS][NT][2]
  int4* meta = reinterpret_cast<int4*>(smem + Sh::RING);              // [NSS][NT]
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + Sh::KEYS_OFF);

  // ---------------- scoring (with the append folded in) ----------------
  const int nsel = min(U, kMaxSelectCtas);
  const bool selector = b < nsel;
  const int nscore = nblk - nsel;
  const int sb = b - nsel;                               // index among scoring CTAs
  const int per_cta = (a.nnz + nscore - 1) / nscore;
  const int s0 = selector ? 0 : min(a.nnz, sb * per_cta);
  const int s1 = selector ? 0 : min(a.nnz, s0 + per_cta);
  const int R = (s1 - s0 + PB - 1) / PB;                 // rounds per head
  const int total = a.h_kv * R;
  if (tid == 0) {
    s_rf = s1 > s0 ? find_req(a.page_indptr, 0, a.batch - 1, s0) : 0;
    s_rl = s1 > s0 ? find_req(a.page_indptr, 0, a.batch - 1, s1 - 1) : -1;
  }
  __syncthreads();
  const int rf = s_rf, rl = s_rl;
  const int pw = tid / LPP, sub = tid % LPP;

  auto issue = [&](int t) {
    const int stage = t % kNSS;
    int4 md = make_int4(-1, 0, 0, -1);        // pp, r, flags (1 valid, 2 tail), e
    if (t < total) {
      const int rd = t % R;
      const int e = s0 + rd * PB + pw;
      const int g = t / R;
      if (e < s1) {
        const int r = rf == rl ? rf : find_req(a.page_indptr, rf, rl, e);
        const int lp = e - __ldg(a.page_indptr + r);
        const int L = __ldg(a.seq_lens + r);
        const int P = (L + S - 1) / S;
        const int pp = __ldg(a.page_indices + e);
        md.y = r;
        md.w = e;
        if (lp < P) {
          if (pp >= 0 && pp < a.n_phys) {
            md.x = pp;
            md.z = 1 | ((a.k_new != nullptr && lp == P - 1) ? 2 : 0);
            const T* sp = static_cast<const T*>(a.summary) + ((size_t)pp * a.h_kv + g) * 2 * D + sub * VEC;
            cp_async16(&ring[(stage * kNT + tid) * 2 + 0], sp);
            cp_async16(&ring[(stage * kNT + tid) * 2 + 1], sp + D);
          } else if (sub == 0) {
            report(a.err, QUEST_DEVERR_PAGE_RANGE);
          }
        }
      }
    }
    meta[stage * kNT + tid] = md;
    cp_async_commit();
  };

  // Select worker: units in head order (k -> g = k / batch, r = k % batch).
  auto run_selects = [&]() {
    for (int k = b; k < U; k += nsel) {
      const int g = k / a.batch, r = k % a.batch;
      const int u = r * a.h_kv + g;
      const int lo = __ldg(a.page_indptr + r);
      const int tp = __ldg(a.page_indptr + r + 1) - lo;
      int P = (__ldg(a.seq_lens + r) + S - 1) / S;
      if (P > tp) {
        if (tid == 0) report(a.err, QUEST_DEVERR_TABLE_RANGE);
        P = tp;
      }
      if (tid == 0) {
        uint32_t it = 0;
        while (ld_acquire(done + u) < (unsigned)P && it < WAIT_LIMIT) { ++it; __nanosleep(32); }
        if (it >= WAIT_LIMIT) report(a.err, QUEST_DEVERR_WAIT_TIMEOUT);
      }
      __syncthreads();
      const int32_t* idx = a.page_indices + lo;
      block_topk<kNT>(a.scores + (size_t)g * a.nnz + lo, P, a.k, keys, kKeysCap, tsm,
                      a.sel_logical + (size_t)u * a.k, a.sel_phys + (size_t)u * a.k,
                      a.sel_count + u, [idx](int j) { return __ldg(idx + j); });
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        done[u] = 0;                         // reset for the next call
        st_release(ready + u, 1u);
      }
    }
  };

#pragma unroll 1
  for (int t = 0; t < kNSS - 1; ++t) issue(t);
  int cur_r = -1, cur_g = -1;
  float q[G][VEC];
#pragma unroll 1
  for (int t = 0; t < total; ++t) {
    issue(t + kNSS - 1);
    cp_async_wait<kNSS - 1>();
    const int stage = t % kNSS;
    const int g = t / R, rd = t % R;
    const int4 md = meta[stage * kNT + tid];
    const int r = md.y;
    float sg[G];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) sg[gi] = 0.f;
    if (md.z & 1) {
      if (r != cur_r || g != cur_g) {
        cur_r = r; cur_g = g;
        const T* qp = static_cast<const T*>(a.q) + ((size_t)r * h_q + (size_t)g * G) * D + sub * VEC;
#pragma unroll
        for (int gi = 0; gi < G; ++gi) unpack16<T>(ld_nc_v4(qp + (size_t)gi * D), q[gi]);
      }
      uint4 vm = ring[(stage * kNT + tid) * 2 + 0];
      uint4 vM = ring[(stage * kNT + tid) * 2 + 1];
      if (md.z & 2) {              // the new token lands in this (tail) page
        const int pos = __ldg(a.seq_lens + r) - 1;
        const int slot = pos % S;
        const size_t src = ((size_t)r * a.h_kv + g) * D + sub * VEC;
        const uint4 kn = ld_nc_v4(static_cast<const T*>(a.k_new) + src);
        const uint4 vn = ld_nc_v4(static_cast<const T*>(a.v_new) + src);
        const size_t dst = (((size_t)md.x * a.h_kv + g) * S + slot) * D + sub * VEC;
        st_v4(static_cast<T*>(a.k_pool) + dst, kn);
        st_v4(static_cast<T*>(a.v_pool) + dst, vn);
        uint4 mn, mx;
        if (slot == 0) {
          mn = make_uint4(KO::to_key(kn.x), KO::to_key(kn.y), KO::to_key(kn.z), KO::to_key(kn.w));
          mx = mn;
        } else {
          mn = make_uint4(KO::kmin(KO::to_key(vm.x), KO::to_key(kn.x)), KO::kmin(KO::to_key(vm.y), KO::to_key(kn.y)),
                          KO::kmin(KO::to_key(vm.z), KO::to_key(kn.z)), KO::kmin(KO::to_key(vm.w), KO::to_key(kn.w)));
          mx = make_uint4(KO::kmax(KO::to_key(vM.x), KO::to_key(kn.x)), KO::kmax(KO::to_key(vM.y), KO::to_key(kn.y)),
                          KO::kmax(KO::to_key(vM.z), KO::to_key(kn.z)), KO::kmax(KO::to_key(vM.w), KO::to_key(kn.w)));
        }
        vm = make_uint4(KO::from_key(mn.x), KO::from_key(mn.y), KO::from_key(mn.z), KO::from_key(mn.w));
        vM = make_uint4(KO::from_key(mx.x), KO::from_key(mx.y), KO::from_key(mx.z), KO::from_key(mx.w));
        T* sp = static_cast<T*>(a.summary) + ((size_t)md.x * a.h_kv + g) * 2 * D + sub * VEC;
        st_v4(sp, vm);
        st_v4(sp + D, vM);
      }
      float m[VEC], M[VEC];
      unpack16<T>(vm, m);
      unpack16<T>(vM, M);
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) sg[gi] += fmaxf(q[gi][v] * m[v], q[gi][v] * M[v]);
      }
    }
    // Sum each query head's bound over the LPP lanes of the page, then take
    // the group maximum (all lanes take part in the shuffles).
    float best = -INFINITY;
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
#pragma unroll
      for (int o = 1; o < LPP; o <<= 1) sg[gi] += __shfl_xor_sync(FULL, sg[gi], o);
      best = fmaxf(best, sg[gi]);
    }
    if (md.w >= 0 && sub == 0) a.scores[(size_t)g * a.nnz + md.w] = (md.z & 1) ? best : -INFINITY;

    if (rd == R - 1) {            // head g of this slice is scored
      __syncthreads();
      if (tid == 0 && rl >= rf) {
        __threadfence();
        for (int r2 = rf; r2 <= rl; ++r2) {
          const int lo = __ldg(a.page_indptr + r2);
          const int P = min((__ldg(a.seq_lens + r2) + S - 1) / S, __ldg(a.page_indptr + r2 + 1) - lo);
          const int n = min(s1, lo + P) - max(s0, lo);
          if (n > 0) atomicAdd(done + r2 * a.h_kv + g, (unsigned)n);
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  if (selector) run_selects();

  // ---------------- attention over the selected pages ----------------
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::BAR_OFF) + warp * NST;
  float* lg = reinterpret_cast<float*>(smem + Sh::LOGIT_OFF) + warp * W::NV;
  int2* desc = reinterpret_cast<int2*>(smem + Sh::DESC_OFF) + warp * NST;
  T* stage_base = reinterpret_cast<T*>(smem) + (size_t)warp * NST * 2 * S * D;
  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(bars + s, 1);
    fence_mbar_init();
  }
  unsigned phase = 0;                       // parity bit per slot
  const int NC = a.n_chunks;
  const int NA = U * NC;
  if (tid == 0) s_item = (int)atomicAdd(q_attn, 1u);
  __syncthreads();
  const size_t head_block = (size_t)S * D;
  const size_t page_stride = (size_t)a.h_kv * head_block;

#pragma unroll 1
  while (true) {
    const int item = s_item;
    if (item >= NA) break;
    unsigned next = 0;
    if (tid == 0) next = atomicAdd(q_attn, 1u);              // claim ahead
    const int c = item % NC;
    const int rest = item / NC;
    const int r = rest % a.batch, g = rest / a.batch;
    const int u = r * a.h_kv + g;
    if (tid == 0) {
      uint32_t it = 0;
      while (ld_acquire(ready + u) == 0u && it < WAIT_LIMIT) { ++it; __nanosleep(64); }
      s_ok = it < WAIT_LIMIT;
      if (!s_ok) report(a.err, QUEST_DEVERR_WAIT_TIMEOUT);
    }
    __syncthreads();
    const bool ok = s_ok;
    W st;
    st.init(static_cast<const T*>(a.q) + ((size_t)r * h_q + (size_t)g * G) * D, a.scale_log2, lane);
    if (ok) {
      const int L = __ldg(a.seq_lens + r);
      const int j0 = c * CP + warp * NST;
      int my_pp = -1, my_valid = 0;
      if (lane < NST && j0 + lane < a.k) {
        const int lp = __ldcg(a.sel_logical + (size_t)u * a.k + j0 + lane);
        const int pp = __ldcg(a.sel_phys + (size_t)u * a.k + j0 + lane);
        if (lp >= 0) {
          const int valid = min(S, L - lp * S);
          if (valid <= 0) report(a.err, QUEST_DEVERR_EMPTY_PAGE);
          else if (pp < 0 || pp >= a.n_phys) report(a.err, QUEST_DEVERR_PAGE_RANGE);
          else { my_pp = pp; my_valid = valid; }
        }
      }
      const unsigned vmask = __ballot_sync(FULL, my_valid > 0);
      const int nv = __popc(vmask);
      if (my_valid > 0) desc[__popc(vmask & ((1u << lane) - 1))] = make_int2(my_pp, my_valid);
      __syncwarp();
      if (lane == 0 && nv > 0) {
        fence_proxy_async_all();     // acquired pool writes and the reused stages
        const T* kb = static_cast<const T*>(a.k_pool) + (size_t)g * head_block;
        const T* vb = static_cast<const T*>(a.v_pool) + (size_t)g * head_block;
        for (int n = 0; n < nv; ++n) {
          T* dst = stage_base + (size_t)n * 2 * head_block;
          mbar_expect_tx(bars + n, 2 * W::BLOCK_BYTES);
          bulk_g2s(dst, kb + (size_t)desc[n].x * page_stride, W::BLOCK_BYTES, bars + n);
          bulk_g2s(dst + head_block, vb + (size_t)desc[n].x * page_stride, W::BLOCK_BYTES, bars + n);
        }
      }
      for (int n = 0; n < nv; ++n) {
        if (!mbar_wait_bounded(bars + n, (phase >> n) & 1u)) {
          if (lane == 0) report(a.err, QUEST_DEVERR_WAIT_TIMEOUT);
        } else {
          const T* Kb = stage_base + (size_t)n * 2 * head_block;
          st.page(Kb, Kb + head_block, desc[n].y, lg, lane);
        }
        phase ^= 1u << n;
      }
    }
    __syncthreads();                         // stages free: reuse for the merge
    float* mo = reinterpret_cast<float*>(smem);
    float* ml = mo + kNW * G * D;
    st.stash(mo, ml, warp, lane);
    __syncthreads();
    const size_t prow = ((size_t)u * G) * NC + c;            // (u, gi=0, c)
    merge_warps<D, G, kNW, kNT>(
        mo, ml,
        [&](int gi, int col, float o) { a.part_o[(prow + (size_t)gi * NC) * D + col] = o; },
        [&](int gi, float mx, float l) {
          a.part_ml[(prow + (size_t)gi * NC) * 2 + 0] = mx;
          a.part_ml[(prow + (size_t)gi * NC) * 2 + 1] = l;
        });
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      s_last = atomicAdd(att_done + u, 1u) == (unsigned)(NC - 1);
      s_item = (int)next;
    }
    __syncthreads();
    if (s_last) {                            // merge all chunks of unit u
      __threadfence();
      for (int idx = tid; idx < G * D; idx += kNT) {
        const int gi = idx / D, col = idx % D;
        const float* pml = a.part_ml + ((size_t)u * G + gi) * NC * 2;
        const float* po = a.part_o + ((size_t)u * G + gi) * NC * D + col;
        float mx = -INFINITY;
        for (int cc = 0; cc < NC; ++cc) mx = fmaxf(mx, __ldcg(pml + cc * 2));
        float o = 0.f, l = 0.f;
        if (mx != -INFINITY) {
          for (int cc = 0; cc < NC; ++cc) {
            const float mc = __ldcg(pml + cc * 2);
            if (mc == -INFINITY) continue;
            const float sc = exp2f(mc - mx);
            l = fmaf(sc, __ldcg(pml + cc * 2 + 1), l);
            o = fmaf(sc, __ldcg(po + (size_t)cc * D), o);
          }
        }
        const size_t orow = (size_t)r * h_q + (size_t)g * G + gi;
        a.out[orow * D + col] = l > 0.f ? o / l : 0.f;
        if (col == 0 && a.lse) a.lse[orow] = l > 0.f ? (mx + log2f(l)) * LN2 : -INFINITY;
      }
      if (tid == 0) {
        att_done[u] = 0;                     // reset for the next call
        ready[u] = 0;
      }
    }
    __syncthreads();
  }

  if (tid == 0) {
    __threadfence();
    if (atomicAdd(exit_cnt, 1u) == (unsigned)(nblk - 1)) {   // last CTA out
      *q_attn = 0;
      *exit_cnt = 0;
    }
  }
}

template <typename T, int D, int S, int G>
cudaError_t launch_t(const StepArgs& a, const StepPlan& p, cudaStream_t s) {
  using Sh = StepShape<T, D, S, G>;
  auto kern = step_kernel<T, D, S, G>;
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_done[64] = {};   // per device; racing setters write the same value
  if (dev >= 64 || !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kNT);
  cfg.dynamicSmemBytes = Sh::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident: the waits end
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T, int D, int S>
cudaError_t launch_g(const StepArgs& a, const StepPlan& p, cudaStream_t s) {
  switch (a.group) {
    case 1: return launch_t<T, D, S, 1>(a, p, s);
    case 2: return launch_t<T, D, S, 2>(a, p, s);
    case 4: return launch_t<T, D, S, 4>(a, p, s);
    case 8: return launch_t<T, D, S, 8>(a, p, s);
  }
  return cudaErrorInvalidValue;
}

template <typename T, int D>
cudaError_t launch_s(const StepArgs& a, const StepPlan& p, cudaStream_t s) {
  return a.page_size == 16 ? launch_g<T, D, 16>(a, p, s) : launch_g<T, D, 32>(a, p, s);
}

template <typename T, int D, int S>
int smem_g(int group) {
  switch (group) {
    case 1: return StepShape<T, D, S, 1>::SMEM;
    case 2: return StepShape<T, D, S, 2>::SMEM;
    case 4: return StepShape<T, D, S, 4>::SMEM;
    case 8: return StepShape<T, D, S, 8>::SMEM;
  }
  return 1 << 30;
}
template <typename T, int D, int S>
int cp_g(int group) {
  switch (group) {
    case 1: return StepShape<T, D, S, 1>::CP;
    case 2: return StepShape<T, D, S, 2>::CP;
    case 4: return StepShape<T, D, S, 4>::CP;
    case 8: return StepShape<T, D, S, 8>::CP;
  }
  return 1;
}
template <typename T, int D>
void shape_s(int S, int group, int* smem, int* cp) {
  if (S == 16) { *smem = smem_g<T, D, 16>(group); *cp = cp_g<T, D, 16>(group); }
  else { *smem = smem_g<T, D, 32>(group); *cp = cp_g<T, D, 32>(group); }
}

}  // namespace

StepPlan plan_step(int32_t batch, int32_t h_kv, int32_t group, int32_t head_dim,
                   int32_t page_size, int32_t dtype, int32_t k) {
  StepPlan p{};
  int smem = 0, cp = 1;
  if (dtype == QUEST_F16) {
    if (head_dim == 128) shape_s<__half, 128>(page_size, group, &smem, &cp);
    else shape_s<__half, 64>(page_size, group, &smem, &cp);
  } else {
    if (head_dim == 128) shape_s<float, 128>(page_size, group, &smem, &cp);
    else shape_s<float, 64>(page_size, group, &smem, &cp);
  }
  const long long units = (long long)batch * h_kv;
  int dev = 0, sms = 148, smem_sm = 228 * 1024;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  }
  cudaGetLastError();
  p.smem = smem;
  p.grid = sms;                                   // one CTA per SM
  p.ok = smem + 8 * 1024 <= 227 * 1024 && p.grid > kMaxSelectCtas;
  p.chunk_pages = cp;
  p.n_chunks = (k + cp - 1) / cp;
  p.counters_bytes = ((size_t)(3 * units + 2) * sizeof(unsigned) + 255) & ~(size_t)255;
  const size_t rows = (size_t)units * group * p.n_chunks;
  p.workspace_bytes = p.counters_bytes + rows * head_dim * sizeof(float) + rows * 2 * sizeof(float);
  p.workspace_bytes = (p.workspace_bytes + 255) & ~(size_t)255;
  return p;
}

cudaError_t launch_step(const StepArgs& a, const StepPlan& p, cudaStream_t s) {
  if (a.dtype == QUEST_F16)
    return a.head_dim == 128 ? launch_s<__half, 128>(a, p, s) : launch_s<__half, 64>(a, p, s);
  return a.head_dim == 128 ? launch_s<float, 128>(a, p, s) : launch_s<float, 64>(a, p, s);
}

}  // namespace quest
