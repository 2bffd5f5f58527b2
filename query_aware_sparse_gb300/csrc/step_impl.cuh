// Fused decode step of one layer, one persistent cooperative launch:
//   a1 append of the new token (eq (8)) folded into the scoring of its page,
//   a2 page upper bounds U_p (Quest page §1.1 eq (2)-(3); GQA group max §2.1),
//   a3 Top-K pages per (request, KV head) (Quest page Fig. 1, §2),
//   a4 attention over the selected pages (Quest page Fig. 1, §2.1), and
//   a5 the log-sum-exp merge of its split-K partials (Quest page §2.1).
//
// Roles. While there are at most one unit (request, KV head) per eight
// CTAs, the first NSEL = units CTAs only select and the others ("workers")
// score and then attend. With more units every CTA is a worker and also
// selects units after scoring.
//
// Scoring. Each worker scores an equal share of the (page, head) items of
// the page table, page-major with a fixed head per thread, so the query
// stays in registers. Start-up is two dependent loads deep (page table ->
// summary): the first items take their physical pages from the table while
// the slice's metadata is staged in shared memory. Summaries stream through
// a register pipeline PD items deep, so the loop never waits on a dependent
// load, a barrier or another CTA. Each score is also stored with the call's
// tag in the upper half of a 64-bit word: a reader tells a score of this
// call from a stale one without any fence on the writer's side. Each worker
// then bumps a "scored" counter with a release; a selecting CTA acquires it
// before reading its rows once (instead of polling it while the workers stream), so
// the appended K/V rows are ordered before the attention's copies of them.
//
// Selection. CTA b takes units b, b + grid, ... in head order: it waits for
// the complete scored count once, reads each unit's tagged row (batches of
// independent loads, re-polling only stale entries; key min and max reduced
// on the way), runs the block-wide Top-K and publishes the unit's ready flag
// (set to the tag) with a release store.
//
// Attention. The selected-page slots of all units, in head order, form one
// list; each worker takes an equal contiguous share. Its warps stream their
// pages with bulk async copies (cp.async.bulk + mbarrier), fold them with the
// online softmax and stash one state per (unit segment, warp); the CTA merges
// each segment into one partial. Per unit, a counter of processed slots
// (acquire-release fetch-and-add) tells the worker that completes the unit
// to merge all the unit's partials into the output, in one round trip to L2.
//
// The launch is cooperative, so every CTA is resident and every wait (select
// workers on scoring, attention on select workers) ends; each wait is also
// bounded and reports QUEST_DEVERR_WAIT_TIMEOUT instead of hanging.
// Publication is release/acquire; a proxy fence orders it before the bulk
// copies read the pool. The call tag lives in the workspace and is advanced
// by the selecting CTAs once every CTA has read it; the per-unit counters are reset
// by their last user and the scored counters are double-buffered by tag parity.
#pragma once

#include <cstdlib>
#include <type_traits>

#include "attn_dev.cuh"
#include "attn_mma.cuh"
#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace quest {
namespace {

constexpr int kNT = 256;              // threads per CTA
constexpr int kNW = kNT / 32;
constexpr int kKeysCap = 8192;        // selector keys cached in shared memory
constexpr int kSliceCap = 1024;       // slice pages whose metadata is staged at once
constexpr int kRounds = 1;            // attention rounds
constexpr int kMaxSeg = 4;            // unit segments per attention pass (G = 1)
constexpr int kTraceSlots = 16;

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
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_proxy_async_all() {
  asm volatile("fence.proxy.async;" ::: "memory");
}
// fetch-and-add that releases this CTA's prior writes (ordered before it by a
// barrier) and acquires those released by earlier adds to the same word
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// CTAs that only select (the rest score and attend): one per unit while
// the units are at most one CTA in eight; with more units every CTA scores
// and the selects are spread over all of them after scoring.
__host__ __device__ __forceinline__ int select_ctas(int units, int nblk) {
  const int n = nblk / 8 > 1 ? nblk / 8 : 1;
  return units <= n ? units : 0;
}


template <typename T, int D, int S, int G>
struct StepShape {
  using W = WarpAttn<T, D, S, G>;
  static constexpr int VEC = Elem<T>::kVec;
  // one CTA per SM (larger groups need the registers; stages of 8 KiB pages
  // do not fit twice): each thread then keeps more bytes in flight, with a
  // deeper scoring pipeline and, where they fit, two attention stages per warp
  static constexpr bool ONE = G >= 4 || S * D * (int)sizeof(T) > 4096;
  static constexpr int MINB = ONE ? 1 : 2;            // resident CTAs per SM
  static constexpr int NST = (ONE && 4 * kNW * W::BLOCK_BYTES <= 128 * 1024) ? 2 : 1;
  static constexpr int MAXSEG = kMaxSeg / G > 0 ? kMaxSeg / G : 1;
  // scoring: VPL 16-byte vectors of m (and of M) per lane, LPP lanes per
  // (page, head) item, IPR items per round, PD items in flight per thread
  static constexpr int VPL = G == 1 ? 2 : 1;
  static constexpr int PD = !ONE ? 2 : VPL == 2 ? 4 : G <= 4 ? 8 : 4;
  static constexpr int LPP = D * (int)sizeof(T) / (16 * VPL);
  static constexpr int IPR = kNT / LPP;
  static constexpr int WPL = 4 * VPL;                 // 32-bit words of m per lane
  // scoring-phase shared memory
  static constexpr int SMETA_OFF = 0;
  static constexpr int SCORE_END = SMETA_OFF + kSliceCap * 8;
  // attention-phase shared memory (same region)
  static constexpr int STAGES = kNW * NST * 2 * W::BLOCK_BYTES;
  static constexpr int STASH_O = STAGES;                                 // [MAXSEG][NW][G][D]
  static constexpr int STASH_ML = STASH_O + MAXSEG * kNW * G * D * 4;    // [MAXSEG][NW][G][2]
  static constexpr int ATT_END = STASH_ML + MAXSEG * kNW * G * 2 * 4;
  static constexpr int MAX_PARTS = MAXSEG * kNW * D - 2;   // final-merge weights fit the stash
  static constexpr int KEYS_END = kKeysCap * 8;              // keys + physical pages
  static constexpr int U1 = SCORE_END > ATT_END ? SCORE_END : ATT_END;
  static constexpr int UNION = U1 > KEYS_END ? U1 : KEYS_END;
  static constexpr int BAR_OFF = (UNION + 15) / 16 * 16;
  static constexpr int LOGIT_OFF = BAR_OFF + kNW * NST * 8;
  static constexpr int DESC_OFF = LOGIT_OFF + kNW * W::NV * 4;
  static constexpr int SMEM = DESC_OFF + kNW * 32 * 8;
};

__device__ __forceinline__ int find_req(const int32_t* indptr, int lo, int hi, int e) {
  while (lo < hi) {                         // largest r in [lo, hi] with indptr[r] <= e
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(indptr + mid) <= e) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Attention round: units [k0, k1) in head order, `len` = units * K slot
// positions over `nblk` worker CTAs; worker b owns positions [start(b),
// start(b+1)). With no more units than workers, unit u gets its own group of
// workers [u*nblk/units, (u+1)*nblk/units) and its K positions are split
// evenly inside the group, so no worker spans two units; otherwise the
// positions are split evenly over all workers.
struct Round {
  long long len;
  int k0, k1, nblk, K;
  __device__ bool aligned() const { return k1 - k0 <= nblk; }
  __device__ int group0(int u) const { return (int)((long long)u * nblk / (k1 - k0)); }
  __device__ long long start(int b) const {
    if (!aligned()) return (long long)b * len / nblk;
    const int nu = k1 - k0;
    const int u = (int)(((long long)(b + 1) * nu - 1) / nblk);   // largest u with group0(u) <= b
    if (u >= nu) return len;
    const int j = b - group0(u), n = group0(u + 1) - group0(u);
    return (long long)u * K + (long long)j * K / n;
  }
  __device__ int owner(long long p) const {      // largest b with start(b) <= p
    if (!aligned()) return (int)(((p + 1) * nblk - 1) / len);
    const int u = (int)(p / K), o = (int)(p % K);
    const int n = group0(u + 1) - group0(u);
    return group0(u) + (int)(((long long)(o + 1) * n - 1) / K);
  }
};

template <typename T, int D, int S, int G, bool F8>
__global__ void __launch_bounds__(kNT, StepShape<T, D, S, G>::MINB)
step_kernel(const StepArgs a) {
  static_assert(!F8 || sizeof(T) == 2, "E4M3 summaries take fp16 keys");
  using Sh = StepShape<T, D, S, G>;
  using W = typename Sh::W;
  using KO = KeyOps<T>;
  constexpr int VEC = Sh::VEC, NST = Sh::NST;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ TopkSmem<kNT> tsm;
  __shared__ int s_rf, s_rl, s_nlast, s_last[kMaxSeg];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nblk = gridDim.x, b = blockIdx.x;
  const int U = a.batch * a.h_kv;
  const int h_q = a.h_kv * G;
  const int K = a.k;
  const int NP = a.n_chunks;                // partial slots per unit
  // programmatic dependent launch: the next kernel on the stream may be
  // scheduled now (its CTAs take SMs as this grid's CTAs exit), and this
  // grid waits here until the previous kernel has completed and its writes
  // (pool, summaries, workspace counters) are visible
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  unsigned* epoch = a.counters;             // tag of the last call
  unsigned* ready = a.counters + 4;         // [U] tag of the published selection
  unsigned* att_done = ready + U;           // [U] attention slots finished
  // tags 1, 2, ..., 0xffffffff, 2, ...: 0 marks never-written entries and the
  // parity alternates from call to call
  unsigned tag = ld_relaxed_u32(epoch) + 1u;
  if (tag == 0u) tag = 2u;
  // CTAs counted in (a worker after scoring, a selector at once; released by
  // each), in one of two banks by tag parity: the bank of the next call was
  // last used by the previous call, which has finished, so this call clears
  // it (no exit protocol at the end)
  unsigned* scored_cnt = a.counters + 2 + (tag & 1u);
  if (b == 0 && tid == 0) a.counters[2 + ((tag + 1u) & 1u)] = 0u;
  // optional phase trace: kTraceSlots globaltimer stamps per CTA
  unsigned long long* trace = a.trace ? a.trace + (size_t)b * kTraceSlots : nullptr;
  auto stamp = [&](int i) { if (trace && tid == 0) trace[i] = global_ns(); };
  stamp(0);
  const uint64_t pol_stream = evict_first_policy();   // summaries and K/V pages: read once

  const int NSEL = select_ctas(U, nblk);    // CTAs [0, NSEL) select; the rest score and attend
  const bool selector = b < NSEL;
  // a selector has read the tag: count it in at once (a worker counts in
  // after scoring), so the complete count means every CTA has read the tag
  if (selector && tid == 0) red_release_add(scored_cnt, 1u);
  const int nbw = nblk - NSEL, bw = b - NSEL;

  // =================== scoring (with the append folded in) ===================
  // Worker bw scores an equal share [t0, t1) of the (page, head) items in
  // page-major order (entries [s0, s1) of the table). Items are taken IPR
  // per round, so with IPR % h_kv == 0 a thread keeps one head (and its
  // query registers) for the whole slice. Start-up is two dependent loads
  // deep: the first kPD items take their physical pages straight from the
  // page table, and the query and the slice's metadata load while those
  // summaries are in flight.
  constexpr int LPP = Sh::LPP, VPL = Sh::VPL, WPL = Sh::WPL, IPR = Sh::IPR, kPD = Sh::PD;
  const long long n_items = (long long)a.nnz * a.h_kv;
  const long long t0 = selector ? 0 : bw * n_items / nbw;
  const long long t1 = selector ? 0 : (bw + 1) * n_items / nbw;
  const int s0 = (int)(t0 / a.h_kv);
  const int s1 = t1 > t0 ? (int)((t1 - 1) / a.h_kv) + 1 : s0;
  if (tid == 0) {
    s_rf = s1 > s0 ? find_req(a.page_indptr, 0, a.batch - 1, s0) : 0;
    s_rl = s1 > s0 ? find_req(a.page_indptr, 0, a.batch - 1, s1 - 1) : -1;
  }
  __syncthreads();
  const int rf = s_rf, rl = s_rl;
  const int gp = tid / LPP, sub = tid % LPP;
  int2* smeta = reinterpret_cast<int2*>(smem + Sh::SMETA_OFF);           // [kSliceCap]

  // query of the current (request, head): per word a select mask (take M
  // where q >= 0) and the query values as fp32
  int q_r = -1, q_g = -1;
  constexpr int QV = WPL * 4 / (int)sizeof(T);        // query values per lane
  uint32_t qmask[G][WPL];
  float qf[G][QV];
  auto query_raw = [&](int r, int g, uint4 (&qr)[G][VPL]) {
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      const T* qp = static_cast<const T*>(a.q) + ((size_t)r * h_q + (size_t)g * G + gi) * D +
                    sub * VPL * VEC;
#pragma unroll
      for (int v = 0; v < VPL; ++v) qr[gi][v] = ld_nc_v4(qp + v * VEC);
    }
  };
  auto set_query = [&](int r, int g, const uint4 (&qr)[G][VPL]) {
    q_r = r; q_g = g;
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        const uint4 qv = qr[gi][v];
        const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if constexpr (sizeof(T) == 2) {
            qmask[gi][v * 4 + j] = ((~w[j] & 0x80008000u) >> 15) * 0xffffu;
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
            qf[gi][(v * 4 + j) * 2 + 0] = f.x;
            qf[gi][(v * 4 + j) * 2 + 1] = f.y;
          } else {
            qmask[gi][v * 4 + j] = (w[j] & 0x80000000u) ? 0u : 0xffffffffu;
            qf[gi][v * 4 + j] = __uint_as_float(w[j]);
          }
        }
      }
    }
  };
  auto load_query = [&](int r, int g) {
    uint4 qr[G][VPL];
    query_raw(r, g, qr);
    set_query(r, g, qr);
  };

  uint4 bm[kPD][F8 ? 1 : VPL], bM[kPD][F8 ? 1 : VPL];
  int sl_i[kPD], sl_g[kPD];                  // page (n = none) and head of each slot

#pragma unroll 1
  for (int seg0 = s0; seg0 < s1; seg0 += kSliceCap) {
    const int seg1 = min(s1, seg0 + kSliceCap);
    const int n = seg1 - seg0;
    const long long ta = max(t0, (long long)seg0 * a.h_kv);   // the segment's items [ta, tb)
    const int nit = (int)(min(t1, (long long)seg1 * a.h_kv) - ta);
    const int rounds = (nit + IPR - 1) / IPR;
    const int dg = IPR % a.h_kv, di = IPR / a.h_kv;
    __syncthreads();                        // previous segment's metadata consumed
    // walker over the thread's items ta + ti (issued kPD ahead of their use):
    // page seg0 + ii, head ig; the physical page comes from smem, or from
    // the table before it is staged
    const int rel0 = (int)(ta - (long long)seg0 * a.h_kv) + gp;
    int ti = gp, ig = rel0 % a.h_kv, ii = rel0 / a.h_kv;
    auto issue = [&](int u, bool staged) {
      int ip = n;
      if (ti < nit) {
        ip = ii;
        const int x = staged ? smeta[ii].x : __ldg(a.page_indices + seg0 + ii);
        if (x >= 0 && x < a.n_phys) {        // reserved entries load harmlessly
          if constexpr (F8) {                // the codes of the lane's VPL * VEC dims
            const uint8_t* sp = static_cast<const uint8_t*>(a.summary) +
                                ((size_t)x * a.h_kv + ig) * 2 * D + sub * VPL * VEC;
            if constexpr (VPL == 2) {
              bm[u][0] = ld_stream_v4_hint(sp, pol_stream);
              bM[u][0] = ld_stream_v4_hint(sp + D, pol_stream);
            } else {
              const uint2 cm = ld_stream_v2_hint(sp, pol_stream), cM = ld_stream_v2_hint(sp + D, pol_stream);
              bm[u][0] = make_uint4(cm.x, cm.y, 0u, 0u);
              bM[u][0] = make_uint4(cM.x, cM.y, 0u, 0u);
            }
          } else {
            const T* sp = static_cast<const T*>(a.summary) + ((size_t)x * a.h_kv + ig) * 2 * D + sub * VPL * VEC;
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
              bm[u][v] = ld_stream_v4_hint(sp + v * VEC, pol_stream);
              bM[u][v] = ld_stream_v4_hint(sp + D + v * VEC, pol_stream);
            }
          }
        }
      }
      sl_i[u] = ip; sl_g[u] = ig;
      ti += IPR; ig += dg; ii += di;
      if (ig >= a.h_kv) { ig -= a.h_kv; ++ii; }
    };
#pragma unroll
    for (int u = 0; u < kPD; ++u) issue(u, false);
    // the first item's query (its request is usually the slice's first):
    // loaded now, converted once the metadata is staged
    const bool pre_q = seg0 == s0 && sl_i[0] < n;
    uint4 qr0[G][VPL];
    if (pre_q) query_raw(rf, sl_g[0], qr0);
    for (int e = seg0 + tid; e < seg1; e += kNT) {
      const int r = rf == rl ? rf : find_req(a.page_indptr, rf, rl, e);
      const int lp = e - __ldg(a.page_indptr + r);
      const int P = (__ldg(a.seq_lens + r) + S - 1) / S;
      const int pp = __ldg(a.page_indices + e);
      int flags = 0, phys = -1;
      if (lp < P) {
        if (pp >= 0 && pp < a.n_phys) {
          flags = 1 | ((a.k_new != nullptr && lp == P - 1) ? 2 : 0);
          phys = pp;
        } else {
          report(a.err, QUEST_DEVERR_PAGE_RANGE);
        }
      }
      smeta[e - seg0] = make_int2(phys, r | (flags << 24));
    }
    if (pre_q) set_query(rf, sl_g[0], qr0);
    __syncthreads();
#pragma unroll 1
    for (int k0 = 0; k0 < rounds; k0 += kPD) {
#pragma unroll
      for (int u = 0; u < kPD; ++u) {
        if (k0 + u < rounds) {               // CTA-uniform
          // take everything of item k out of slot u before refilling it
          const int g = sl_g[u], i = sl_i[u];
          uint4 vm[VPL], vM[VPL];
#pragma unroll
          for (int v = 0; v < (F8 ? 1 : VPL); ++v) { vm[v] = bm[u][v]; vM[v] = bM[u][v]; }
          issue(u, true);                    // refill the slot kPD items ahead
          const int2 md = i < n ? smeta[i] : make_int2(-1, 0);
          const int flags = md.y >> 24;
          const int r = md.y & 0xffffff, pp = md.x;
          float sg[G];
#pragma unroll
          for (int gi = 0; gi < G; ++gi) sg[gi] = 0.f;
          if (flags & 1) {
            if (r != q_r || g != q_g) load_query(r, g);
            if (flags & 2) {                 // the new token lands in this (tail) page
              const int pos = __ldg(a.seq_lens + r) - 1;
              const int slot = pos % S;
              const size_t src = ((size_t)r * a.h_kv + g) * D + sub * VPL * VEC;
              const size_t dst = (((size_t)pp * a.h_kv + g) * S + slot) * D + sub * VPL * VEC;
              T* sp = static_cast<T*>(a.summary) + ((size_t)pp * a.h_kv + g) * 2 * D + sub * VPL * VEC;
              uint32_t c8m[2 * VPL], c8M[2 * VPL];   // E4M3: new codes of the lane's dims
              bool ovf = false;
#pragma unroll
              for (int v = 0; v < VPL; ++v) {
                const uint4 kn = ld_nc_v4(static_cast<const T*>(a.k_new) + src + v * VEC);
                const uint4 vn = ld_nc_v4(static_cast<const T*>(a.v_new) + src + v * VEC);
                st_v4(static_cast<T*>(a.k_pool) + dst + v * VEC, kn);
                st_v4(static_cast<T*>(a.v_pool) + dst + v * VEC, vn);
                if constexpr (F8) {
                  // the old codes of these 8 dims decode exactly to fp16; fold
                  // the new key in, then round out again (min down, max up)
                  const uint32_t kw[4] = {kn.x, kn.y, kn.z, kn.w};
#pragma unroll
                  for (int h = 0; h < 2; ++h) {
                    const int cw = v * 2 + h;          // code word: dims 4cw .. 4cw+3
                    const uint32_t om = cw == 0 ? vm[0].x : cw == 1 ? vm[0].y : cw == 2 ? vm[0].z : vm[0].w;
                    const uint32_t oM = cw == 0 ? vM[0].x : cw == 1 ? vM[0].y : cw == 2 ? vM[0].z : vM[0].w;
                    uint32_t m01 = KO::to_key(kw[2 * h]), m23 = KO::to_key(kw[2 * h + 1]);
                    uint32_t M01 = m01, M23 = m23;
                    if (slot != 0) {
                      m01 = KO::kmin(KO::to_key(e4m3x4_lo_h2(om)), m01);
                      m23 = KO::kmin(KO::to_key(e4m3x4_hi_h2(om)), m23);
                      M01 = KO::kmax(KO::to_key(e4m3x4_lo_h2(oM)), M01);
                      M23 = KO::kmax(KO::to_key(e4m3x4_hi_h2(oM)), M23);
                    }
                    c8m[cw] = e4m3x4_floor_h(KO::from_key(m01), KO::from_key(m23), ovf);
                    c8M[cw] = e4m3x4_ceil_h(KO::from_key(M01), KO::from_key(M23), ovf);
                  }
                  continue;
                }
                uint4 mn, mx;
                if (slot == 0) {
                  mn = make_uint4(KO::to_key(kn.x), KO::to_key(kn.y), KO::to_key(kn.z), KO::to_key(kn.w));
                  mx = mn;
                } else {
                  mn = make_uint4(KO::kmin(KO::to_key(vm[v].x), KO::to_key(kn.x)), KO::kmin(KO::to_key(vm[v].y), KO::to_key(kn.y)),
                                  KO::kmin(KO::to_key(vm[v].z), KO::to_key(kn.z)), KO::kmin(KO::to_key(vm[v].w), KO::to_key(kn.w)));
                  mx = make_uint4(KO::kmax(KO::to_key(vM[v].x), KO::to_key(kn.x)), KO::kmax(KO::to_key(vM[v].y), KO::to_key(kn.y)),
                                  KO::kmax(KO::to_key(vM[v].z), KO::to_key(kn.z)), KO::kmax(KO::to_key(vM[v].w), KO::to_key(kn.w)));
                }
                vm[v] = make_uint4(KO::from_key(mn.x), KO::from_key(mn.y), KO::from_key(mn.z), KO::from_key(mn.w));
                vM[v] = make_uint4(KO::from_key(mx.x), KO::from_key(mx.y), KO::from_key(mx.z), KO::from_key(mx.w));
                st_v4(sp + v * VEC, vm[v]);
                st_v4(sp + D + v * VEC, vM[v]);
              }
              if constexpr (F8) {
                uint8_t* sp8 = static_cast<uint8_t*>(a.summary) +
                               ((size_t)pp * a.h_kv + g) * 2 * D + sub * VPL * VEC;
                if constexpr (VPL == 2) {
                  vm[0] = make_uint4(c8m[0], c8m[1], c8m[2], c8m[3]);
                  vM[0] = make_uint4(c8M[0], c8M[1], c8M[2], c8M[3]);
                  st_v4(sp8, vm[0]);
                  st_v4(sp8 + D, vM[0]);
                } else {
                  vm[0] = make_uint4(c8m[0], c8m[1], 0u, 0u);
                  vM[0] = make_uint4(c8M[0], c8M[1], 0u, 0u);
                  st_v2(sp8, make_uint2(c8m[0], c8m[1]));
                  st_v2(sp8 + D, make_uint2(c8M[0], c8M[1]));
                }
                if (ovf) report(a.err, QUEST_DEVERR_FP8_RANGE);
              }
            }
            // sum_j max(q_j m_j, q_j M_j) = sum_j q_j * (q_j >= 0 ? M_j : m_j)
            if constexpr (F8) {              // codes decoded to fp16 (exact), FMA in fp32
              const uint32_t mw[4] = {vm[0].x, vm[0].y, vm[0].z, vm[0].w};
              const uint32_t Mw[4] = {vM[0].x, vM[0].y, vM[0].z, vM[0].w};
#pragma unroll
              for (int cw = 0; cw < 2 * VPL; ++cw) {
#pragma unroll
                for (int gi = 0; gi < G; ++gi) {
                  const uint32_t sel = e4m3_qsel_from_masks(qmask[gi][2 * cw], qmask[gi][2 * cw + 1]);
                  const uint32_t xw = (Mw[cw] & sel) | (mw[cw] & ~sel);
                  const float2 lo = e4m3x4_lo_f2(xw), hi = e4m3x4_hi_f2(xw);
                  sg[gi] = fmaf(qf[gi][4 * cw + 0], lo.x, sg[gi]);
                  sg[gi] = fmaf(qf[gi][4 * cw + 1], lo.y, sg[gi]);
                  sg[gi] = fmaf(qf[gi][4 * cw + 2], hi.x, sg[gi]);
                  sg[gi] = fmaf(qf[gi][4 * cw + 3], hi.y, sg[gi]);
                }
              }
            } else {
#pragma unroll
              for (int v = 0; v < VPL; ++v) {
                const uint32_t mw[4] = {vm[v].x, vm[v].y, vm[v].z, vm[v].w};
                const uint32_t Mw[4] = {vM[v].x, vM[v].y, vM[v].z, vM[v].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
#pragma unroll
                  for (int gi = 0; gi < G; ++gi) {
                    const uint32_t mk = qmask[gi][v * 4 + j];
                    const uint32_t xw = (Mw[j] & mk) | (mw[j] & ~mk);
                    if constexpr (sizeof(T) == 2) {
                      const float2 xf = __half22float2(*reinterpret_cast<const __half2*>(&xw));
                      sg[gi] = fmaf(qf[gi][(v * 4 + j) * 2 + 0], xf.x, sg[gi]);
                      sg[gi] = fmaf(qf[gi][(v * 4 + j) * 2 + 1], xf.y, sg[gi]);
                    } else {
                      sg[gi] = fmaf(qf[gi][v * 4 + j], __uint_as_float(xw), sg[gi]);
                    }
                  }
                }
              }
            }
          }
          float best = -INFINITY;
#pragma unroll
          for (int gi = 0; gi < G; ++gi) {
#pragma unroll
            for (int o = 1; o < LPP; o <<= 1) sg[gi] += __shfl_xor_sync(FULL, sg[gi], o);
            best = fmaxf(best, sg[gi]);
          }
          if (i < n && sub == 0) {
            const float sc = (flags & 1) ? best : -INFINITY;
            const size_t at = (size_t)g * a.nnz + seg0 + i;
            a.scores[at] = sc;
            st_relaxed_u64(a.tagged + at, ((unsigned long long)tag << 32) | __float_as_uint(sc));
          }
        }
      }
    }
  }
  __syncthreads();
  // release: the appends and tagged scores of this worker happen before a
  // selector's acquire of the count (and so before the attention that
  // follows the selection)
  if (!selector && tid == 0) red_release_add(scored_cnt, 1u);
  stamp(1);

  // ============ selection (CTA b takes units b, b + nblk, ... in head order) ============
  // with dedicated selectors these are exactly the selectors' units
  if (b < U) {
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem);                      // [kKeysCap]
    int32_t* physs = reinterpret_cast<int32_t*>(smem + kKeysCap * 4);        // [kKeysCap]
    for (int i = tid; i < kTopkBins; i += kNT) tsm.hist[i] = 0;   // block_topk_smem keeps it zero
    for (int kk = b; kk < U; kk += nblk) {
      const int g = kk / a.batch, r = kk % a.batch;
      const int u = r * a.h_kv + g;
      const int lo = __ldg(a.page_indptr + r);
      const int tp = __ldg(a.page_indptr + r + 1) - lo;
      int P = (__ldg(a.seq_lens + r) + S - 1) / S;
      if (P > tp) {
        if (tid == 0) report(a.err, QUEST_DEVERR_TABLE_RANGE);
        P = tp;
      }
      const unsigned long long* row = a.tagged + (size_t)g * a.nnz + lo;
      const int32_t* idx = a.page_indices + lo;
      const bool cached = P <= kKeysCap;
      // local window + sink pages (hybrid budget) are kept outright:
      // forced = [0, f_lo) and [f_hi, P)
      const int f_lo = min(a.n_sink, P), f_hi = max(f_lo, P - a.n_local);
      auto forced = [f_lo, f_hi](int i) { return i < f_lo || i >= f_hi; };
      // gate: one thread waits (bounded) until every worker has finished
      // scoring, so the block reads the row once instead of polling it while
      // the workers stream; the row's tags still decide below
      if (tid == 0 && kk == b) {
        for (uint32_t it = 0; ld_acquire(scored_cnt) < (unsigned)nblk && it < (1u << 20); ++it)
          __nanosleep(128);
        // every CTA read the epoch before its release of this count: advance it
        *epoch = tag;
      }
      __syncthreads();
      // each thread waits for its own entries to carry this call's tag: a
      // batch of PB independent loads (with the entries' physical pages),
      // then a re-poll of only those still stale; the keys' min and max are
      // reduced on the way
      constexpr int PB = 8;
      bool late = false;
      uint32_t kmin = 0xffffffffu, kmax = 0u;
      for (int i0 = tid; i0 < P; i0 += kNT * PB) {
        unsigned long long v[PB];
        int32_t ph[PB];
#pragma unroll
        for (int j = 0; j < PB; ++j) {
          const int i = i0 + j * kNT;
          v[j] = i < P ? ld_relaxed_u64(row + i) : (unsigned long long)tag << 32;
          ph[j] = (cached && i < P) ? __ldg(idx + i) : 0;
        }
#pragma unroll
        for (int j = 0; j < PB; ++j) {
          const int i = i0 + j * kNT;
          // after one wait has run out the rest take what is there: a stuck
          // row costs one limit, not one per entry
          for (uint32_t it = 0; !late && (unsigned)(v[j] >> 32) != tag; ++it) {
            if (it >= WAIT_LIMIT) { late = true; break; }
            __nanosleep(32);
            v[j] = ld_relaxed_u64(row + i);
          }
          if (cached && i < P) {
            const uint32_t key = score_key(__uint_as_float((unsigned)v[j]));
            keys[i] = key;
            physs[i] = ph[j];
            if (i >= f_lo && i < f_hi) {     // min/max over the pages that compete
              kmin = min(kmin, key);
              kmax = max(kmax, key);
            }
          }
        }
      }
      if (late) report(a.err, QUEST_DEVERR_WAIT_TIMEOUT);
      kmin = warp_min_u32(kmin);
      kmax = warp_max_u32(kmax);
      if (lane == 0) { tsm.red[0][warp] = kmin; tsm.red[1][warp] = kmax; }
      __syncthreads();
#pragma unroll
      for (int w = 0; w < kNW; ++w) { kmin = min(kmin, tsm.red[0][w]); kmax = max(kmax, tsm.red[1][w]); }
      const int nth = (kk - b) / nblk;       // this CTA's n-th select
      if (nth == 0) stamp(6);
      if (selector && nth < 3) stamp(10 + 2 * nth);
      int32_t* ol = a.sel_logical + (size_t)u * K;
      int32_t* op = a.sel_phys + (size_t)u * K;
      const int nsel = min(P, K);
      for (int q = nsel + tid; q < K; q += kNT) { ol[q] = -1; op[q] = -1; }
      if (tid == 0) a.sel_count[u] = nsel;
      auto emit = [&](int pos, int i) { ol[pos] = i; op[pos] = cached ? physs[i] : __ldg(idx + i); };
      if (cached)
        block_topk_smem<kNT>(P, K, keys, kmin, kmax, tsm, emit, forced, f_lo + (P - f_hi));
      else
        block_topk_keys<kNT>(P, K, [row, forced](int i) {
                               return forced(i) ? 0xffffffffu
                                                : score_key(__uint_as_float((unsigned)ld_relaxed_u64(row + i)));
                             }, tsm, emit);
      __syncthreads();
      if (tid == 0) st_release(ready + u, tag);   // releases the block's selection writes
      if (selector && nth < 3) stamp(11 + 2 * nth);
      stamp(7);
    }
    __syncthreads();
  }
  stamp(2);

  // =================== attention over the selected pages ===================
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::BAR_OFF) + warp * NST;
  float* lg = reinterpret_cast<float*>(smem + Sh::LOGIT_OFF) + warp * W::NV;
  int2* desc = reinterpret_cast<int2*>(smem + Sh::DESC_OFF) + warp * 32;
  T* stage_base = reinterpret_cast<T*>(smem) + (size_t)warp * NST * 2 * S * D;
  float* stash_o = reinterpret_cast<float*>(smem + Sh::STASH_O);
  float* stash_ml = reinterpret_cast<float*>(smem + Sh::STASH_ML);
  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(bars + s, 1);
    fence_mbar_init();
  }
  __syncwarp();
  unsigned phase = 0;                       // parity bit per slot
  const size_t head_block = (size_t)S * D;
  const size_t page_stride = (size_t)a.h_kv * head_block;
  const int nrounds = selector ? 0 : min(kRounds, U);

#pragma unroll 1
  for (int qr = 0; qr < nrounds; ++qr) {
    Round rd;
    rd.k0 = (int)((long long)qr * U / nrounds);
    rd.k1 = (int)((long long)(qr + 1) * U / nrounds);
    rd.len = (long long)(rd.k1 - rd.k0) * K;
    rd.nblk = nbw;
    rd.K = K;
    const long long pb = rd.start(bw), pe = rd.start(bw + 1);   // relative to unit k0
#pragma unroll 1
    for (long long pa = pb; pa < pe;) {
      // one pass: the positions [pa, pz) of at most MAXSEG consecutive units
      const int ka = (int)(pa / K);
      const int kb = min((int)((pe - 1) / K), ka + Sh::MAXSEG - 1);
      const long long pz = min(pe, (long long)(kb + 1) * K);
      const int ns = kb - ka + 1;
      const int npass = (int)(pz - pa);
      if (tid == 0) {                        // the pass's units must be selected
        for (int s = 0; s < ns; ++s) {
          const int kk = rd.k0 + ka + s;
          const int u = (kk % a.batch) * a.h_kv + kk / a.batch;
          uint32_t it = 0;
          while (ld_acquire(ready + u) != tag && it < WAIT_LIMIT) { ++it; __nanosleep(64); }
          if (it >= WAIT_LIMIT) report(a.err, QUEST_DEVERR_WAIT_TIMEOUT);
        }
      }
      if (pa == pb && qr == 0) stamp(3);
      // every warp starts each segment of the pass empty
      for (int s = 0; s < ns; ++s) {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
          for (int col = lane; col < D; col += 32)
            stash_o[((s * kNW + warp) * G + gi) * D + col] = 0.f;
          if (lane == 0) {
            stash_ml[((s * kNW + warp) * G + gi) * 2 + 0] = -INFINITY;
            stash_ml[((s * kNW + warp) * G + gi) * 2 + 1] = 0.f;
          }
        }
      }
      __syncthreads();
      // fp16 groups of 4 or 8 query heads: QK and AV on the warp MMA, each
      // page loaded straight into registers (a second page in flight spills)
      constexpr bool kMma = sizeof(T) == 2 && G >= 4 && S == 16;
      using WA = std::conditional_t<kMma, WarpAttnMma<D, G>, W>;
      WA st;
      int cs = -1;                           // segment of the running state
#pragma unroll 1
      for (int base = 0; base * kNW < npass; base += 32) {
        // descriptors of this warp's next (up to) 32 pages: i = warp + NW*(base+lane)
        int my_pp = -1, my_val = 0;
        const int i = warp + kNW * (base + lane);
        if (i < npass) {
          const long long pos = pa + i;
          const int kk = rd.k0 + (int)(pos / K);
          const int j = (int)(pos % K);
          const int r = kk % a.batch, g = kk / a.batch;
          const int u = r * a.h_kv + g;
          const int lp = __ldcg(a.sel_logical + (size_t)u * K + j);
          const int pp = __ldcg(a.sel_phys + (size_t)u * K + j);
          if (lp >= 0) {
            const int valid = min(S, __ldg(a.seq_lens + r) - lp * S);
            if (valid <= 0) report(a.err, QUEST_DEVERR_EMPTY_PAGE);
            else if (pp < 0 || pp >= a.n_phys) report(a.err, QUEST_DEVERR_PAGE_RANGE);
            else { my_pp = pp; my_val = valid | ((kk - rd.k0 - ka) << 8); }
          }
        }
        const unsigned vmask = __ballot_sync(FULL, my_val > 0);
        const int nv = __popc(vmask);
        if (my_val > 0) desc[__popc(vmask & ((1u << lane) - 1))] = make_int2(my_pp, my_val);
        __syncwarp();
        if (pa == pb && base == 0) stamp(10);
        auto set_seg = [&](int n) {
          const int seg = desc[n].y >> 8;
          if (seg != cs) {                   // unit changes: stash the running state
            if (cs >= 0)
              st.stash(stash_o + (size_t)cs * kNW * G * D, stash_ml + (size_t)cs * kNW * G * 2, warp, lane);
            const int kk = rd.k0 + ka + seg;
            const int r = kk % a.batch, g = kk / a.batch;
            st.init(static_cast<const T*>(a.q) + ((size_t)r * h_q + (size_t)g * G) * D, a.scale_log2, lane);
            cs = seg;
          }
        };
        if constexpr (kMma) {
          typename WA::Page pA;
          auto load = [&](int n, typename WA::Page& pg) {
            const int kk = rd.k0 + ka + (desc[n].y >> 8);
            const size_t off = (size_t)desc[n].x * page_stride + (size_t)(kk / a.batch) * head_block;
            WA::load(static_cast<const T*>(a.k_pool) + off, static_cast<const T*>(a.v_pool) + off, lane,
                     pol_stream, pg);
          };
          for (int n = 0; n < nv; ++n) {
            load(n, pA);
            set_seg(n);
            st.page(pA, desc[n].y & 0xff, lg, lane);
            if (pa == pb && base == 0 && n == 0) stamp(11);
          }
          __syncwarp();
          continue;
        } else {
        auto issue = [&](int n) {
          const int slot = n % NST;
          const int kk = rd.k0 + ka + (desc[n].y >> 8);
          const int g = kk / a.batch;
          T* dst = stage_base + (size_t)slot * 2 * head_block;
          const size_t off = (size_t)desc[n].x * page_stride + (size_t)g * head_block;
          mbar_expect_tx(bars + slot, 2 * W::BLOCK_BYTES);
          bulk_g2s_hint(dst, static_cast<const T*>(a.k_pool) + off, W::BLOCK_BYTES, bars + slot, pol_stream);
          bulk_g2s_hint(dst + head_block, static_cast<const T*>(a.v_pool) + off, W::BLOCK_BYTES, bars + slot, pol_stream);
        };
        if (lane == 0 && nv > 0) {
          fence_proxy_async_all();           // acquired pool writes and reused stages
          for (int n = 0; n < min(NST, nv); ++n) issue(n);
        }
        for (int n = 0; n < nv; ++n) {
          const int slot = n % NST;
          set_seg(n);
          if (!mbar_wait_bounded(bars + slot, (phase >> slot) & 1u)) {
            if (lane == 0) report(a.err, QUEST_DEVERR_WAIT_TIMEOUT);
          } else {
            const T* Kb = stage_base + (size_t)slot * 2 * head_block;
            st.page(Kb, Kb + head_block, desc[n].y & 0xff, lg, lane);
          }
          if (pa == pb && base == 0 && n == 0) stamp(11);
          phase ^= 1u << slot;
          __syncwarp();
          if (lane == 0 && n + NST < nv) {
            fence_proxy_async_all();
            issue(n + NST);
          }
        }
        __syncwarp();
        }
      }
      if (cs >= 0)
        st.stash(stash_o + (size_t)cs * kNW * G * D, stash_ml + (size_t)cs * kNW * G * 2, warp, lane);
      __syncthreads();
      if (qr == 0) stamp(4);

      // merge each segment's warps into this CTA's partial of the unit
      for (int s = 0; s < ns; ++s) {
        const int kk = rd.k0 + ka + s;
        const int u = (kk % a.batch) * a.h_kv + kk / a.batch;
        const int pslot = bw - rd.owner((long long)(ka + s) * K);
        const size_t prow = (size_t)u * G * NP + pslot;          // (u, gi = 0, pslot)
        merge_warps<D, G, kNW, kNT>(
            stash_o + (size_t)s * kNW * G * D, stash_ml + (size_t)s * kNW * G * 2,
            [&](int gi, int col, float o) { a.part_o[(prow + (size_t)gi * NP) * D + col] = o; },
            [&](int gi, float mx, float l) {   // (max, sum, call tag, 0): the tag marks it current
              reinterpret_cast<float4*>(a.part_ml)[prow + (size_t)gi * NP] =
                  make_float4(mx, l, __uint_as_float(tag), 0.f);
            });
      }
      __syncthreads();
      if (tid == 0) {
        int nl = 0;
        for (int s = 0; s < ns; ++s) {
          const int kk = rd.k0 + ka + s;
          const int u = (kk % a.batch) * a.h_kv + kk / a.batch;
          const long long u0 = (long long)(ka + s) * K, u1 = u0 + K;
          const unsigned n = (unsigned)(min(pz, u1) - max(pa, u0));
          if (atom_add_acq_rel(att_done + u, n) + n == (unsigned)K) s_last[nl++] = s;
        }
        s_nlast = nl;
      }
      __syncthreads();
      stamp(12);
      if (s_nlast > 0) stamp(13);
      // this CTA completed these units: final merges, kUP units at a time
      // (each on its own part of the block when a unit needs at most half)
      constexpr int kUP = (G * D * 2 <= kNT) ? 2 : 1;
      constexpr int kTPU = kNT / kUP, kWPU = kNW / kUP;
      for (int x0 = 0; x0 < s_nlast; x0 += kUP) {
        const int hx = tid / kTPU, ltid = tid % kTPU, lwarp = warp % kWPU;
        const int x = x0 + hx;
        const bool act = x < s_nlast;
        const int s = act ? s_last[x] : 0;
        const int kk = rd.k0 + ka + s;
        const int r = kk % a.batch, g = kk / a.batch;
        const int u = r * a.h_kv + g;
        const int nparts = NP;               // every slot; those not written this call weigh 0
        // one round trip to L2: every thread loads its columns' first kFC
        // partial outputs while warp gi loads group gi's (max, sum) pairs
        // lane-parallel and turns them into weights; after one barrier the
        // columns combine from registers (later partials, if any, from L2)
        float* wbuf = stash_o + hx * (G * NP + 2 * G);   // [G][NP] weights + [G][2] (max, sum)
        constexpr int kCPT = (G * D + kTPU - 1) / kTPU;      // columns per thread
        constexpr int kFC = kCPT >= 4 ? 4 : 16 / kCPT;      // partials prefetched per column
        float ov[kCPT][kFC];
#pragma unroll
        for (int c = 0; c < kCPT; ++c) {
          const int idx = ltid + c * kTPU;
          if (act && idx < G * D) {
            const size_t row0 = ((size_t)u * G + idx / D) * NP;
#pragma unroll
            for (int j = 0; j < kFC; ++j)
              ov[c][j] = j < nparts ? __ldcg(a.part_o + (row0 + j) * D + idx % D) : 0.f;
          }
        }
        if (act && lwarp < G) {
          const int gi = lwarp;
          const size_t row0 = ((size_t)u * G + gi) * NP;
          const float4* mlr = reinterpret_cast<const float4*>(a.part_ml) + row0;
          // a slot holds a partial of this call iff it carries the call's tag
          // (workers with no position of the unit leave theirs stale)
          constexpr int kML = 2;             // (max, sum) pairs per lane held in registers
          float2 ml[kML];
#pragma unroll
          for (int t = 0; t < kML; ++t) {
            const int j = lane + 32 * t;
            float4 v = j < nparts ? __ldcg(mlr + j) : make_float4(-INFINITY, 0.f, 0.f, 0.f);
            if (__float_as_uint(v.z) != tag) v.x = -INFINITY;
            ml[t] = make_float2(v.x, v.y);
          }
          float mx = -INFINITY;
#pragma unroll
          for (int t = 0; t < kML; ++t) mx = fmaxf(mx, ml[t].x);
          for (int j = lane + 32 * kML; j < nparts; j += 32) {      // more than 64 partials
            const float4 v = __ldcg(mlr + j);
            if (__float_as_uint(v.z) == tag) mx = fmaxf(mx, v.x);
          }
          mx = warp_max(mx);
          float l = 0.f;
#pragma unroll
          for (int t = 0; t < kML; ++t) {
            const int j = lane + 32 * t;
            float w = 0.f;
            if (mx != -INFINITY && ml[t].x != -INFINITY) {
              w = exp2f(ml[t].x - mx);
              l = fmaf(w, ml[t].y, l);
            }
            if (j < nparts) wbuf[gi * NP + j] = w;
          }
          for (int j = lane + 32 * kML; j < nparts; j += 32) {
            const float4 v = __ldcg(mlr + j);
            float w = 0.f;
            if (__float_as_uint(v.z) == tag && mx != -INFINITY && v.x != -INFINITY) {
              w = exp2f(v.x - mx);
              l = fmaf(w, v.y, l);
            }
            wbuf[gi * NP + j] = w;
          }
          l = warp_sum(l);
          if (lane == 0) {
            wbuf[G * NP + gi * 2 + 0] = mx;
            wbuf[G * NP + gi * 2 + 1] = l;
          }
        }
        __syncthreads();
#pragma unroll
        for (int c = 0; c < kCPT; ++c) {
          const int idx = ltid + c * kTPU;
          if (!act || idx >= G * D) break;
          const int gi = idx / D, col = idx % D;
          const size_t row0 = ((size_t)u * G + gi) * NP;
          const float mx = wbuf[G * NP + gi * 2 + 0], l = wbuf[G * NP + gi * 2 + 1];
          float o = 0.f;
#pragma unroll
          for (int j = 0; j < kFC; ++j)          // absent partials hold anything: weight 0 skips them
            if (j < nparts) { const float w = wbuf[gi * NP + j]; o = fmaf(w, w != 0.f ? ov[c][j] : 0.f, o); }
#pragma unroll 4
          for (int j = kFC; j < nparts; ++j) {
            const float w = wbuf[gi * NP + j];
            const float v = __ldcg(a.part_o + (row0 + j) * D + col);
            o = fmaf(w, w != 0.f ? v : 0.f, o);
          }
          const size_t orow = (size_t)r * h_q + (size_t)g * G + gi;
          a.out[orow * D + col] = l > 0.f ? o / l : 0.f;
          if (col == 0 && a.lse) a.lse[orow] = l > 0.f ? (mx + log2f(l)) * LN2 : -INFINITY;
        }
        if (act && ltid == 0) att_done[u] = 0;   // reset for the next call
        __syncthreads();
      }
      if (s_nlast > 0) stamp(14);
      __syncthreads();
      pa = pz;
      if (pa >= pe && qr == 0) stamp(5);
    }
  }
  stamp(9);
}

template <typename T, int D, int S, int G, bool F8>
bool set_attr() {
  return cudaFuncSetAttribute(step_kernel<T, D, S, G, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              StepShape<T, D, S, G>::SMEM) == cudaSuccess;
}

// Shared memory and resident CTAs per SM of one instantiation (cached per
// device; the large shared-memory opt-in is set before the query).
template <typename T, int D, int S, int G, bool F8>
void shape_of(int dev, int* smem, int* per_sm) {
  static std::atomic<int> cached[64];   // per device: 0 unknown
  *smem = StepShape<T, D, S, G>::SMEM;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_acquire);
    if (c > 0) { *per_sm = c; return; }
  }
  int n = 0;
  if (!set_attr<T, D, S, G, F8>() ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, step_kernel<T, D, S, G, F8>, kNT, *smem) !=
          cudaSuccess)
    n = 0;
  cudaGetLastError();
  if (dev >= 0 && dev < 64 && n > 0) cached[dev].store(n, std::memory_order_release);
  *per_sm = n;
}

template <typename T, int D, int S, int G, bool F8>
cudaError_t launch_t(const StepArgs& a, const StepPlan& p, cudaStream_t s) {
  using Sh = StepShape<T, D, S, G>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kNT);
  cfg.dynamicSmemBytes = Sh::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident: the waits end
  attr[0].val.cooperative = 1;
  // the launch may overlap the previous kernel's tail (the kernel waits for
  // it with griddepcontrol.wait before touching memory)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  // -1 untried, 0 refused (or QUEST_NO_PDL set in the environment), 1 accepted
  static std::atomic<int> pdl_ok{getenv("QUEST_NO_PDL") ? 0 : -1};
  cfg.numAttrs = pdl_ok.load() == 0 ? 1 : 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, step_kernel<T, D, S, G, F8>, a);
  if (e != cudaSuccess && cfg.numAttrs == 2 && pdl_ok.load() == -1) {   // not with this launch: plain
    cudaGetLastError();
    pdl_ok = 0;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, step_kernel<T, D, S, G, F8>, a);
  } else if (e == cudaSuccess) {
    if (cfg.numAttrs == 2) pdl_ok = 1;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T, int D, int S, bool F8>
cudaError_t launch_g(const StepArgs& a, const StepPlan& p, cudaStream_t s) {
  switch (a.group) {
    case 1: return launch_t<T, D, S, 1, F8>(a, p, s);
    case 2: return launch_t<T, D, S, 2, F8>(a, p, s);
    case 4: return launch_t<T, D, S, 4, F8>(a, p, s);
    case 8: return launch_t<T, D, S, 8, F8>(a, p, s);
  }
  return cudaErrorInvalidValue;
}

template <typename T, int D, bool F8>
cudaError_t launch_s(const StepArgs& a, const StepPlan& p, cudaStream_t s) {
  return a.page_size == 16 ? launch_g<T, D, 16, F8>(a, p, s) : launch_g<T, D, 32, F8>(a, p, s);
}

template <typename T, int D, int S, bool F8>
void shape_g(int dev, int group, int* smem, int* per_sm) {
  switch (group) {
    case 1: shape_of<T, D, S, 1, F8>(dev, smem, per_sm); return;
    case 2: shape_of<T, D, S, 2, F8>(dev, smem, per_sm); return;
    case 4: shape_of<T, D, S, 4, F8>(dev, smem, per_sm); return;
    case 8: shape_of<T, D, S, 8, F8>(dev, smem, per_sm); return;
  }
  *smem = 1 << 30;
  *per_sm = 0;
}
template <typename T, int D, bool F8>
void shape_s(int dev, int S, int group, int* smem, int* per_sm) {
  if (S == 16) shape_g<T, D, 16, F8>(dev, group, smem, per_sm);
  else shape_g<T, D, 32, F8>(dev, group, smem, per_sm);
}

}  // namespace
}  // namespace quest
