// Fused decode step of one layer on thread-block clusters: every (request,
// KV head) unit is scored, selected and attended inside ONE cluster of kCL
// CTAs (one per SM), so no step of the path waits on another cluster:
//   a1 append of the new token (Quest page §1.2 eq (8)) folded into the
//      scoring of its page,
//   a2 page upper bounds U_p (Quest page §1.1 eq (2)-(3); GQA group max §2.1),
//   a3 Top-K pages, ties to the lower page index (Quest page Fig. 1, §2),
//   a4 attention over the selected pages (Quest page Fig. 1, §2.1), and
//   a5 the log-sum-exp merge of the partial results (Quest page §2.1).
//
// Each cluster takes a list of units (one, or several in a snake order over
// the requests sorted by length) and works through them in the order
// S(0), S(1), A(0), S(2), A(1), ..., A(n-1): the selection of a unit runs
// while the next unit's summaries stream. Warps of a CTA have fixed roles:
//   * consumer warps feed themselves. In S(t) the unit's pages are split
//     into kCL contiguous ranges (one per CTA) and each range into NCW
//     contiguous runs (one per consumer warp); a warp copies its run's
//     summaries, CHUNK pages at a time, into its own buffer with cp.async (16
//     bytes per lane, one chunk in flight while one is scored; for the FMA
//     bound each warp copy takes 128-byte slices of four pages), bounds them
//     (sign-select and FMA for groups of 1 and 2; for groups of 4 and 8 a
//     contraction on the warp MMA over XOR-swizzled chunks), folds the new
//     token into its page's staged summary, and writes each score as an
//     order-preserving key into the row buffer of every CTA of the cluster
//     (distributed shared memory).
//     In A(t) it streams its share of the CTA's selected pages, the next
//     page's K block loading while the current V block is folded into the
//     warp's online softmax: 1-D bulk copies and FMA for groups of 1 and 2,
//     16-byte cp.async pieces into swizzled 16-token tiles and the warp MMA
//     for groups of 4 and 8; the state is stashed per unit.
//   * select warps wait until every CTA has delivered the unit's keys, run
//     the block Top-K (every CTA computes the same set), look up the
//     selected pages' physical ids, release the unit to the consumers, then
//     merge the consumers' states into the CTA's partial and send it to the
//     unit's owner CTA, which combines the kCL partials into the output row.
//     (A cluster with a single unit of groups 1 or 2 has eight consumer
//     warps run its Top-K instead: nothing else would run meanwhile.)
// Hand-offs are mbarrier phases (bulk-copy completion, local and remote
// arrivals); every wait is bounded and sets QUEST_DEVERR_WAIT_TIMEOUT rather
// than hanging, after which the CTA stops issuing and drains its copies.
// The launch needs no workspace and no grid-wide synchronisation.
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

constexpr int kCL = 4;                       // CTAs per cluster
constexpr int kCSW = 4;                      // select warps (the last ones)
constexpr int kCSelT = kCSW * 32;
constexpr int kCMaxCW = 11;                  // consumer warps at most
constexpr int kCMaxU = 64;                   // units per cluster
constexpr int kCRowCap = 8192;               // keys of a row held in shared memory
constexpr int kCKCap = 512;                  // selected pages listed in shared memory
constexpr int kCSmemMax = 227 * 1024;
constexpr int kCTrace = 16;

struct CUnit {
  int r, g, lo, P;       // request, KV head, first table entry, scored pages
  int L, nsel, app, tp;  // valid tokens, selected pages, appends (1/0), table pages
};

template <typename T, int D, int S, int G, bool F8>
struct CShape {
  static constexpr int ES = (int)sizeof(T);
  static constexpr int ESS = F8 ? 1 : ES;           // summary element bytes
  static constexpr int RB = D * ESS;                // one summary row (m or M)
  static constexpr int SUMB = 2 * RB;               // summary of one (page, head)
  static constexpr int BLK = S * D * ES;            // K (or V) block of one (page, head)
  static constexpr int HALF = BLK < 4096 ? BLK : 4096;   // a K (or V) sub-block
  static constexpr int NSB = BLK / HALF;            // sub-blocks per block
  static constexpr int TB = HALF / (D * ES);        // tokens per sub-block
  static constexpr int SLOT = 2 * HALF;             // a warp's buffer: K | V, or two chunks
  // fp16 groups of 4 or 8: QK and AV on the warp MMA, from tiles of 16 tokens
  // staged swizzled by cp.async; otherwise FMA from bulk-copied sub-blocks
  static constexpr bool MMAA = ES == 2 && G >= 4;
  using W = std::conditional_t<MMAA, WarpAttnMmaS<D, G>, WarpAttn<T, D, TB, G>>;
  static constexpr int WNV = MMAA ? 64 : WarpAttn<T, D, TB, G>::NV;   // warp scratch floats
  // scoring chunks: half of a warp's buffer (at least one round of PPR
  // pages), so that one streams while the other is scored (finer chunks,
  // more in flight, measured slower: the per-chunk reduction dominates)
  static constexpr int CHB0 = HALF, CHBR = (32 / (RB / 16 < 8 ? RB / 16 : 8)) * SUMB;
  static constexpr int CHB = CHB0 >= CHBR ? CHB0 : CHBR;   // bytes of a chunk
  static constexpr int NQ = SLOT / CHB;                    // chunks a warp's buffer holds
  static constexpr int CHUNK = CHB / SUMB < 32 ? CHB / SUMB : 32;   // pages per chunk
  static constexpr int CPI = 512 / SUMB > 0 ? 512 / SUMB : 1;        // pages per warp copy
  static constexpr int NCPY = CHUNK * SUMB / 512;   // warp copies (16 B per lane) per chunk
  static constexpr int LPP = RB / 16 < 8 ? RB / 16 : 8;   // lanes per page when scoring
  static constexpr int VPL = RB / (16 * LPP);       // 16-byte vectors of m per lane
  static constexpr int PPR = 32 / LPP;              // pages per round
  static constexpr int NR = CHUNK / PPR;            // rounds per chunk
  static constexpr int VECS = 16 / ESS;             // summary elements per vector
  static constexpr int NV = NR * G;                 // partial bounds per lane (FMA bound)
  // fp16 keys and groups of 4 or 8: the bound on the warp MMA,
  // U = [m | M] . [q- ; q+] over the 2D summary elements (k), 8 pages per
  // n-tile, the group's heads as A rows (for one or two heads the FMA bound
  // is faster: measured)
  static constexpr bool MMAS = ES == 2 && G >= 4;
  static constexpr int KT = 2 * D / 16;             // k-steps of 16 summary elements
  static constexpr int NT8 = CHUNK / 8;             // n-tiles of 8 pages per chunk
  static constexpr int LGN = WNV > CHUNK * G ? WNV : CHUNK * G;
  static_assert(CHUNK % PPR == 0 && LPP * VPL * 16 == RB && NCPY >= 1, "scoring layout");
  static_assert(CHUNK * SUMB % 512 == 0 && NQ >= 2 && 32 % CHUNK == 0, "chunks");
  // a warp copy of a chunk: 128-byte slices of four pages (8 lanes each)
  static constexpr int NPL = CHUNK / 4;              // pages per lane
  static_assert(CHUNK % 4 == 0 && SUMB % 128 == 0 && NCPY % NPL == 0, "chunk copies");
  static_assert(!MMAS || (CHUNK % 8 == 0 && G <= 8), "MMA bound: whole n-tiles, at most 8 heads");

  static constexpr int al(int x, int a) { return (x + a - 1) / a * a; }
  // consumer warps: eleven (measured best of 10-12), or eight for groups of 4 or 8 (their per-warp
  // states take the room); one stash buffer for groups of 8
  static constexpr int NCW = G >= 4 ? 8 : kCMaxCW;
  static constexpr int NSTASH = G >= 8 ? 1 : 2;
  static constexpr int NT = (NCW + kCSW) * 32;
  static constexpr int SEL0 = NCW * 32;             // first select thread
  using SelGrp = BarGrp<2, NCW * 32, kCSelT>;      // the select warps
  static constexpr int HANDS = 8;                  // consumer warps that select a lone unit
  // ... for groups of 1 and 2 only (with the larger groups' code, the hands'
  // select and its failure path measured slower on every unit, lone or not)
  static constexpr bool HANDSOK = G <= 2;
  using AllGrp = BarGrp<3, 0, HANDS * 32>;

  static constexpr int ROWS_OFF = 0;                                  // [2][kCRowCap] keys
  static constexpr int SELL_OFF = ROWS_OFF + 2 * kCRowCap * 4;       // [2][kCKCap] logical ids
  static constexpr int SELP_OFF = SELL_OFF + 2 * kCKCap * 4;         // [2][kCKCap] physical ids
  static constexpr int STO_OFF = SELP_OFF + 2 * kCKCap * 4;          // [NSTASH][NCW][G][D]
  static constexpr int STML_OFF = STO_OFF + NSTASH * NCW * G * D * 4;   // [NSTASH][NCW][G][2]
  static constexpr int PART_OFF = STML_OFF + NSTASH * NCW * G * 2 * 4;  // [kCL][G][D]
  static constexpr int PARTML_OFF = PART_OFF + kCL * G * D * 4;      // [kCL][G][2]
  static constexpr int UNITS_OFF = PARTML_OFF + kCL * G * 2 * 4;     // [kCMaxU] CUnit
  static constexpr int ORDER_OFF = UNITS_OFF + kCMaxU * (int)sizeof(CUnit);   // [64] requests
  static constexpr int LG_OFF = ORDER_OFF + 64 * 4;                  // [NCW][LGN]
  static constexpr int TOPK_OFF = al(LG_OFF + NCW * LGN * 4, 16);
  static constexpr int BAR_OFF = al(TOPK_OFF + (int)sizeof(TopkSmem<NT>), 8);
  // kv[NCW][2] (K and V halves of each consumer's buffer), row_full[2],
  // row_free[2], sel_ready[2], attn_done[2], stash_free[2], part_full, never
  static constexpr int NBAR = 2 * NCW + 12;
  static constexpr int FLAG_OFF = BAR_OFF + NBAR * 8;
  static constexpr int BUF_OFF = al(FLAG_OFF + 64, 128);              // [NCW][SLOT]
  static constexpr int SMEM = BUF_OFF + NCW * SLOT;
  static_assert(SMEM <= kCSmemMax, "shared memory");
};

// ---------------------------------------------------------------------------
// Cluster helpers (PTX).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cl_u32(uint32_t caddr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(caddr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cl_f32(uint32_t caddr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(caddr), "f"(v) : "memory");
}
// arrive on an mbarrier of CTA `rank` of the cluster, releasing this
// thread's prior writes at cluster scope
__device__ __forceinline__ void arrive_cl(const uint64_t* bar, uint32_t rank) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
               :: "r"(cl_map(smem_u32(bar), rank)) : "memory");
}
__device__ __forceinline__ void arrive_local(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool try_wait_cl(const uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(1000u) : "memory");
  return ok != 0;
}
__device__ __forceinline__ void red_cl_min(uint32_t caddr, uint32_t v) {
  asm volatile("red.shared::cluster.min.u32 [%0], %1;" :: "r"(caddr), "r"(v) : "memory");
}
__device__ __forceinline__ void red_cl_max(uint32_t caddr, uint32_t v) {
  asm volatile("red.shared::cluster.max.u32 [%0], %1;" :: "r"(caddr), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
__device__ __forceinline__ void fence_acq_rel_cluster() {
  asm volatile("fence.acq_rel.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit_grp() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_grp() {
  asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Whole-warp bounded wait for phase `parity` of a CTA-local mbarrier (its
// completion may come from TMA, local or remote arrivals). Returns false if
// the CTA is aborting or the limit runs out (then the CTA aborts and the
// error word says so). Warp-uniform.
__device__ __forceinline__ bool cwait_warp(const uint64_t* bar, uint32_t parity,
                                           volatile int* abort, unsigned* err, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    const bool ok = try_wait_cl(bar, parity);
    if (__all_sync(FULL, ok)) return true;
    if (__any_sync(FULL, *abort != 0)) return false;
  }
  if ((threadIdx.x & 31) == 0) {
    *abort = 1;
    report(err, QUEST_DEVERR_WAIT_TIMEOUT);
  }
  __syncwarp();
  return false;
}
// Single-thread form of the same wait.
__device__ __forceinline__ bool cwait_one(const uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned* err, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (try_wait_cl(bar, parity)) return true;
    if (*abort) return false;
  }
  *abort = 1;
  report(err, QUEST_DEVERR_WAIT_TIMEOUT);
  return false;
}

// Sums N per-lane values over aligned groups of 2*O lanes, halving the
// values each step (transposed butterfly); afterwards a lane holds values
// [sub_base(lane), sub_base(lane) + max(1, N / (2*O))).
template <int N, int O>
__device__ __forceinline__ void sub_reduce(float* v, int lane) {
  if constexpr (O >= 1) {
    if constexpr (N >= 2) {
      tr_step<N>(v, lane, O);
      sub_reduce<N / 2, O / 2>(v, lane);
    } else {
      v[0] += __shfl_xor_sync(FULL, v[0], O);
      sub_reduce<1, O / 2>(v, lane);
    }
  }
}
// Byte offset of byte `byte` of page row p in a chunk staged for the MMA
// bound: 16-byte units XOR-swizzled by the row (so that the eight rows of an
// n-tile, SUMB apart, fall in different banks).
template <int SUMB>
__device__ __forceinline__ int sw_off(int p, int byte) {
  return p * SUMB + ((((byte >> 4) ^ (p & 7)) << 4) | (byte & 15));
}

template <int N, int O>
__device__ __forceinline__ int sub_base(int lane) {
  if constexpr (O >= 1 && N >= 2) return ((lane & O) ? N / 2 : 0) + sub_base<N / 2, O / 2>(lane);
  else return 0;
}

// LR: rows longer than the register-resident Top-K takes (32 keys per select
// thread) may occur. Tables of at most kCShortRows entries cannot hold one,
// and their launches take the LR = false instance, which leaves the long-row
// Top-K out of the kernel (measured: llama_layer 20.23 -> 19.94 us).
constexpr int kCShortRows = 32 * kCSelT;

template <typename T, int D, int S, int G, bool F8, bool LR>
__global__ void __cluster_dims__(kCL, 1, 1) __launch_bounds__(CShape<T, D, S, G, F8>::NT, 1)
cstep_kernel(const StepArgs a) {
  static_assert(!F8 || sizeof(T) == 2, "E4M3 summaries take fp16 keys");
  using Sh = CShape<T, D, S, G, F8>;
  using W = typename Sh::W;
  using KO = KeyOps<T>;
  using SelGrp = typename Sh::SelGrp;
  constexpr int NCW = Sh::NCW, NT = Sh::NT;
  constexpr int CHUNK = Sh::CHUNK, LPP = Sh::LPP, VPL = Sh::VPL, PPR = Sh::PPR, NR = Sh::NR;
  constexpr int VECS = Sh::VECS, SLOT = Sh::SLOT, SUMB = Sh::SUMB, RB = Sh::RB, BLK = Sh::BLK;
  constexpr int NCPY = Sh::NCPY, HALF = Sh::HALF, NQ = Sh::NQ, CHB = Sh::CHB;
  extern __shared__ __align__(128) unsigned char smem[];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cl_rank();
  const int cid = (int)(blockIdx.x / kCL), ncl = (int)(gridDim.x / kCL);
  const int h_q = a.h_kv * G;
  const int K = a.k;
  const uint32_t lim = a.wait_limit;

  uint32_t* rows = reinterpret_cast<uint32_t*>(smem + Sh::ROWS_OFF);
  int32_t* sell = reinterpret_cast<int32_t*>(smem + Sh::SELL_OFF);
  int32_t* selp = reinterpret_cast<int32_t*>(smem + Sh::SELP_OFF);
  float* sto = reinterpret_cast<float*>(smem + Sh::STO_OFF);
  float* stml = reinterpret_cast<float*>(smem + Sh::STML_OFF);
  float* part = reinterpret_cast<float*>(smem + Sh::PART_OFF);
  float* partml = reinterpret_cast<float*>(smem + Sh::PARTML_OFF);
  CUnit* units = reinterpret_cast<CUnit*>(smem + Sh::UNITS_OFF);
  int32_t* order = reinterpret_cast<int32_t*>(smem + Sh::ORDER_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::BAR_OFF);
  uint64_t* kvb = bars;                        // [NCW][2] K and V halves of each consumer
  uint64_t* row_full = bars + 2 * NCW;         // [2] every CTA's keys of the unit delivered
  uint64_t* row_free = row_full + 2;           // [2] every CTA done reading the row
  uint64_t* sel_ready = row_full + 4;          // [2] this CTA's selection published
  uint64_t* attn_done = row_full + 6;          // [2] consumer states of the unit stashed
  uint64_t* stash_free = row_full + 8;         // [2] stash merged
  uint64_t* part_full = row_full + 10;         // partials of an owned unit delivered
  uint64_t* never = row_full + 11;             // nothing arrives (the failure-handling test)
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + Sh::FLAG_OFF);
  volatile int* s_n = s_abort + 1;             // units of this cluster
  volatile int* s_ok = s_abort + 2;            // select group's wait result
  volatile int* s_ok_all = s_abort + 3;        // the all-warp group's wait result
  uint32_t* kmm = reinterpret_cast<uint32_t*>(smem + Sh::FLAG_OFF) + 4;   // [2][2] key min, max
  unsigned char* bufs = smem + Sh::BUF_OFF;

  unsigned long long* trace = a.trace ? a.trace + (size_t)blockIdx.x * kCTrace : nullptr;
  auto stamp = [&](int i) { if (trace) trace[i] = global_ns(); };
  if (tid == 0) stamp(0);

  if (tid == 0) {
    for (int w = 0; w < NCW; ++w) { mbar_init(kvb + 2 * w, 1); mbar_init(kvb + 2 * w + 1, 1); }
    for (int b = 0; b < 2; ++b) {
      mbar_init(row_full + b, kCL * NCW);
      mbar_init(row_free + b, kCL);
      mbar_init(sel_ready + b, 1);
      mbar_init(attn_done + b, NCW);
      mbar_init(stash_free + b, 1);
    }
    mbar_init(part_full, kCL);
    mbar_init(never, 1);
    *s_abort = 0;
    for (int b = 0; b < 2; ++b) { kmm[2 * b] = 0xffffffffu; kmm[2 * b + 1] = 0u; }
    fence_mbar_init();
  }
  // the next kernel on the stream may be scheduled now; this grid waits for
  // the previous one (and its writes) before touching global memory
  pdl_launch_dependents();
  cluster_sync_all();                          // barriers of every CTA initialised
  pdl_wait();
  if (tid == 0) stamp(1);

  // ---------------------- unit list (first select warp) ----------------------
  if (warp == NCW) {
    const int B = a.batch, H = a.h_kv, U = B * H;
    // requests by decreasing length (ties to the lower index), for B <= 64;
    // longer batches keep their order
    const bool sorted = U > ncl && B <= 64;
    if (sorted) {
      int Pl[2];
      for (int h = 0; h < 2; ++h) {
        const int r = lane + 32 * h;
        Pl[h] = r < B ? (__ldg(a.seq_lens + r) + S - 1) / S : -1;
      }
      for (int h = 0; h < 2; ++h) {
        const int r = lane + 32 * h;
        int rk = 0;
        for (int x = 0; x < B; ++x) {
          const int px = __shfl_sync(FULL, Pl[x >> 5], x & 31);
          rk += (px > Pl[h]) || (px == Pl[h] && x < r);
        }
        if (r < B) order[rk] = r;
      }
      __syncwarp();
    }
    // snake over the clusters: pass p gives cluster c the unit p*ncl + c
    // (even p) or p*ncl + ncl-1-c (odd p)
    int n = 0;
    if (U <= ncl) {
      n = cid < U ? 1 : 0;
    } else {
      for (int p = 0; p * ncl < U; ++p)
        if (p * ncl + ((p & 1) ? ncl - 1 - cid : cid) < U) ++n;
    }
    if (n > kCMaxU) {                        // the host keeps units per cluster within the cap
      n = kCMaxU;
      if (lane == 0) report(a.err, QUEST_DEVERR_TABLE_RANGE);
    }
    for (int i = lane; i < n; i += 32) {
      int k = cid;
      if (U > ncl) {                         // the i-th unit of this cluster in pass order
        int cnt = -1;
        for (int p = 0; p * ncl < U; ++p) {
          const int kk = p * ncl + ((p & 1) ? ncl - 1 - cid : cid);
          if (kk < U && ++cnt == i) { k = kk; break; }
        }
      }
      const int r = sorted ? order[k / H] : k / H, g = k % H;
      CUnit un;
      un.r = r; un.g = g;
      un.lo = __ldg(a.page_indptr + r);
      un.tp = __ldg(a.page_indptr + r + 1) - un.lo;
      un.L = __ldg(a.seq_lens + r);
      int P = (un.L + S - 1) / S;
      un.app = (a.k_new != nullptr && P >= 1 && P <= un.tp) ? 1 : 0;
      if (P > un.tp) {
        report(a.err, QUEST_DEVERR_TABLE_RANGE);
        P = un.tp;
      }
      un.P = P;
      un.nsel = P < K ? P : K;
      units[i] = un;
    }
    if (lane == 0) *s_n = n;
    __syncwarp();
  }
  // one request: the consumers' first page-table windows and scoring
  // query, fetched before the list. They wait in the second chunk slot of the
  // warp's buffer (untouched until the first unit's chunk loop), not in
  // registers, which would stay allocated across the whole unit loop.
  constexpr int QLD = Sh::MMAS ? 1 : Sh::VPL * (F8 ? 2 : 1);   // 16-byte query vectors per lane, head
  constexpr int QL8 = Sh::MMAS ? D / 16 : 1;                   // 8-byte pieces (MMA layout)
  constexpr int QB0 = Sh::MMAS ? QL8 * 8 : G * QLD * 16;       // query bytes per lane
  constexpr bool EARLYQ = 32 * (QB0 + 16) <= CHB;               // (not for fp32 head dim 128)
  constexpr int QB = EARLYQ ? QB0 : 0;
  static_assert(32 * (QB + 16) <= CHB && QB % 16 == 0, "early values fit the second chunk slot");
  const bool pre = a.batch == 1 && warp < NCW && cid < a.h_kv;
  if (pre) {
    int pw[4] = {-1, -1, -1, -1};
    uint4 qpre[Sh::MMAS ? 1 : G][QLD];
    uint2 qpre8[QL8];
    unsigned char* early = smem + Sh::BUF_OFF + (size_t)warp * SLOT + CHB;
    if constexpr (!EARLYQ) {
    } else if constexpr (Sh::MMAS) {                // head gid's dims 16j + 4t .. + 3
      const int gid = lane >> 2, tq = lane & 3;
      const T* qh = static_cast<const T*>(a.q) + ((size_t)cid * G + (gid < G ? gid : 0)) * D;
#pragma unroll
      for (int j = 0; j < QL8; ++j) qpre8[j] = *reinterpret_cast<const uint2*>(qh + 16 * j + 4 * tq);
    } else {
      const int sub0 = lane % Sh::LPP;
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        const T* qp = static_cast<const T*>(a.q) + ((size_t)cid * G + gi) * D;
#pragma unroll
        for (int v = 0; v < Sh::VPL; ++v)
#pragma unroll
          for (int h = 0; h < (F8 ? 2 : 1); ++h)
            qpre[gi][v * (F8 ? 2 : 1) + h] = ld_nc_v4(qp + (v * Sh::LPP + sub0) * Sh::VECS + h * 8);
      }
    }
    const int span = a.nnz, nch = (span + CHUNK - 1) / CHUNK;
    const int cc0 = (int)((long long)nch * (int)rank / kCL);
    const int ncc = (int)((long long)nch * ((int)rank + 1) / kCL) - cc0;
    const int pb = (cc0 + ncc * warp / NCW) * CHUNK;
    const int pe = min(span, (cc0 + ncc * (warp + 1) / NCW) * CHUNK);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int p = pb + 32 * k + lane;
      pw[k] = p < pe ? __ldg(a.page_indices + p) : -1;
    }
    // ... and the first NQ - 1 chunks of the warp's run start streaming
    // (unit = cluster: KV head cid of the request)
    const int nm0 = (cc0 + ncc * (warp + 1) / NCW) - (cc0 + ncc * warp / NCW);
    unsigned char* buf0 = smem + Sh::BUF_OFF + (size_t)warp * SLOT;
#pragma unroll
    for (int m = 0; m < NQ - 1; ++m) {
      if (m < nm0) {
        const int o = m * CHUNK;
        const int srcw = ((o >> 5) & 1) ? pw[1] : pw[0];
        if constexpr (Sh::MMAS) {                  // copy k: bytes [512k, 512k + 512)
          const int ph = __shfl_sync(FULL, srcw, (o & 31) + (lane & (CHUNK - 1)));
#pragma unroll
          for (int k = 0; k < NCPY; ++k) {
            const int byte = k * 512 + lane * 16;
            const int phj = __shfl_sync(FULL, ph, byte / SUMB);
            if (phj >= 0 && phj < a.n_phys)
              cp_async16(buf0 + m * CHB + sw_off<SUMB>(byte / SUMB, byte % SUMB),
                         static_cast<const unsigned char*>(a.summary) +
                             ((size_t)phj * a.h_kv + cid) * SUMB + byte % SUMB);
          }
        } else {                                   // copy k: slices of four pages
          // page j of the chunk: table entry o + j, in lane (o & 31) + j of the window
          constexpr int NPL = Sh::NPL;
          int phs[NPL];
#pragma unroll
          for (int i = 0; i < NPL; ++i) phs[i] = __shfl_sync(FULL, srcw, (o & 31) + (lane >> 3) + 4 * i);
#pragma unroll
          for (int k = 0; k < NCPY; ++k) {
            const int i = k % NPL, j = (lane >> 3) + 4 * i;        // page j of the chunk
            const int byte = (k / NPL) * 128 + (lane & 7) * 16;   // its 16-byte piece
            if (phs[i] >= 0 && phs[i] < a.n_phys)
              cp_async16(buf0 + m * CHB + j * SUMB + byte, static_cast<const unsigned char*>(a.summary) +
                                                                ((size_t)phs[i] * a.h_kv + cid) * SUMB + byte);
          }
        }
      }
      cp_async_commit_grp();
    }
    if constexpr (!EARLYQ) {
    } else if constexpr (Sh::MMAS) {
#pragma unroll
      for (int j = 0; j < QL8; ++j) *reinterpret_cast<uint2*>(early + lane * QB + 8 * j) = qpre8[j];
    } else {
#pragma unroll
      for (int gi = 0; gi < G; ++gi)
#pragma unroll
        for (int j = 0; j < QLD; ++j)
          *reinterpret_cast<uint4*>(early + lane * QB + 16 * (gi * QLD + j)) = qpre[gi][j];
    }
    *reinterpret_cast<int4*>(early + 32 * QB + lane * 16) = make_int4(pw[0], pw[1], pw[2], pw[3]);
  }
  {   // the Top-K's histogram starts at zero (each Top-K leaves it so):
      // zeroed before the barrier, which orders it before any select,
      // including a lone unit's select by the consumer warps
    TopkSmem<NT>& tsm = *reinterpret_cast<TopkSmem<NT>*>(smem + Sh::TOPK_OFF);
    for (int i = tid; i < kTopkBins; i += NT) tsm.hist[i] = 0;
  }
  asm volatile("bar.sync 1, %0;" :: "n"(NT) : "memory");
  const int n = *s_n;


  // this CTA's chunks of the unit's pages (CTA r takes chunks
  // [nch r / kCL, nch (r+1) / kCL)) and its share of the selection (winner
  // w belongs to CTA w % kCL)
  // (one request: over its table pages, known before any load, so that the
  // consumers can fetch their page-table windows while the unit list forms)
  auto c_lo = [&](const CUnit& un, int r) {
    const int span = a.batch == 1 ? un.tp : un.P;
    return (int)((long long)((span + CHUNK - 1) / CHUNK) * r / kCL);
  };
  auto n_at = [&](const CUnit& un) {
    return un.nsel > (int)rank ? (un.nsel - (int)rank + kCL - 1) / kCL : 0;
  };

  // A cluster with a single unit has nothing to stream while it selects:
  // then the first HANDS consumer warps run the select (AllGrp; more
  // threads would only add barrier latency) and publish it through
  // sel_ready, else the select warps do (SelGrp) while the consumers stream
  // the next unit.
  const bool all_hands = Sh::HANDSOK && n == 1;

  // T(u) on thread group Grp: wait for every CTA's keys of unit u, Top-K,
  // the selected pages' physical ids. Returns false if the CTA aborts.
  auto select_core = [&](auto grp, int u) -> bool {
    using Grp = decltype(grp);
    constexpr int NTH = Grp::kN;
    const int gt = Grp::tid(), gw = gt >> 5;
    TopkSmem<NTH>& tsm = *reinterpret_cast<TopkSmem<NTH>*>(smem + Sh::TOPK_OFF);
    volatile int* okf = NTH == kCSelT ? s_ok : s_ok_all;
    const int b = u & 1;
    const CUnit un = units[u];
    if (gt == 0) *okf = cwait_one(row_full + b, (u >> 1) & 1, s_abort, a.err, lim) ? 1 : 0;
    Grp::sync();
    if (!*okf) return false;
    if (u == 0 && gt == 0) stamp(5);
    const int P = un.P, nsel = un.nsel;
    const bool listed = nsel <= kCKCap;
    int32_t* ol = a.sel_logical + ((size_t)un.r * a.h_kv + un.g) * K;
    int32_t* sl = sell + b * kCKCap;
    int32_t* sp = selp + b * kCKCap;
    const int f_lo = min(a.n_sink, P), f_hi = max(f_lo, P - a.n_local);
    auto forced = [f_lo, f_hi](int i) { return i < f_lo || i >= f_hi; };
    auto emit = [&](int pos, int i) {   // (the owner writes the outputs afterwards)
      if (listed) sl[pos] = i;
      else ol[pos] = i;
    };
    uint32_t* keys = rows + b * kCRowCap;
    if (P <= kCRowCap && P <= 32 * NTH) {
      // min and max of the competing keys, folded in by the consumers
      const uint32_t kmin = kmm[2 * b], kmax = kmm[2 * b + 1];
      (void)gw;
      block_topk_smem<NTH, decltype(emit), decltype(forced), Grp, NoEarly,
                      LR ? 32 * NTH : (kCShortRows < 32 * NTH ? kCShortRows : 32 * NTH)>(
          P, K, keys, kmin, kmax, tsm, emit, forced, f_lo + (P - f_hi));
    } else if constexpr (LR) {
      if (P <= kCRowCap) {
        auto key_at = [keys, forced](int i) { return forced(i) ? 0xffffffffu : keys[i]; };
        block_topk_keys<NTH, decltype(key_at), decltype(emit), Grp>(P, K, key_at, tsm, emit);
      } else {                                    // keys of long rows from the scores in L2
        const float* sc = a.scores + (size_t)un.g * a.nnz + un.lo;
        auto key_at = [sc, forced](int i) { return forced(i) ? 0xffffffffu : score_key(__ldcg(sc + i)); };
        block_topk_keys<NTH, decltype(key_at), decltype(emit), Grp>(P, K, key_at, tsm, emit);
      }
    } else if (gt == 0) {                         // (a table of at most kCShortRows entries)
      report(a.err, QUEST_DEVERR_TABLE_RANGE);
    }
    Grp::sync();
    if (u == 0 && gt == 0) stamp(10);
    if (listed && P > K) {                        // physical pages of the listed selection
      for (int pos = gt; pos < nsel; pos += NTH) {
        const int lp = sl[pos];
        sp[pos] = (lp >= 0 && lp < P) ? __ldg(a.page_indices + un.lo + lp) : -1;
      }
      Grp::sync();
    }
    if (u == 0 && gt == 0) stamp(11);
    return true;
  };

  if (warp < NCW) {
    // ================================ consumers ================================
    // Warp cw takes the CTA's chunks and pages cw, cw + NCW, ...: it loads
    // them itself into its own buffer (two chunks in flight, or the K and V
    // halves of a page) and folds them in.
    const int cw = warp;
    float* lg = reinterpret_cast<float*>(smem + Sh::LG_OFF) + cw * Sh::LGN;
    unsigned char* buf = bufs + (size_t)cw * SLOT;
    uint64_t* kbar = kvb + 2 * cw;
    uint64_t* vbar = kbar + 1;
    uint32_t kph = 0, vph = 0;               // completed phases of kbar, vbar
    bool kpend = false, vpend = false;       // a copy issued and not yet waited for
    const uint64_t pol = evict_first_policy();
    const int pg = lane / LPP, sub = lane % LPP;
    bool dead = false;
    bool joined = false;                     // took part in the all-hands select
    for (int t = 0; t <= n && !dead; ++t) {
      if (t < n) {
        // ------------------------------ S(t) ------------------------------
        if (a.test_fault == 1 && t == 0 && rank == 0 && cw == 0 &&
            !cwait_warp(never, 0, s_abort, a.err, lim)) {   // runs out: the test's failure
          dead = true;
          break;
        }
        const CUnit un = units[t];
        const int b = t & 1;
        // my chunks: a contiguous run [mc0, mc0 + nm) of the CTA's chunks
        const int cc0 = c_lo(un, (int)rank), ncc = c_lo(un, (int)rank + 1) - cc0;
        const int mc0 = cc0 + ncc * cw / NCW;
        const int nm = cc0 + ncc * (cw + 1) / NCW - mc0;
        const bool cached = !LR || un.P <= kCRowCap;   // (short tables: always)
        const int f_lo = min(a.n_sink, un.P), f_hi = max(f_lo, un.P - a.n_local);
        uint32_t kmn = 0xffffffffu, kmx = 0u;        // over my competing pages' keys
        // the physical pages of my run, 64 table entries per window (two per
        // lane): the current window and the next one are held in registers
        const int pb = mc0 * CHUNK, pe = min(un.P, (mc0 + nm) * CHUNK);
        const int32_t* idx = a.page_indices + un.lo;
        auto ldwin = [&](int k, int& w0, int& w1) {
          const int p = pb + 64 * k + lane;
          w0 = p < pe ? __ldg(idx + p) : -1;
          w1 = p + 32 < pe ? __ldg(idx + p + 32) : -1;
        };
        int cw0, cw1, nw0, nw1, kcur = 0;
        const unsigned char* early = buf + CHB;         // the values fetched before the list
        if (t == 0 && pre && un.lo == 0 && un.tp == a.nnz) {
          const int4 p4 = *reinterpret_cast<const int4*>(early + 32 * QB + lane * 16);
          cw0 = p4.x; cw1 = p4.y; nw0 = p4.z; nw1 = p4.w;
        } else {
          ldwin(0, cw0, cw1);
          ldwin(1, nw0, nw1);
        }
        // lane j < CHUNK: physical page of page j of my chunk m (a chunk lies
        // in one half of one window), -1 past the row
        auto tbl = [&](int m) -> int {
          if (m >= nm) return -1;
          const int o = m * CHUNK, k = o >> 6, h = (o >> 5) & 1;
          const int src = k == kcur ? (h ? cw1 : cw0) : (h ? nw1 : nw0);
          const int v = __shfl_sync(FULL, src, (o & 31) + (lane & (CHUNK - 1)));
          return lane < CHUNK ? v : -1;
        };
        // 16 bytes per lane per copy. MMA bound: copy k holds bytes [512k,
        // 512k + 512) of the chunk, swizzled. FMA bound: copy k holds a
        // 128-byte slice of four pages (lanes 8q .. 8q + 7: page q + 4 (k %
        // NPL)), so a lane fetches the physical ids of its NPL pages only.
        auto issue = [&](int m, int ph) {
          if (m < nm) {
            unsigned char* dst = buf + (m % NQ) * CHB;
            if constexpr (Sh::MMAS) {
#pragma unroll
              for (int k = 0; k < NCPY; ++k) {
                const int byte = k * 512 + lane * 16;
                const int j = byte / SUMB;
                const int phj = __shfl_sync(FULL, ph, j);
                if (phj >= 0 && phj < a.n_phys)
                  cp_async16(dst + sw_off<SUMB>(j, byte % SUMB), static_cast<const unsigned char*>(a.summary) +
                                                                    ((size_t)phj * a.h_kv + un.g) * SUMB + byte % SUMB);
              }
            } else {
              constexpr int NPL = Sh::NPL;
              int phs[NPL];
#pragma unroll
              for (int i = 0; i < NPL; ++i) phs[i] = __shfl_sync(FULL, ph, (lane >> 3) + 4 * i);
#pragma unroll
              for (int k = 0; k < NCPY; ++k) {
                const int i = k % NPL, j = (lane >> 3) + 4 * i;    // page j of the chunk
                const int byte = (k / NPL) * 128 + (lane & 7) * 16;   // its 16-byte piece
                if (phs[i] >= 0 && phs[i] < a.n_phys)
                  cp_async16(dst + j * SUMB + byte, static_cast<const unsigned char*>(a.summary) +
                                                        ((size_t)phs[i] * a.h_kv + un.g) * SUMB + byte);
              }
            }
          }
          cp_async_commit_grp();
        };
        // the first NQ - 1 chunks (one request: issued before the unit list)
        const bool preissued = t == 0 && pre && un.lo == 0 && un.tp == a.nnz;
        if (!preissued) {
          cp_async_wait_grp<0>();            // (none pending but a stale early issue)
#pragma unroll
          for (int m = 0; m < NQ - 1; ++m) issue(m, tbl(m));
        }
        // query of the unit for the bound. FMA bound: per 32-bit word a select
        // mask (take M where q >= 0) and the values as fp32. MMA bound: A
        // fragments of [q- ; q+] (k-step kk < D/16: q- against m, else q+
        // against M), head gid's elements 16 kk + 4t .. + 3 of the k order
        // that the staged summaries are read in.
        constexpr int QW = Sh::MMAS ? 1 : VPL * (F8 ? 8 : 4);
        // E4M3 summaries: the queries stay packed fp16 pairs for the
        // mixed-precision FMA (measured faster there; with fp16 summaries the
        // converted fp32 queries measured faster)
        constexpr bool QH = F8 && !Sh::MMAS;
        constexpr int QV = (Sh::MMAS || QH) ? 1 : (Sh::ES == 2 ? QW * 2 : QW);
        uint32_t qmask[G][QW];
        uint32_t qh[G][QH ? QW : 1];
        float qf[G][QV];
        constexpr int KQ = Sh::MMAS ? Sh::KT : 1;
        uint32_t qa[KQ], qb[KQ];
        if constexpr (Sh::MMAS) {
          const int gid = lane >> 2, tq = lane & 3;
          const bool hv = gid < G;
          const T* qh = static_cast<const T*>(a.q) + ((size_t)un.r * h_q + (size_t)un.g * G + (hv ? gid : 0)) * D;
          const __half2 z2 = __float2half2_rn(0.f);
#pragma unroll
          for (int j = 0; j < D / 16; ++j) {
            uint2 w = (EARLYQ && t == 0 && pre && un.g == cid) ? *reinterpret_cast<const uint2*>(early + lane * QB + 8 * j)
                                                       : *reinterpret_cast<const uint2*>(qh + 16 * j + 4 * tq);
            if (!hv) w = make_uint2(0u, 0u);
            const __half2 x = *reinterpret_cast<const __half2*>(&w.x), y = *reinterpret_cast<const __half2*>(&w.y);
            const __half2 xn = __hmin2(x, z2), yn = __hmin2(y, z2), xp = __hmax2(x, z2), yp = __hmax2(y, z2);
            qa[j] = *reinterpret_cast<const uint32_t*>(&xn);
            qb[j] = *reinterpret_cast<const uint32_t*>(&yn);
            qa[j + D / 16] = *reinterpret_cast<const uint32_t*>(&xp);
            qb[j + D / 16] = *reinterpret_cast<const uint32_t*>(&yp);
          }
        } else {
#pragma unroll
          for (int gi = 0; gi < G; ++gi) {
            const T* qp = static_cast<const T*>(a.q) + ((size_t)un.r * h_q + (size_t)un.g * G + gi) * D;
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
              const int d0 = (v * LPP + sub) * VECS;
#pragma unroll
              for (int h = 0; h < (F8 ? 2 : 1); ++h) {
                const uint4 qv = (EARLYQ && t == 0 && pre && un.g == cid)
                                     ? *reinterpret_cast<const uint4*>(early + lane * QB +
                                                                       16 * (gi * QLD + v * (F8 ? 2 : 1) + h))
                                                                 : ld_nc_v4(qp + d0 + h * 8);
                const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const int wi = (v * (F8 ? 2 : 1) + h) * 4 + j;
                  if constexpr (QH) {
                    qmask[gi][wi] = ((~w4[j] & 0x80008000u) >> 15) * 0xffffu;
                    qh[gi][wi] = w4[j];
                  } else if constexpr (Sh::ES == 2) {
                    qmask[gi][wi] = ((~w4[j] & 0x80008000u) >> 15) * 0xffffu;
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[j]));
                    qf[gi][wi * 2] = f.x;
                    qf[gi][wi * 2 + 1] = f.y;
                  } else {
                    qmask[gi][wi] = (w4[j] & 0x80000000u) ? 0u : 0xffffffffu;
                    qf[gi][wi] = __uint_as_float(w4[j]);
                  }
                }
              }
            }
          }
        }
        // the appended token: its key dims of this lane, if this warp scores
        // the tail page
        const int ct = (un.P - 1) / CHUNK;                  // chunk of the tail page
        const int pin = (un.P - 1) - ct * CHUNK;
        const int m_tail = ct - mc0;
        const bool tail_warp = un.app && m_tail >= 0 && m_tail < nm;
        // lane l < D/4 takes dims 4l .. 4l + 3 of the new token's key and value
        // (fetched now, used when the tail page's chunk is scored)
        constexpr int NB4 = 4 * Sh::ES;                     // bytes of 4 dims
        uint4 kq = make_uint4(0u, 0u, 0u, 0u), vq = make_uint4(0u, 0u, 0u, 0u);
        if (tail_warp && lane < D / 4) {
          const unsigned char* kp = static_cast<const unsigned char*>(a.k_new) +
                                    ((size_t)un.r * a.h_kv + un.g) * D * Sh::ES + (size_t)lane * NB4;
          const unsigned char* vp = static_cast<const unsigned char*>(a.v_new) +
                                    ((size_t)un.r * a.h_kv + un.g) * D * Sh::ES + (size_t)lane * NB4;
          if constexpr (NB4 == 16) {
            kq = ld_nc_v4(kp);
            vq = ld_nc_v4(vp);
          } else {
            const uint2 k2 = *reinterpret_cast<const uint2*>(kp), v2 = *reinterpret_cast<const uint2*>(vp);
            kq = make_uint4(k2.x, k2.y, 0u, 0u);
            vq = make_uint4(v2.x, v2.y, 0u, 0u);
          }
        }
        // append (eq (8)): the new token's K/V into the pool, and the staged
        // summary of its page (row pin of the chunk at sbw) folded with the
        // key (a fresh page starts from it), written back to the cache too
        auto tail_patch = [&](unsigned char* sbw) {
          const int slot = (un.L - 1) % S;
          const int pp = __ldg(a.page_indices + un.lo + un.P - 1);
          if (pp >= 0 && pp < a.n_phys && lane < D / 4) {
            const size_t row = ((size_t)pp * a.h_kv + un.g) * S + slot;
            unsigned char* kd = static_cast<unsigned char*>(a.k_pool) + row * D * Sh::ES + (size_t)lane * NB4;
            unsigned char* vd = static_cast<unsigned char*>(a.v_pool) + row * D * Sh::ES + (size_t)lane * NB4;
            unsigned char* gs = static_cast<unsigned char*>(a.summary) + ((size_t)pp * a.h_kv + un.g) * SUMB;
            auto at = [&](int byte) { return sbw + (Sh::MMAS ? sw_off<SUMB>(pin, byte) : pin * SUMB + byte); };
            if constexpr (NB4 == 16) {                     // fp32: 4 keys per lane
              st_v4(kd, kq);
              st_v4(vd, vq);
              const int bm = 16 * lane, bM = RB + 16 * lane;
              uint4* sm_m = reinterpret_cast<uint4*>(at(bm));
              uint4* sm_M = reinterpret_cast<uint4*>(at(bM));
              const uint32_t kw[4] = {kq.x, kq.y, kq.z, kq.w};
              const uint4 om = *sm_m, oM = *sm_M;
              const uint32_t omw[4] = {om.x, om.y, om.z, om.w}, oMw[4] = {oM.x, oM.y, oM.z, oM.w};
              uint32_t nmw[4], nMw[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint32_t kk = KO::to_key(kw[j]);
                nmw[j] = KO::from_key(slot != 0 ? KO::kmin(KO::to_key(omw[j]), kk) : kk);
                nMw[j] = KO::from_key(slot != 0 ? KO::kmax(KO::to_key(oMw[j]), kk) : kk);
              }
              const uint4 nm4 = make_uint4(nmw[0], nmw[1], nmw[2], nmw[3]);
              const uint4 nM4 = make_uint4(nMw[0], nMw[1], nMw[2], nMw[3]);
              *sm_m = nm4;
              *sm_M = nM4;
              st_v4(gs + bm, nm4);
              st_v4(gs + bM, nM4);
            } else {
              *reinterpret_cast<uint2*>(kd) = make_uint2(kq.x, kq.y);
              *reinterpret_cast<uint2*>(vd) = make_uint2(vq.x, vq.y);
              if constexpr (F8) {
                const int bm = 4 * lane, bM = D + 4 * lane;   // code bytes of m, M
                uint32_t* sm_m = reinterpret_cast<uint32_t*>(at(bm));
                uint32_t* sm_M = reinterpret_cast<uint32_t*>(at(bM));
                uint32_t m01 = KO::to_key(kq.x), m23 = KO::to_key(kq.y);
                uint32_t M01 = m01, M23 = m23;
                if (slot != 0) {
                  m01 = KO::kmin(KO::to_key(e4m3x4_lo_h2(*sm_m)), m01);
                  m23 = KO::kmin(KO::to_key(e4m3x4_hi_h2(*sm_m)), m23);
                  M01 = KO::kmax(KO::to_key(e4m3x4_lo_h2(*sm_M)), M01);
                  M23 = KO::kmax(KO::to_key(e4m3x4_hi_h2(*sm_M)), M23);
                }
                bool ovf = false;
                const uint32_t cm = e4m3x4_floor_h(KO::from_key(m01), KO::from_key(m23), ovf);
                const uint32_t cM = e4m3x4_ceil_h(KO::from_key(M01), KO::from_key(M23), ovf);
                *sm_m = cm;
                *sm_M = cM;
                *reinterpret_cast<uint32_t*>(gs + bm) = cm;
                *reinterpret_cast<uint32_t*>(gs + bM) = cM;
                if (ovf) report(a.err, QUEST_DEVERR_FP8_RANGE);
              } else {
                const int bm = 8 * lane, bM = RB + 8 * lane;   // bytes of m, M dims
                uint2* sm_m = reinterpret_cast<uint2*>(at(bm));
                uint2* sm_M = reinterpret_cast<uint2*>(at(bM));
                uint2 mn = make_uint2(KO::to_key(kq.x), KO::to_key(kq.y)), mx = mn;
                if (slot != 0) {
                  const uint2 om = *sm_m, oM = *sm_M;
                  mn = make_uint2(KO::kmin(KO::to_key(om.x), mn.x), KO::kmin(KO::to_key(om.y), mn.y));
                  mx = make_uint2(KO::kmax(KO::to_key(oM.x), mx.x), KO::kmax(KO::to_key(oM.y), mx.y));
                }
                const uint2 nm2 = make_uint2(KO::from_key(mn.x), KO::from_key(mn.y));
                const uint2 nM2 = make_uint2(KO::from_key(mx.x), KO::from_key(mx.y));
                *sm_m = nm2;
                *sm_M = nM2;
                *reinterpret_cast<uint2*>(gs + bm) = nm2;
                *reinterpret_cast<uint2*>(gs + bM) = nM2;
              }
            }
          }
          __syncwarp();
        };
        __syncwarp();                        // every lane's early values read: slot 1 may refill
        // keys of unit t go to row buffer b of every CTA: it must be free
        if (t >= 2 && !cwait_warp(row_free + b, ((t >> 1) - 1) & 1, s_abort, a.err, lim)) {
          dead = true;
          break;
        }
        for (int m = 0; m < nm; ++m) {
          if (((m + NQ - 1) * CHUNK) >> 6 > kcur + 1) {   // past the next window
            ++kcur;
            cw0 = nw0; cw1 = nw1;
            ldwin(kcur + 1, nw0, nw1);
          }
          issue(m + NQ - 1, tbl(m + NQ - 1));   // streams while chunk m is scored
          const int phm = tbl(m);
          cp_async_wait_grp<NQ - 1>();
          __syncwarp();
          const int p0 = (mc0 + m) * CHUNK;
          const int np = min(CHUNK, un.P - p0);
          const unsigned bad = __ballot_sync(FULL, lane < np && !(phm >= 0 && phm < a.n_phys));
          if (bad && lane == 0) report(a.err, QUEST_DEVERR_PAGE_RANGE);
          const unsigned char* sb = buf + (m % NQ) * CHB;
          if (tail_warp && m == m_tail) tail_patch(buf + (m % NQ) * CHB);
          if constexpr (Sh::MMAS) {
            // U for the chunk's pages, n-tile by n-tile: C[head][page] over
            // the 2D summary elements, then the max over the group's heads
            const int gid = lane >> 2, tq = lane & 3;
#pragma unroll
            for (int nt = 0; nt < Sh::NT8; ++nt) {
              const int pr = nt * 8 + gid;                   // this lane's page of the tile
              float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int kk = 0; kk < Sh::KT; ++kk) {
                uint32_t b0, b1;
                if constexpr (F8) {                          // 4 codes, decoded to fp16 pairs
                  const uint32_t c = *reinterpret_cast<const uint32_t*>(sb + sw_off<SUMB>(pr, 16 * kk + 4 * tq));
                  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(b0) : "h"((uint16_t)c));
                  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(b1) : "h"((uint16_t)(c >> 16)));
                } else {
                  const uint2 c = *reinterpret_cast<const uint2*>(sb + sw_off<SUMB>(pr, 32 * kk + 8 * tq));
                  b0 = c.x;
                  b1 = c.y;
                }
                if (kk & 1) mma_f16_16816(c1, qa[kk], 0u, qb[kk], 0u, b0, b1);
                else mma_f16_16816(c0, qa[kk], 0u, qb[kk], 0u, b0, b1);
              }
              // rows gid < G are the heads (the rest of the 16 rows are zero)
              float v0 = gid < G ? c0[0] + c1[0] : -INFINITY;
              float v1 = gid < G ? c0[1] + c1[1] : -INFINITY;
#pragma unroll
              for (int o = 4; o < 32; o <<= 1) {
                v0 = fmaxf(v0, __shfl_xor_sync(FULL, v0, o));
                v1 = fmaxf(v1, __shfl_xor_sync(FULL, v1, o));
              }
              if (gid == 0) {
                lg[nt * 8 + 2 * tq] = v0;
                lg[nt * 8 + 2 * tq + 1] = v1;
              }
            }
          } else {
            float vals[Sh::NV];
#pragma unroll
            for (int ro = 0; ro < NR; ++ro) {
              const int p = ro * PPR + pg;
              uint4 vm[VPL], vM[VPL];
#pragma unroll
              for (int v = 0; v < VPL; ++v) {
                vm[v] = *reinterpret_cast<const uint4*>(sb + p * SUMB + (v * LPP + sub) * 16);
                vM[v] = *reinterpret_cast<const uint4*>(sb + p * SUMB + RB + (v * LPP + sub) * 16);
              }
              // sum_j max(q_j m_j, q_j M_j) = sum_j q_j * (q_j >= 0 ? M_j : m_j)
#pragma unroll
              for (int gi = 0; gi < G; ++gi) {
                float sg = 0.f;
#pragma unroll
                for (int v = 0; v < VPL; ++v) {
                  const uint32_t mw[4] = {vm[v].x, vm[v].y, vm[v].z, vm[v].w};
                  const uint32_t Mw[4] = {vM[v].x, vM[v].y, vM[v].z, vM[v].w};
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    if constexpr (F8) {              // codes decoded to fp16 pairs (exact)
                      const int wi = v * 8 + 2 * j;
                      const uint32_t sel = e4m3_qsel_from_masks(qmask[gi][wi], qmask[gi][wi + 1]);
                      const uint32_t xw = (Mw[j] & sel) | (mw[j] & ~sel);
                      uint32_t lo, hi;
                      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"((uint16_t)xw));
                      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"((uint16_t)(xw >> 16)));
                      sg = fma2_h_f32(qh[gi][wi], lo, sg);
                      sg = fma2_h_f32(qh[gi][wi + 1], hi, sg);
                    } else if constexpr (Sh::ES == 2) {
                      const uint32_t mk = qmask[gi][v * 4 + j];
                      const uint32_t xw = (Mw[j] & mk) | (mw[j] & ~mk);
                      const float2 xf = __half22float2(*reinterpret_cast<const __half2*>(&xw));
                      sg = fmaf(qf[gi][(v * 4 + j) * 2 + 0], xf.x, sg);
                      sg = fmaf(qf[gi][(v * 4 + j) * 2 + 1], xf.y, sg);
                    } else {
                      const uint32_t mk = qmask[gi][v * 4 + j];
                      const uint32_t xw = (Mw[j] & mk) | (mw[j] & ~mk);
                      sg = fmaf(qf[gi][v * 4 + j], __uint_as_float(xw), sg);
                    }
                  }
                }
                vals[gi * NR + ro] = sg;
              }
            }
            // sums over the LPP lanes of each page, then the group max
            sub_reduce<Sh::NV, LPP / 2>(vals, lane);
            {
              constexpr int NF = Sh::NV / LPP > 1 ? Sh::NV / LPP : 1;
              const int base = sub_base<Sh::NV, LPP / 2>(lane);
#pragma unroll
              for (int i = 0; i < NF; ++i) lg[(base + i) * PPR + pg] = vals[i];
            }
          }
          __syncwarp();
          if (lane < np) {
            float sc = -INFINITY;
            if (!((bad >> lane) & 1u)) {
              sc = lg[lane];
              if constexpr (!Sh::MMAS) {
#pragma unroll
                for (int gi = 1; gi < G; ++gi) sc = fmaxf(sc, lg[gi * NR * PPR + lane]);
              }
            }
            if (cached) {
              const uint32_t key = score_key(sc);
              const uint32_t ra = smem_u32(rows + b * kCRowCap + p0 + lane);
#pragma unroll
              for (int c = 0; c < kCL; ++c) st_cl_u32(cl_map(ra, c), key);
              if (p0 + lane >= f_lo && p0 + lane < f_hi) {
                kmn = min(kmn, key);
                kmx = max(kmx, key);
              }
            } else {                         // long rows: the select reads the scores
              a.scores[(size_t)un.g * a.nnz + un.lo + p0 + lane] = sc;
            }
          }
          __syncwarp();                      // chunk slot m % NQ may be refilled
        }
        cp_async_wait_grp<0>();
        kmn = warp_min_u32(kmn);
        kmx = warp_max_u32(kmx);
        if (lane < kCL && cached && nm > 0) {   // into every CTA's min and max of row b
          red_cl_min(cl_map(smem_u32(kmm + 2 * b), lane), kmn);
          red_cl_max(cl_map(smem_u32(kmm + 2 * b + 1), lane), kmx);
        }
        // this warp's keys (and appended rows) of unit t are out: tell every
        // CTA (the lanes' stores are ordered before the release by the warp
        // barrier)
        __syncwarp();
        if (lane < kCL) arrive_cl(row_full + b, lane);
        if (cached) {
          // the scores output, from the keys (after the release, which then
          // does not wait for these stores; row b holds them until the
          // select of unit t has released it)
          float* so = a.scores + (size_t)un.g * a.nnz + un.lo;
          for (int p = pb + lane; p < pe; p += 32) so[p] = __uint_as_float(key_to_f32(rows[b * kCRowCap + p]));
        }
      }
      if (t >= 1) {
        // ------------------------------ A(t-1) ------------------------------
        const int u = t - 1, b = u & 1;
        const CUnit un = units[u];
        const int nal = n_at(un);
        const int na = nal > cw ? (nal - cw + NCW - 1) / NCW : 0;   // my pages
        W st;
        bool inited = false;                 // q loads once the first copies are out
        const T* qrow = static_cast<const T*>(a.q) + ((size_t)un.r * h_q + (size_t)un.g * G) * D;
        if (all_hands && cw < Sh::HANDS) {
          joined = true;
          if (!select_core(typename Sh::AllGrp{}, u)) { dead = true; break; }
          if (cw == 0 && lane == 0) arrive_local(sel_ready + b);   // the group synced: all of it
        } else if (!cwait_warp(sel_ready + b, (u >> 1) & 1, s_abort, a.err, lim)) {
          dead = true;
          break;
        }
        const bool ident = un.P <= K;        // every page is selected, in page order
        const bool listed = un.nsel <= kCKCap;
        const int32_t* gl = a.sel_logical + ((size_t)un.r * a.h_kv + un.g) * K;
        // the appended rows were acquired through sel_ready: order them
        // before the bulk copies that read the pool
        if (lane == 0 && na > 0) fence_proxy_async_global();
        __syncwarp();
        for (int i0 = 0; i0 < na && !dead; i0 += 32) {
          const int i = i0 + lane;
          int lp = -1, ph = -1;
          if (i < na) {
            const int wi = (int)rank + kCL * (cw + NCW * i);    // place in the selection
            if (ident) lp = wi;
            else lp = listed ? sell[b * kCKCap + wi] : __ldcg(gl + wi);
            if (lp >= 0 && lp < un.P) ph = (listed && !ident) ? selp[b * kCKCap + wi]
                                                               : __ldg(a.page_indices + un.lo + lp);
          }
          const int valid = (lp >= 0 && lp < un.P) ? min(S, un.L - lp * S) : 0;
          const bool ok = i < na && valid > 0 && ph >= 0 && ph < a.n_phys;
          if (i < na && !ok) {
            if (lp < 0 || lp >= un.P) report(a.err, QUEST_DEVERR_TABLE_RANGE);
            else if (valid <= 0) report(a.err, QUEST_DEVERR_EMPTY_PAGE);
            else report(a.err, QUEST_DEVERR_PAGE_RANGE);
          }
          // items: (page li, sub-block sb) with valid tokens, in order; each
          // is one attention tile of up to TB tokens
          unsigned rem = __ballot_sync(FULL, ok);
          int li = rem ? __ffs(rem) - 1 : -1, sb = 0;
          auto next_item = [&](int& l, int& s) {   // the item after (l, s), l = -1 at the end
            const int vl = __shfl_sync(FULL, valid, l);
            if (s + 1 < Sh::NSB && (s + 1) * Sh::TB < vl) { ++s; return; }
            const unsigned r = rem & ~((2u << l) - 1u);
            l = r ? __ffs(r) - 1 : -1;
            s = 0;
          };
          if constexpr (Sh::MMAA) {
            // 16-byte pieces by cp.async into swizzled rows (conflict-free
            // ldmatrix); one commit group per half, K and V of an item
            constexpr int KRB = D * Sh::ES;                  // bytes of a K (V) row
            auto issue_half = [&](int l, int s, int half) {
              const int pk = __shfl_sync(FULL, ph, l);
              const unsigned char* src = static_cast<const unsigned char*>(half ? a.v_pool : a.k_pool) +
                                         ((size_t)pk * a.h_kv + un.g) * BLK + (size_t)s * HALF;
              unsigned char* dst = buf + half * HALF;
#pragma unroll
              for (int k = 0; k < HALF / 512; ++k) {
                const int pc = k * 32 + lane;               // 16-byte piece of the sub-block
                cp_async16(dst + W::sw(pc / (KRB / 16), pc % (KRB / 16)), src + (size_t)pc * 16);
              }
              cp_async_commit_grp();
            };
            if (li >= 0) {
              issue_half(li, 0, 0);
              issue_half(li, 0, 1);
            }
            if (!inited) {
              st.init(qrow, a.scale_log2, lane);
              inited = true;
            }
            __half* ps = reinterpret_cast<__half*>(lg);
            const uint32_t kb = smem_u32(buf), vb = smem_u32(buf + HALF);
            while (li >= 0) {
              const int vk = min(Sh::TB, __shfl_sync(FULL, valid, li) - sb * Sh::TB);
              int l1 = li, s1 = sb;
              next_item(l1, s1);
              if constexpr (Sh::TB == 16) {
                cp_async_wait_grp<1>();                     // this K (its V may still stream)
                __syncwarp();
                st.qk(kb, vk, ps, lane);
                if (l1 >= 0) {
                  issue_half(l1, s1, 0);                    // the next K while this V is folded
                  cp_async_wait_grp<1>();
                } else {
                  cp_async_wait_grp<0>();
                }
                __syncwarp();
                st.av(vb, vk, ps, lane);
                __syncwarp();
                if (l1 >= 0) issue_half(l1, s1, 1);
              } else {                                      // several tiles: each folds whole
                cp_async_wait_grp<0>();
                __syncwarp();
                for (int j = 0; j * 16 < vk; ++j) {
                  st.qk(kb + j * 16 * KRB, vk - j * 16, ps, lane);
                  st.av(vb + j * 16 * KRB, vk - j * 16, ps, lane);
                }
                __syncwarp();
                if (l1 >= 0) {
                  issue_half(l1, s1, 0);
                  issue_half(l1, s1, 1);
                }
              }
              if (u == 0 && cw == 0 && lane == 0 && i0 == 0 && li == __ffs(rem) - 1 && sb == 0) stamp(4);
              li = l1;
              sb = s1;
            }
          } else {
            auto issue_half = [&](int l, int s, int half) {   // K (half 0) or V (half 1) of an item
              const int pk = __shfl_sync(FULL, ph, l);
              if (lane == 0) {
                uint64_t* bar = half ? vbar : kbar;
                mbar_arrive_tx(bar, HALF);
                bulk_g2s_hint(buf + half * HALF,
                              static_cast<const unsigned char*>(half ? a.v_pool : a.k_pool) +
                                  ((size_t)pk * a.h_kv + un.g) * BLK + (size_t)s * HALF,
                              HALF, bar, pol);
              }
              if (half) vpend = true; else kpend = true;
            };
            if (li >= 0) {
              issue_half(li, 0, 0);
              issue_half(li, 0, 1);
            }
            if (!inited) {
              st.init(qrow, a.scale_log2, lane);
              inited = true;
            }
            while (li >= 0) {
              const int vk = min(Sh::TB, __shfl_sync(FULL, valid, li) - sb * Sh::TB);
              int l1 = li, s1 = sb;
              next_item(l1, s1);
              if (!cwait_warp(kbar, kph & 1, s_abort, a.err, lim)) { dead = true; break; }
              ++kph;
              kpend = false;
              st.qk(reinterpret_cast<const T*>(buf), vk, lg, lane);
              if (l1 >= 0) issue_half(l1, s1, 0);          // the next K while this V is folded
              if (!cwait_warp(vbar, vph & 1, s_abort, a.err, lim)) { dead = true; break; }
              ++vph;
              vpend = false;
              st.av(reinterpret_cast<const T*>(buf + HALF), vk, lg, lane);
              if (l1 >= 0) issue_half(l1, s1, 1);
              if (u == 0 && cw == 0 && lane == 0 && i0 == 0 && vph == 1) stamp(4);
              li = l1;
              sb = s1;
            }
          }
        }
        if (dead) break;
        if (!inited) st.init(qrow, a.scale_log2, lane);   // no pages: the empty state
        const int sbf = u % Sh::NSTASH, ku = u / Sh::NSTASH;   // stash slot, its use number
        if (ku >= 1 && !cwait_warp(stash_free + sbf, (ku - 1) & 1, s_abort, a.err, lim)) {
          dead = true;
          break;
        }
        st.stash(sto + (size_t)sbf * NCW * G * D, stml + (size_t)sbf * NCW * G * 2, cw, lane);
        __syncwarp();
        if (lane == 0) arrive_local(attn_done + sbf);
      }
    }
    // a hand that gave up before the lone unit's select (so before its
    // arrival on the unit's row_full, which therefore never completes) still
    // meets the group's one barrier of a failing select: the select's verdict
    // is "failed" whoever writes it
    if constexpr (Sh::HANDSOK) {
      if (dead && all_hands && cw < Sh::HANDS && !joined) {
        if (lane == 0) *s_ok_all = 0;
        Sh::AllGrp::sync();
      }
    }
    // nothing may still be copying into this warp's buffer when the CTA exits
    cp_async_wait_grp<0>();
    for (uint32_t i = 0; kpend && i < lim; ++i) kpend = !__all_sync(FULL, try_wait_cl(kbar, kph & 1));
    for (uint32_t i = 0; vpend && i < lim; ++i) vpend = !__all_sync(FULL, try_wait_cl(vbar, vph & 1));
  } else {
    // ============================ select group ============================
    const int gt = tid - Sh::SEL0;
    bool dead = false;
    // one thread waits, the group follows its verdict
    auto gwait = [&](const uint64_t* bar, uint32_t parity) {
      if (gt == 0) *s_ok = cwait_one(bar, parity, s_abort, a.err, lim) ? 1 : 0;
      SelGrp::sync();
      const bool ok = *s_ok != 0;
      SelGrp::sync();
      return ok;
    };
    for (int t = 0; t <= n && !dead; ++t) {
      if (t < n) {
        // ------------------------------ T(t) ------------------------------
        const int u = t, b = u & 1;
        const CUnit un = units[u];
        const bool ok = all_hands ? gwait(sel_ready + b, (u >> 1) & 1) : select_core(SelGrp{}, u);
        if (!ok) { dead = true; break; }
        SelGrp::sync();
        const int P = un.P, nsel = un.nsel;
        const bool owner = (int)rank == u % kCL;
        const bool listed = nsel <= kCKCap;
        const size_t ug = (size_t)un.r * a.h_kv + un.g;
        int32_t* ol = a.sel_logical + ug * K;
        int32_t* sl = sell + b * kCKCap;
        int32_t* sp = selp + b * kCKCap;
        if (gt == 0 && !all_hands) {             // (the group's reads precede it by the barrier)
          kmm[2 * b] = 0xffffffffu;              // ready for unit u + 2
          kmm[2 * b + 1] = 0u;
          arrive_local(sel_ready + b);           // the consumers may stream the pages
#pragma unroll
          for (int c = 0; c < kCL; ++c) arrive_cl(row_free + b, c);   // row b may be refilled
        }
        if (u == 0 && gt == 0) stamp(6);
        if (owner) {                             // the call's selection outputs
          int32_t* op = a.sel_phys + ug * K;
          for (int pos = nsel + gt; pos < K; pos += kCSelT) { ol[pos] = -1; op[pos] = -1; }
          if (gt == 0) a.sel_count[ug] = nsel;
          for (int pos = gt; pos < nsel; pos += kCSelT) {
            if (listed) ol[pos] = sl[pos];
            if (listed && P > K) {
              op[pos] = sp[pos];
            } else {
              const int lp = listed ? sl[pos] : __ldcg(ol + pos);
              op[pos] = (lp >= 0 && lp < P) ? __ldg(a.page_indices + un.lo + lp) : -1;
            }
          }
          for (int i = P + gt; i < un.tp; i += kCSelT)
            a.scores[(size_t)un.g * a.nnz + un.lo + i] = -INFINITY;
        }
      }
      if (t >= 1) {
        // ------------------------------ M(t-1) ------------------------------
        const int u = t - 1;
        const CUnit un = units[u];
        const int owner = u % kCL;
        const int sbf = u % Sh::NSTASH;          // stash slot of the unit
        if (!gwait(attn_done + sbf, (u / Sh::NSTASH) & 1)) { dead = true; break; }
        const float* mo = sto + (size_t)sbf * NCW * G * D;
        const float* ml = stml + (size_t)sbf * NCW * G * 2;
        const uint32_t po = cl_map(smem_u32(part), owner);
        const uint32_t pm = cl_map(smem_u32(partml), owner);
        for (int idx = gt; idx < G * D; idx += kCSelT) {
          const int gi = idx / D, col = idx % D;
          float mx = -INFINITY;
#pragma unroll
          for (int w = 0; w < NCW; ++w) mx = fmaxf(mx, ml[(w * G + gi) * 2]);
          float o = 0.f, l = 0.f;
          if (mx != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NCW; ++w) {
              const float sc = exp2f(ml[(w * G + gi) * 2] - mx);
              o = fmaf(sc, mo[(w * G + gi) * D + col], o);
              l = fmaf(sc, ml[(w * G + gi) * 2 + 1], l);
            }
          }
          st_cl_f32(po + (uint32_t)((rank * G + gi) * D + col) * 4u, o);
          if (col == 0) {
            st_cl_f32(pm + (uint32_t)((rank * G + gi) * 2) * 4u, mx);
            st_cl_f32(pm + (uint32_t)((rank * G + gi) * 2 + 1) * 4u, l);
          }
        }
        SelGrp::sync();                           // the group's stores precede the release
        if (gt == 0) {
          arrive_cl(part_full, owner);
          arrive_local(stash_free + sbf);        // the consumers may stash unit u + NSTASH
        }
        if ((int)rank == owner) {
          if (!gwait(part_full, (u / kCL) & 1)) { dead = true; break; }
          for (int idx = gt; idx < G * D; idx += kCSelT) {
            const int gi = idx / D, col = idx % D;
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kCL; ++c) mx = fmaxf(mx, partml[(c * G + gi) * 2]);
            float o = 0.f, l = 0.f;
            if (mx != -INFINITY) {
#pragma unroll
              for (int c = 0; c < kCL; ++c) {
                const float w = exp2f(partml[(c * G + gi) * 2] - mx);
                o = fmaf(w, part[(c * G + gi) * D + col], o);
                l = fmaf(w, partml[(c * G + gi) * 2 + 1], l);
              }
            }
            const size_t orow = (size_t)un.r * h_q + (size_t)un.g * G + gi;
            a.out[orow * D + col] = l > 0.f ? o / l : 0.f;
            if (col == 0 && a.lse) a.lse[orow] = l > 0.f ? (mx + log2f(l)) * LN2 : -INFINITY;
          }
          SelGrp::sync();                         // part read before the next owned unit
        }
        if (u == n - 1 && gt == 0) stamp(7);
      }
    }
  }
  // no CTA leaves while another may still write into its shared memory
  cluster_sync_all();
  if (tid == 0) stamp(9);
}

template <typename T, int D, int S, int G, bool F8>
int cstep_clusters(int dev) {
  static std::atomic<int> cached[64];   // per device: 0 untried
  using Sh = CShape<T, D, S, G, F8>;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_acquire);
    if (c != 0) return c;
  }
  int n = 0;
  if (cudaFuncSetAttribute(cstep_kernel<T, D, S, G, F8, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Sh::SMEM) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCL * 64);
    cfg.blockDim = dim3(Sh::NT);
    cfg.dynamicSmemBytes = Sh::SMEM;
    if (cudaOccupancyMaxActiveClusters(&n, (void*)cstep_kernel<T, D, S, G, F8, true>, &cfg) != cudaSuccess)
      n = 0;
  }
  cudaGetLastError();
  if (n <= 0) n = -1;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_release);
  return n;
}

template <typename T, int D, int S, int G, bool F8>
cudaError_t cstep_launch(const StepArgs& a, const StepPlan& p, cudaStream_t s) {
  using Sh = CShape<T, D, S, G, F8>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(Sh::NT);
  cfg.dynamicSmemBytes = Sh::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  // the launch may overlap the previous kernel's tail (the kernel waits for
  // it with griddepcontrol.wait before touching global memory)
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  static std::atomic<int> pdl_ok{getenv("QUEST_NO_PDL") ? 0 : -1};   // -1 untried, 0 off, 1 on
  cfg.numAttrs = pdl_ok.load() == 0 ? 0 : 1;
  // fp16 tables of at most kCShortRows entries: the instance without the
  // long-row Top-K (fp32 keeps one instance)
  auto kern = cstep_kernel<T, D, S, G, F8, true>;
  if constexpr (sizeof(T) == 2) {
    if (a.nnz <= kCShortRows) {
      kern = cstep_kernel<T, D, S, G, F8, false>;
      int dev = 0;
      cudaGetDevice(&dev);
      static std::atomic<bool> attr_done[64];   // per device
      if (dev < 0 || dev >= 64 || !attr_done[dev].load(std::memory_order_acquire)) {
        const cudaError_t ea = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM);
        if (ea != cudaSuccess) return ea;
        if (dev >= 0 && dev < 64) attr_done[dev].store(true, std::memory_order_release);
      }
    }
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess && cfg.numAttrs == 1 && pdl_ok.load() == -1) {
    cudaGetLastError();
    pdl_ok = 0;
    cfg.numAttrs = 0;
    e = cudaLaunchKernelEx(&cfg, kern, a);
  } else if (e == cudaSuccess && cfg.numAttrs == 1) {
    pdl_ok = 1;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T, int D, bool F8>
cudaError_t cstep_launch_sg(const StepArgs& a, const StepPlan& p, cudaStream_t s) {
  if (a.page_size == 16) {
    if (a.group == 1) return cstep_launch<T, D, 16, 1, F8>(a, p, s);
    if (a.group == 2) return cstep_launch<T, D, 16, 2, F8>(a, p, s);
    if constexpr (sizeof(T) == 2) {          // groups of 4 and 8: fp16 K/V (the warp MMA)
      if (a.group == 4) return cstep_launch<T, D, 16, 4, F8>(a, p, s);
      if (a.group == 8) return cstep_launch<T, D, 16, 8, F8>(a, p, s);
    }
  } else {
    if (a.group == 1) return cstep_launch<T, D, 32, 1, F8>(a, p, s);
    if (a.group == 2) return cstep_launch<T, D, 32, 2, F8>(a, p, s);
    if constexpr (sizeof(T) == 2) {
      if (a.group == 4) return cstep_launch<T, D, 32, 4, F8>(a, p, s);
      if (a.group == 8) return cstep_launch<T, D, 32, 8, F8>(a, p, s);
    }
  }
  return cudaErrorInvalidValue;
}

template <typename T, int D, bool F8>
int cstep_clusters_sg(int dev, int page_size, int group) {
  if (page_size == 16) {
    if (group == 1) return cstep_clusters<T, D, 16, 1, F8>(dev);
    if (group == 2) return cstep_clusters<T, D, 16, 2, F8>(dev);
    if constexpr (sizeof(T) == 2) {
      if (group == 4) return cstep_clusters<T, D, 16, 4, F8>(dev);
      if (group == 8) return cstep_clusters<T, D, 16, 8, F8>(dev);
    }
  } else if (page_size == 32) {
    if (group == 1) return cstep_clusters<T, D, 32, 1, F8>(dev);
    if (group == 2) return cstep_clusters<T, D, 32, 2, F8>(dev);
    if constexpr (sizeof(T) == 2) {
      if (group == 4) return cstep_clusters<T, D, 32, 4, F8>(dev);
      if (group == 8) return cstep_clusters<T, D, 32, 8, F8>(dev);
    }
  }
  return -1;
}

}  // namespace
}  // namespace quest
