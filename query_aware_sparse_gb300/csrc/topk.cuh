// Block-wide fixed-budget Top-K over one (request, KV head) row of page
// scores (Quest page Fig. 1, §1.1, §2): the K largest scores, ties to the
// lower page index, emitted in ascending page order. Used by the standalone
// select kernel and by the fused decode step.
//
// Scores map to order-preserving 32-bit keys (-0 folded onto +0). The block
// first reduces min and max: bits above the highest bit where they differ
// are common to every key, so the MSB-first radix select starts below them
// with 11-bit digits (2048 shared-memory bins: a row of a few thousand
// scores rarely puts many keys in one bin, so the bin atomics do not pile
// up), and stops as soon as the digit bucket holding the K-th key is taken
// whole. A block scan in page order then emits the winners. Rows whose keys
// sit in shared memory (up to 32 per thread) take block_topk_smem, which
// holds each thread's keys in registers: once the first digit has isolated a
// boundary bucket of at most kTopkGather keys, that bucket is ranked directly
// instead of taking further digits.
#pragma once

#include "common.cuh"

namespace quest {

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t x = __float_as_uint(f == 0.f ? 0.f : f);   // -0 -> +0
  return x ^ ((x & 0x80000000u) ? 0xffffffffu : 0x80000000u);
}

// Thread groups the routines below run on: the whole CTA (__syncthreads),
// or NTH threads starting at thread BASE (a multiple of 32) that meet at
// named barrier ID.
struct CtaGrp {
  __device__ __forceinline__ static int tid() { return threadIdx.x; }
  __device__ __forceinline__ static void sync() { __syncthreads(); }
};
template <int ID, int BASE, int NTH>
struct BarGrp {
  static_assert(BASE % 32 == 0 && NTH % 32 == 0, "groups are whole warps");
  static constexpr int kN = NTH;
  __device__ __forceinline__ static int tid() { return (int)threadIdx.x - BASE; }
  __device__ __forceinline__ static void sync() {
    asm volatile("bar.sync %0, %1;" :: "n"(ID), "n"(NTH) : "memory");
  }
};

// Hook told about pages that are certain to be selected as soon as the first
// radix digit is known (before the boundary bucket is resolved): the caller
// may start fetching them early. The default does nothing.
struct NoEarly {
  __device__ __forceinline__ void operator()(int) const {}
};

constexpr int kTopkBits = 11;                 // radix digit width
constexpr int kTopkBins = 1 << kTopkBits;

constexpr int kTopkGather = 256;              // largest boundary bucket ranked directly

template <int NT>
struct TopkSmem {
  alignas(16) uint32_t hist[kTopkBins];
  uint32_t red[2][NT / 32];
  unsigned long long scan[NT / 32];
  alignas(16) uint32_t gkey[kTopkGather];
  alignas(16) int32_t gidx[kTopkGather];
  uint32_t gmark[kTopkGather];
  uint32_t digit, krem, done, bcnt, gcount;
};

// Exclusive block scan of a 64-bit value.
template <int NT, class Grp = CtaGrp>
__device__ __forceinline__ unsigned long long topk_excl_scan(unsigned long long v,
                                                             TopkSmem<NT>& sm) {
  constexpr int NWP = NT / 32;
  const int lane = Grp::tid() & 31, warp = Grp::tid() >> 5;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned long long t = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sm.scan[warp] = incl;
  Grp::sync();
  if (warp == 0) {
    unsigned long long w = lane < NWP ? sm.scan[lane] : 0ull;
    unsigned long long wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      unsigned long long t = __shfl_up_sync(FULL, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < NWP) sm.scan[lane] = wi - w;
  }
  Grp::sync();
  const unsigned long long r = sm.scan[warp] + incl - v;
  Grp::sync();   // scan[] may be reused right after
  return r;
}

// Top-K of the P keys of one row, read through `key_at(i)` (shared memory or
// global): emit(pos, i) is called once for each of the min(P, K) selected
// pages i, pos being its place in ascending page order. All NT threads of
// the block must call it (it synchronises the block).
template <int NT, typename KeyAt, typename Emit, class Grp = CtaGrp>
__device__ void block_topk_keys(int P, int K, KeyAt key_at, TopkSmem<NT>& sm, Emit emit) {
  const int tid = Grp::tid(), lane = tid & 31, warp = tid >> 5;
  constexpr int NWP = NT / 32;

  if (P <= K) {                     // every scored page is selected
    for (int i = tid; i < P; i += NT) emit(i, i);
    return;
  }
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (int i = tid; i < P; i += NT) {
    const uint32_t k = key_at(i);
    kmin = min(kmin, k);
    kmax = max(kmax, k);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(FULL, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(FULL, kmax, o));
  }
  if (lane == 0) { sm.red[0][warp] = kmin; sm.red[1][warp] = kmax; }
  for (int i = tid; i < kTopkBins; i += NT) sm.hist[i] = 0;
  Grp::sync();
  kmin = sm.red[0][0];
  kmax = sm.red[1][0];
#pragma unroll
  for (int w = 1; w < NWP; ++w) { kmin = min(kmin, sm.red[0][w]); kmax = max(kmax, sm.red[1][w]); }

  // Radix select below the common prefix of min and max.
  constexpr int BPT = kTopkBins / NT;            // bins per thread in the digit search
  static_assert(BPT * NT == kTopkBins, "bins must split evenly over the block");
  uint32_t T, need;
  bool ge_mode;            // select key >= T (bucket taken whole) vs the tie rule
  if (kmin == kmax) {
    T = kmin; need = K; ge_mode = false;
  } else {
    int hi = 31 - __clz(kmin ^ kmax);           // highest differing bit
    uint32_t prefix = kmin & ~((hi == 31) ? 0xffffffffu : ((2u << hi) - 1u));
    uint32_t krem = K;
    ge_mode = false;
    T = 0; need = 0;
    while (true) {
      const int shift = max(hi - (kTopkBits - 1), 0);
      const int nbits = hi - shift + 1;
      const uint32_t dmask = (1u << nbits) - 1u;
      const uint32_t hi_mask = (hi == 31) ? 0u : ~((2u << hi) - 1u);
      for (int i = tid; i < P; i += NT) {
        const uint32_t k = key_at(i);
        if ((k & hi_mask) == prefix) atomicAdd(&sm.hist[(k >> shift) & dmask], 1u);
      }
      Grp::sync();
      // thread t owns bins [t*BPT, t*BPT + BPT); count of keys in higher bins
      uint32_t h[BPT], tot = 0;
#pragma unroll
      for (int j = 0; j < BPT; ++j) { h[j] = sm.hist[tid * BPT + j]; tot += h[j]; }
      uint32_t incl = tot;                         // suffix sum within the warp
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t t = __shfl_down_sync(FULL, incl, o);
        if (lane + o < 32) incl += t;
      }
      if (lane == 0) sm.red[0][warp] = incl;       // warp totals
      Grp::sync();
      uint32_t above = incl - tot;
      for (int w = warp + 1; w < NWP; ++w) above += sm.red[0][w];
      uint32_t cum = above;
#pragma unroll
      for (int j = BPT - 1; j >= 0; --j) {
        if (cum < krem && krem <= cum + h[j]) {
          sm.digit = tid * BPT + j;
          sm.krem = krem - cum;
          sm.done = (h[j] == krem - cum) ? 1u : 0u;   // bucket taken whole
        }
        cum += h[j];
      }
#pragma unroll
      for (int j = 0; j < BPT; ++j) sm.hist[tid * BPT + j] = 0;   // ready for the next pass
      Grp::sync();
      prefix |= sm.digit << shift;
      krem = sm.krem;
      if (sm.done || shift == 0) {
        T = prefix;
        need = krem;
        ge_mode = sm.done && shift > 0;
        break;
      }
      hi = shift - 1;
    }
    Grp::sync();   // everyone has read sm.digit/krem/done
  }

  // Stable compaction in page order.
  const int per = (P + NT - 1) / NT;
  const int c0 = min(P, tid * per), c1 = min(P, c0 + per);
  uint32_t gt = 0, eq = 0;
  for (int i = c0; i < c1; ++i) {
    const uint32_t k = key_at(i);
    if (ge_mode) gt += k >= T;
    else { gt += k > T; eq += k == T; }
  }
  const unsigned long long ex = topk_excl_scan<NT, Grp>(((unsigned long long)gt << 32) | eq, sm);
  uint32_t gt_b = (uint32_t)(ex >> 32), eq_b = (uint32_t)ex;
  for (int i = c0; i < c1; ++i) {
    const uint32_t k = key_at(i);
    int pos = -1;
    if (ge_mode) {
      if (k >= T) pos = gt_b++;
    } else if (k > T) {
      pos = gt_b + min(eq_b, need);
      ++gt_b;
    } else if (k == T) {
      if (eq_b < need) pos = gt_b + eq_b;
      ++eq_b;
    }
    if (pos >= 0 && pos < K) emit(pos, i);
  }
}

// Top-K of P fp32 scores `sc` (global) for one row; `keys` caches up to `cap`
// keys in shared memory (a longer row re-reads the scores from L2 per pass).
// Pages with forced(i) (nforced of [0, P), at most K: the local window +
// sink pages of the hybrid budget) are always kept.
template <int NT, typename PhysOf, typename Forced>
__device__ void block_topk(const float* __restrict__ sc, int P, int K, uint32_t* keys, int cap,
                           TopkSmem<NT>& sm, int32_t* out_logical, int32_t* out_phys,
                           int32_t* out_count, PhysOf phys_of, Forced forced, int nforced);

// Top-K of P <= 32 * NT keys held in shared memory (`keys`, P rounded up to
// a multiple of 4 * NT readable, 16-byte aligned; only read), whose
// block-wide min and max the caller has already reduced. Same result as
// block_topk_keys. Pages with forced(i) (nforced of them, at most K) are kept
// outright and the other pages compete for the remaining K - nforced;
// kmin / kmax are over the other pages' keys only. `sm.hist` must be all
// zero on entry and is all zero on return.
//
// Thread t holds the keys [t*per, t*per + per) in registers (per a multiple
// of 4, at most KPT), read once with 16-byte loads; every pass then works on
// registers. After the first radix digit, a boundary bucket of at most
// kTopkGather keys is ranked directly (key, then lower index) instead of
// taking more digits: its winners are marked with the top key and its
// losers with 0 (through the gather slot each thread remembers for its
// bucket keys), so one threshold then selects exactly K keys. The page-
// order compaction packs (greater, equal) counts into 32 bits (P < 65536).
template <int NT, int KPT, typename Emit, typename Forced, class Grp = CtaGrp,
          typename Early = NoEarly>
__device__ void topk_regs(int P, int K, uint32_t* keys, uint32_t kmin, uint32_t kmax,
                          TopkSmem<NT>& sm, Emit emit, Forced forced, int nforced,
                          Early early = Early()) {
  static_assert(KPT % 4 == 0 && KPT <= 32, "keys per thread: a multiple of 4, at most 32");
  const int tid = Grp::tid(), lane = tid & 31, warp = tid >> 5;
  constexpr int NWP = NT / 32;
  constexpr int BPT = kTopkBins / NT;            // bins per thread in the digit search
  static_assert(BPT % 4 == 0, "bins are read as 16-byte vectors");

  const int per = (P + 4 * NT - 1) / (4 * NT) * 4;
  const int c0 = tid * per;
  uint32_t kr[KPT];
  uint32_t inr = 0, comp = 0;                    // bit j: key c0 + j exists / competes
#pragma unroll
  for (int v = 0; v < KPT / 4; ++v) {
    const uint4 x = 4 * v < per ? *reinterpret_cast<const uint4*>(keys + c0 + 4 * v)
                                : make_uint4(0u, 0u, 0u, 0u);
    kr[4 * v] = x.x; kr[4 * v + 1] = x.y; kr[4 * v + 2] = x.z; kr[4 * v + 3] = x.w;
#pragma unroll
    for (int j = 4 * v; j < 4 * v + 4; ++j) {
      const int i = c0 + j;
      if (j < per && i < P) {
        inr |= 1u << j;
        if (!forced(i)) comp |= 1u << j;
      }
    }
  }
  const int Kq = K - nforced;                    // the competing pages' share
  uint32_t T = 0xffffffffu, need = 0;
  bool ge_mode = false;    // select key >= T vs (key > T, then `need` of key == T)
  if (Kq <= 0) {
    need = 0;              // no competing key passes: (> 0xffffffff) is false, need 0
  } else if (kmin == kmax) {
    T = kmin; need = Kq;
  } else {
    int hi = 31 - __clz(kmin ^ kmax);           // highest differing bit
    uint32_t prefix = kmin & ~((hi == 31) ? 0xffffffffu : ((2u << hi) - 1u));
    uint32_t krem = Kq;
    bool first = true;
    while (true) {
      const int shift = max(hi - (kTopkBits - 1), 0);
      const int nbits = hi - shift + 1;
      const uint32_t dmask = (1u << nbits) - 1u;
      const uint32_t hi_mask = (hi == 31) ? 0u : ~((2u << hi) - 1u);
#pragma unroll
      for (int j = 0; j < KPT; ++j)
        if (((comp >> j) & 1u) && (kr[j] & hi_mask) == prefix)
          atomicAdd(&sm.hist[(kr[j] >> shift) & dmask], 1u);
      if (tid == 0) sm.gcount = 0;
      Grp::sync();
      // thread t owns bins [t*BPT, t*BPT + BPT); count of keys in higher bins
      uint32_t h[BPT], tot = 0;
#pragma unroll
      for (int j = 0; j < BPT; j += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(&sm.hist[tid * BPT + j]);
        h[j] = v.x; h[j + 1] = v.y; h[j + 2] = v.z; h[j + 3] = v.w;
        tot += v.x + v.y + v.z + v.w;
        *reinterpret_cast<uint4*>(&sm.hist[tid * BPT + j]) = make_uint4(0u, 0u, 0u, 0u);
      }
      uint32_t incl = tot;                         // suffix sum within the warp
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t t = __shfl_down_sync(FULL, incl, o);
        if (lane + o < 32) incl += t;
      }
      if (lane == 0) sm.red[0][warp] = incl;       // warp totals
      Grp::sync();
      uint32_t cum = incl - tot;
#pragma unroll
      for (int w = 0; w < NWP; ++w)
        if (w > warp) cum += sm.red[0][w];
#pragma unroll
      for (int j = BPT - 1; j >= 0; --j) {
        if (cum < krem && krem <= cum + h[j]) {
          sm.digit = tid * BPT + j;
          sm.krem = krem - cum;
          sm.bcnt = h[j];
          sm.done = (h[j] == krem - cum) ? 1u : 0u;   // bucket taken whole
        }
        cum += h[j];
      }
      Grp::sync();
      prefix |= sm.digit << shift;
      krem = sm.krem;
      const uint32_t bcnt = sm.bcnt;
      if (first) {
        // keys above the boundary bucket (or in it, when it is taken whole)
        // and the forced pages are selected whatever the rest of the select
        // decides
        first = false;
        const unsigned long long thr =
            (sm.done || shift == 0) ? prefix : (unsigned long long)prefix + (1ull << shift);
#pragma unroll
        for (int j = 0; j < KPT; ++j)
          if ((((comp >> j) & 1u) && kr[j] >= thr) || (((inr & ~comp) >> j) & 1u)) early(c0 + j);
      }
      if (sm.done || shift == 0) {
        T = prefix;
        need = krem;
        ge_mode = sm.done && shift > 0;
        break;
      }
      if (bcnt <= (uint32_t)kTopkGather) {
        // rank the bucket [prefix, prefix + 2^shift) directly
        const uint32_t span = (1u << shift) - 1u;
        uint32_t inb = 0;                          // bit j: key c0 + j is in the bucket
        uint32_t slots[KPT / 4];                   // byte j % 4 of word j / 4: its gather slot
#pragma unroll
        for (int j = 0; j < KPT / 4; ++j) slots[j] = 0u;
#pragma unroll
        for (int j = 0; j < KPT; ++j) {
          if (((comp >> j) & 1u) && (kr[j] & ~span) == prefix) {
            inb |= 1u << j;
            const uint32_t at = atomicAdd(&sm.gcount, 1u);
            sm.gkey[at] = kr[j];
            sm.gidx[at] = c0 + j;
            slots[j / 4] |= (at & 0xffu) << (8 * (j % 4));
          }
        }
        Grp::sync();
        if (tid < (int)bcnt) {
          const uint32_t mk = sm.gkey[tid];
          const int mi = sm.gidx[tid];
          uint32_t r4[4] = {0u, 0u, 0u, 0u};
          const int n4 = (int)bcnt & ~3;
#pragma unroll 1
          for (int j = 0; j < n4; j += 4) {          // four independent counts per step
            const uint4 kj = *reinterpret_cast<const uint4*>(&sm.gkey[j]);
            const int4 ij = *reinterpret_cast<const int4*>(&sm.gidx[j]);
            r4[0] += (kj.x > mk) || (kj.x == mk && ij.x < mi);
            r4[1] += (kj.y > mk) || (kj.y == mk && ij.y < mi);
            r4[2] += (kj.z > mk) || (kj.z == mk && ij.z < mi);
            r4[3] += (kj.w > mk) || (kj.w == mk && ij.w < mi);
          }
          for (int j = n4; j < (int)bcnt; ++j) {
            const uint32_t kj = sm.gkey[j];
            r4[0] += (kj > mk) || (kj == mk && sm.gidx[j] < mi);
          }
          sm.gmark[tid] = (r4[0] + r4[1] + r4[2] + r4[3]) < krem ? 0xffffffffu : 0u;
        }
        Grp::sync();
#pragma unroll
        for (int j = 0; j < KPT; ++j)               // take the marks back
          if ((inb >> j) & 1u) kr[j] = sm.gmark[(slots[j / 4] >> (8 * (j % 4))) & 0xffu];
        const unsigned long long top = (unsigned long long)prefix + (1ull << shift);
        T = top > 0xffffffffull ? 0xffffffffu : (uint32_t)top;
        need = 0;
        ge_mode = true;
        break;
      }
      hi = shift - 1;
    }
    Grp::sync();   // sm.digit/krem/done/bcnt read by all before any reuse
  }

  // Stable compaction in page order over the register keys (branch-free:
  // `win` = selected outright, `tie` = a key equal to T competing for `need`).
  // In ge_mode, keys >= T win: the same as keys > T - 1 with no ties (T > 0
  // there, as a digit bucket above the lowest one was taken whole).
  const uint32_t Tg = ge_mode ? T - 1u : T;
  uint32_t wins = 0, ties = 0;                   // bit j: key c0 + j wins / ties
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const uint32_t f = (inr & ~comp) >> j & 1u;
    const uint32_t w = f | (uint32_t)(kr[j] > Tg);
    const uint32_t t = (uint32_t)(!ge_mode) & (comp >> j & 1u) & (uint32_t)(kr[j] == T);
    wins |= (w & (inr >> j)) << j;
    ties |= t << j;
  }
  const uint32_t cnt = ((uint32_t)__popc(wins) << 16) | (uint32_t)__popc(ties);
  uint32_t incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sm.red[1][warp] = incl;
  Grp::sync();
  uint32_t ex = incl - cnt;
#pragma unroll
  for (int w = 0; w < NWP; ++w)
    if (w < warp) ex += sm.red[1][w];
  // a winner's place: winners before it (all of them precede it in page
  // order) + ties before it that were taken (at most `need`); a tie's place
  // likewise, if it is among the first `need` ties
  const uint32_t gt_b = ex >> 16, eq_b = ex & 0xffffu;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const uint32_t below = (1u << j) - 1u;
    const uint32_t gt = gt_b + (uint32_t)__popc(wins & below);
    const uint32_t eq = eq_b + (uint32_t)__popc(ties & below);
    const bool w = (wins >> j) & 1u, t = ((ties >> j) & 1u) && eq < need;
    const int pos = (int)(gt + min(eq, need));
    if ((w || t) && pos < K) emit(pos, c0 + j);
  }
}

// Top-K of P <= 32 * NT keys in shared memory (see topk_regs): picks the
// register footprint for the row length.
// MAXP bounds P where the caller knows a smaller bound: the register forms
// no row can need are left out.
template <int NT, typename Emit, typename Forced, class Grp = CtaGrp, typename Early = NoEarly,
          int MAXP = 32 * NT>
__device__ void block_topk_smem(int P, int K, uint32_t* keys, uint32_t kmin, uint32_t kmax,
                                TopkSmem<NT>& sm, Emit emit, Forced forced, int nforced,
                                Early early = Early()) {
  if (P <= K) {                     // every scored page is selected
    for (int i = Grp::tid(); i < P; i += NT) emit(i, i);
    return;
  }
  if (P <= 8 * NT)
    topk_regs<NT, 8, Emit, Forced, Grp, Early>(P, K, keys, kmin, kmax, sm, emit, forced, nforced, early);
  else if (MAXP <= 16 * NT || P <= 16 * NT)
    topk_regs<NT, 16, Emit, Forced, Grp, Early>(P, K, keys, kmin, kmax, sm, emit, forced, nforced, early);
  else if constexpr (MAXP > 16 * NT)
    topk_regs<NT, 32, Emit, Forced, Grp, Early>(P, K, keys, kmin, kmax, sm, emit, forced, nforced, early);
}

template <int NT, typename PhysOf, typename Forced>
__device__ void block_topk(const float* __restrict__ sc, int P, int K, uint32_t* keys, int cap,
                           TopkSmem<NT>& sm, int32_t* out_logical, int32_t* out_phys,
                           int32_t* out_count, PhysOf phys_of, Forced forced, int nforced) {
  // outputs: out_logical / out_phys [K] in ascending page order, -1 padded
  auto emit = [&](int pos, int i) { out_logical[pos] = i; out_phys[pos] = phys_of(i); };
  const int n = P < K ? P : K;
  for (int i = n + threadIdx.x; i < K; i += NT) { out_logical[i] = -1; out_phys[i] = -1; }
  if (threadIdx.x == 0) *out_count = n;
  const bool cached = P <= cap && P > K;
  if (!cached) {
    block_topk_keys<NT>(P, K, [sc, forced](int i) {
                          return forced(i) ? 0xffffffffu : score_key(__ldcg(sc + i));
                        }, sm, emit);
    return;
  }
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (int i = tid; i < P; i += NT) {
    const uint32_t k = score_key(__ldcg(sc + i));
    keys[i] = k;
    if (!forced(i)) {
      kmin = min(kmin, k);
      kmax = max(kmax, k);
    }
  }
  kmin = warp_min_u32(kmin);
  kmax = warp_max_u32(kmax);
  if (lane == 0) { sm.red[0][warp] = kmin; sm.red[1][warp] = kmax; }
  for (int i = tid; i < kTopkBins; i += NT) sm.hist[i] = 0;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) { kmin = min(kmin, sm.red[0][w]); kmax = max(kmax, sm.red[1][w]); }
  if (P <= 32 * NT && P <= cap) {
    block_topk_smem<NT>(P, K, keys, kmin, kmax, sm, emit, forced, nforced);
  } else {        // longer cached rows: the general routine over the shared-memory keys
    block_topk_keys<NT>(P, K, [keys, forced](int i) { return forced(i) ? 0xffffffffu : keys[i]; },
                        sm, emit);
  }
}

}  // namespace quest
