// Device helpers shared by the libquest kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/quest.h"

namespace quest {

constexpr unsigned FULL = 0xffffffffu;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// Iteration limit of every in-kernel wait; a wait that runs out sets
// QUEST_DEVERR_WAIT_TIMEOUT instead of spinning forever.
constexpr uint32_t WAIT_LIMIT = 1u << 24;

__device__ __forceinline__ void report(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------------------
// Element traits: 16-byte vectors of the stored type and fp32 conversion.
// ---------------------------------------------------------------------------
template <typename T> struct Elem;

template <> struct Elem<float> {
  static constexpr int kVec = 4;  // elements per 16 B
  __device__ __forceinline__ static float to_f(float x) { return x; }
};
template <> struct Elem<__half> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static float to_f(__half x) { return __half2float(x); }
};

// Order-preserving unsigned keys for exact min/max in the order -0 < +0.
// fp16 halves are processed two per 32-bit word; fp32 one per word.
__device__ __forceinline__ uint32_t f16x2_to_key(uint32_t x) {
  uint32_t neg = (x & 0x80008000u) >> 15;         // 1 in each negative half
  return x ^ (neg * 0x7fffu | 0x80008000u);       // neg: ~h ; pos: h | 0x8000
}
__device__ __forceinline__ uint32_t key_to_f16x2(uint32_t k) {
  uint32_t neg = ((~k) & 0x80008000u) >> 15;      // key top bit clear => was negative
  return k ^ (neg * 0x7fffu | 0x80008000u);
}
__device__ __forceinline__ uint32_t f32_to_key(uint32_t x) {
  return x ^ ((x & 0x80000000u) ? 0xffffffffu : 0x80000000u);
}
__device__ __forceinline__ uint32_t key_to_f32(uint32_t k) {
  return k ^ ((k & 0x80000000u) ? 0x80000000u : 0xffffffffu);
}

template <typename T> struct KeyOps;
template <> struct KeyOps<__half> {
  static constexpr uint32_t kMinInit = 0xffffffffu;   // +inf-like for both halves
  static constexpr uint32_t kMaxInit = 0x00000000u;
  __device__ __forceinline__ static uint32_t to_key(uint32_t w) { return f16x2_to_key(w); }
  __device__ __forceinline__ static uint32_t from_key(uint32_t k) { return key_to_f16x2(k); }
  __device__ __forceinline__ static uint32_t kmin(uint32_t a, uint32_t b) { return __vminu2(a, b); }
  __device__ __forceinline__ static uint32_t kmax(uint32_t a, uint32_t b) { return __vmaxu2(a, b); }
};
template <> struct KeyOps<float> {
  static constexpr uint32_t kMinInit = 0xffffffffu;
  static constexpr uint32_t kMaxInit = 0x00000000u;
  __device__ __forceinline__ static uint32_t to_key(uint32_t w) { return f32_to_key(w); }
  __device__ __forceinline__ static uint32_t from_key(uint32_t k) { return key_to_f32(k); }
  __device__ __forceinline__ static uint32_t kmin(uint32_t a, uint32_t b) { return a < b ? a : b; }
  __device__ __forceinline__ static uint32_t kmax(uint32_t a, uint32_t b) { return a > b ? a : b; }
};

// 16-byte loads/stores.
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 ld_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
// Streaming 16-byte load that does not allocate in L1 (read-once data).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
// L2 policy that evicts the lines it tags first (for data streamed once).
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint4 ld_stream_v4_hint(const void* p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p), "l"(pol));
  return r;
}
// 8-byte forms of the two above (E4M3 summary halves of 8 dims).
__device__ __forceinline__ uint2 ld_stream_v2_hint(const void* p, uint64_t pol) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;"
               : "=r"(r.x), "=r"(r.y) : "l"(p), "l"(pol));
  return r;
}
__device__ __forceinline__ void st_v2(void* p, uint2 v) {
  asm volatile("st.global.v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// Unpack a 16-byte vector of T into fp32.
template <typename T> __device__ __forceinline__ void unpack16(uint4 v, float* out);
template <> __device__ __forceinline__ void unpack16<float>(uint4 v, float* out) {
  out[0] = __uint_as_float(v.x); out[1] = __uint_as_float(v.y);
  out[2] = __uint_as_float(v.z); out[3] = __uint_as_float(v.w);
}
template <> __device__ __forceinline__ void unpack16<__half>(uint4 v, float* out) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}

// s + a.lo * b.lo + a.hi * b.hi for two packed fp16 pairs, accumulated in
// fp32 in that order: each product of two fp16 values is exact in fp32, so
// the mixed-precision FMA (fp16 sources, fp32 addend) rounds exactly as an
// fp32 FMA of the converted values would, without the conversions.
__device__ __forceinline__ float fma2_h_f32(uint32_t a2, uint32_t b2, float s) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
      : "+f"(s) : "r"(a2), "r"(b2));
  return s;
}

// Page upper-bound contribution of one 16-byte vector of dims (Quest page
// §1.1 eq (2)): sum_j max(q_j m_j, q_j M_j). Since m_j <= M_j, the larger
// product is q_j M_j when q_j >= 0 and q_j m_j otherwise, so each dim costs a
// select and one FMA. For fp16 the select works on packed halves (sign mask)
// and the products of two fp16 values are exact in fp32.
template <typename T> __device__ __forceinline__ float bound16(uint4 q, uint4 m, uint4 M);
template <> __device__ __forceinline__ float bound16<__half>(uint4 q, uint4 m, uint4 M) {
  const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
  const uint32_t mw[4] = {m.x, m.y, m.z, m.w};
  const uint32_t Mw[4] = {M.x, M.y, M.z, M.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t mk = ((~qw[i] & 0x80008000u) >> 15) * 0xffffu;   // halves with q >= 0
    const uint32_t xw = (Mw[i] & mk) | (mw[i] & ~mk);
    const float2 qf = __half22float2(*reinterpret_cast<const __half2*>(&qw[i]));
    const float2 xf = __half22float2(*reinterpret_cast<const __half2*>(&xw));
    s = fmaf(qf.x, xf.x, s);
    s = fmaf(qf.y, xf.y, s);
  }
  return s;
}
template <> __device__ __forceinline__ float bound16<float>(uint4 q, uint4 m, uint4 M) {
  const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
  const uint32_t mw[4] = {m.x, m.y, m.z, m.w};
  const uint32_t Mw[4] = {M.x, M.y, M.z, M.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float qf = __uint_as_float(qw[i]);
    const float xf = __uint_as_float((qw[i] & 0x80000000u) ? mw[i] : Mw[i]);
    s = fmaf(qf, xf, s);
  }
  return s;
}

// ---------------------------------------------------------------------------
// E4M3 page summaries (Quest page §3, the paragraph on the summary dtype).
// Format: the OCP 8-bit float without infinities -- sign bit, 4 exponent bits
// (bias 7), 3 mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6);
// S.1111.111 is NaN; the largest finite magnitude is 448. The min of a page
// is rounded toward -inf and the max toward +inf, so the stored box still
// contains the page's keys and its bound stays an upper bound (eq (4)). A
// rounded zero is stored as +0 (code 0x00), so codes and values correspond
// one to one and min/max may be taken on either.
// ---------------------------------------------------------------------------

// Code of the largest E4M3 value <= x (x finite). Sets `ovf` when x < -448:
// nothing representable lies below, the code saturates at -448.
__device__ __forceinline__ uint32_t e4m3_floor(float x, bool& ovf) {
  const float a = fabsf(x);
  const bool neg = x < 0.f;
  float n;   // a in steps of its E4M3 binade
  int base;  // code of that binade's first value, less the 8 implied steps
  if (a < 0x1p-6f) {
    n = a * 512.f;                                   // subnormal step 2^-9
    base = 0;
  } else {
    const int e = (int)((__float_as_uint(a) >> 23) & 0xffu) - 127;   // 2^e <= a
    n = a * __uint_as_float((uint32_t)(130 - e) << 23);              // a / 2^(e-3) in [8, 16)
    base = (e + 7) * 8 - 8;
  }
  // x >= 0 rounds its magnitude down, x < 0 up; a carry out of the mantissa
  // lands on the next binade's first code, which is the next value
  int c = base + (int)(neg ? ceilf(n) : floorf(n));
  if (c > 0x7e) {
    ovf = ovf || neg;
    c = 0x7e;
  }
  return c == 0 ? 0u : ((neg ? 0x80u : 0u) | (uint32_t)c);
}

// Code of the smallest E4M3 value >= x, i.e. -floor(-x). Sets `ovf` when x > 448.
__device__ __forceinline__ uint32_t e4m3_ceil(float x, bool& ovf) {
  const uint32_t c = e4m3_floor(-x, ovf);
  return c == 0 ? 0u : (c ^ 0x80u);
}

// Two E4M3 codes (bytes lo, hi of `pair`, already placed at bits 8..15 and
// 24..31) -> the fp16 pair of their values times 2^-8. Moving the 7 magnitude
// bits down by one puts the exponent field e at fp16 exponent e and the
// mantissa on top of fp16's, i.e. the value 2^(e-15) (1 + m/8), or m 2^-17
// for e = 0 (an fp16 subnormal): exactly the E4M3 value times 2^-8.
__device__ __forceinline__ uint32_t e4m3x2_placed_to_h2_scaled(uint32_t placed) {
  return ((placed >> 1) & 0x3f803f80u) | (placed & 0x80008000u);
}
// Codes 0,1 / 2,3 of a word of four codes, as fp32 values: the hardware
// conversion of a pair of E4M3 codes to an fp16 pair (exact), then to fp32.
__device__ __forceinline__ float2 e4m3x2_to_f2(uint16_t pair) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(pair));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}
__device__ __forceinline__ float2 e4m3x4_lo_f2(uint32_t w) { return e4m3x2_to_f2((uint16_t)w); }
__device__ __forceinline__ float2 e4m3x4_hi_f2(uint32_t w) {
  return e4m3x2_to_f2((uint16_t)(w >> 16));
}
// Codes 0,1 / 2,3 of a word of four codes as an exact fp16 pair (raw bits).
__device__ __forceinline__ uint32_t e4m3x4_lo_h2(uint32_t w) {
  uint32_t h = e4m3x2_placed_to_h2_scaled(__byte_perm(w, 0u, 0x1404));
  const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&h), __float2half2_rn(256.f));
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t e4m3x4_hi_h2(uint32_t w) {
  uint32_t h = e4m3x2_placed_to_h2_scaled(__byte_perm(w, 0u, 0x3424));
  const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&h), __float2half2_rn(256.f));
  return *reinterpret_cast<const uint32_t*>(&v);
}
// Per-code select mask of a word of four codes: 0xff where the query of that
// dim is >= 0 (take the max), from the fp16 query words of dims 0,1 and 2,3.
__device__ __forceinline__ uint32_t e4m3_qsel(uint32_t q01, uint32_t q23) {
  const uint32_t hi = __byte_perm(q01, q23, 0x7531);   // the high byte of each half
  return ((~hi & 0x80808080u) >> 7) * 0xffu;
}
// The same mask from per-half masks (0xffff where q >= 0) of dims 0,1 and 2,3.
__device__ __forceinline__ uint32_t e4m3_qsel_from_masks(uint32_t m01, uint32_t m23) {
  return __byte_perm(m01, m23, 0x6420);
}
// Page-bound contribution (eq (2)) of 4 dims with E4M3 summary words m, M and
// fp32 queries q[0..3]: sum_j q_j * (q_j >= 0 ? M_j : m_j).
__device__ __forceinline__ float bound4_e4m3(const float* q, uint32_t sel, uint32_t m,
                                             uint32_t M, float s) {
  const uint32_t x = (M & sel) | (m & ~sel);
  const float2 lo = e4m3x4_lo_f2(x), hi = e4m3x4_hi_f2(x);
  s = fmaf(q[0], lo.x, s);
  s = fmaf(q[1], lo.y, s);
  s = fmaf(q[2], hi.x, s);
  s = fmaf(q[3], hi.y, s);
  return s;
}
// eq (2) over 8 dims: fp16 queries (one 16-byte vector) against E4M3 codes
// of m and M (8 bytes each). Exact up to fp32 rounding of the sum.
__device__ __forceinline__ float bound8_e4m3(uint4 q, uint2 m, uint2 M) {
  const float2 q0 = __half22float2(*reinterpret_cast<const __half2*>(&q.x));
  const float2 q1 = __half22float2(*reinterpret_cast<const __half2*>(&q.y));
  const float2 q2 = __half22float2(*reinterpret_cast<const __half2*>(&q.z));
  const float2 q3 = __half22float2(*reinterpret_cast<const __half2*>(&q.w));
  const float qa[4] = {q0.x, q0.y, q1.x, q1.y}, qb[4] = {q2.x, q2.y, q3.x, q3.y};
  float s = bound4_e4m3(qa, e4m3_qsel(q.x, q.y), m.x, M.x, 0.f);
  return bound4_e4m3(qb, e4m3_qsel(q.z, q.w), m.y, M.y, s);
}
// Four fp16 keys (two words) -> floor / ceil codes packed in one word.
__device__ __forceinline__ uint32_t e4m3x4_floor_h(uint32_t k01, uint32_t k23, bool& ovf) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&k01));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&k23));
  return e4m3_floor(a.x, ovf) | (e4m3_floor(a.y, ovf) << 8) | (e4m3_floor(b.x, ovf) << 16) |
         (e4m3_floor(b.y, ovf) << 24);
}
__device__ __forceinline__ uint32_t e4m3x4_ceil_h(uint32_t k01, uint32_t k23, bool& ovf) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&k01));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&k23));
  return e4m3_ceil(a.x, ovf) | (e4m3_ceil(a.y, ovf) << 8) | (e4m3_ceil(b.x, ovf) << 16) |
         (e4m3_ceil(b.y, ovf) << 24);
}

// ---------------------------------------------------------------------------
// mbarrier + 1-D bulk async copy (global -> shared), CTA-local.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// try_wait that lets the thread sleep (up to `ns`) until the phase completes,
// instead of spinning on the barrier.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(ns) : "memory");
  return ok != 0;
}
// Bounded wait: returns false (and the caller reports) if the limit is hit
// (2^21 tries of up to 1 us each).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 21); ++i)
    if (mbar_try_wait_sleep(bar, parity, 1000u)) return true;
  return false;
}

// Warp-uniform form: every lane polls and the warp agrees on the outcome;
// false once `limit` tries (up to about 1 us each) pass without the phase.
__device__ __forceinline__ bool warp_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (__all_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity, 1000u))) return true;
  return false;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(smem_u32(dst_smem)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint(void* dst_smem, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      :: "r"(smem_u32(dst_smem)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol) : "memory");
}

// Programmatic dependent launch controls (no-ops when launched without PDL).
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Warp helpers.
__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
__device__ __forceinline__ uint32_t warp_min_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = min(v, __shfl_xor_sync(FULL, v, o));
  return v;
}
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = max(v, __shfl_xor_sync(FULL, v, o));
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

}  // namespace quest
