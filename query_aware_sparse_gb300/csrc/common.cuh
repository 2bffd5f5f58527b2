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
