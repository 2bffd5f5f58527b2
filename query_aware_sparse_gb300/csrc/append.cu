// a1: cache append with incremental per-page key min/max
// (Quest page §1.2 eq (8), §3 eq (14); page recycling in §3).
//
// One CTA per touched (request, page) segment: the new tokens of one request
// that land in one page are contiguous in k_new, so a CTA copies them into
// the pool and folds them into that page's summary for every KV head without
// any cross-CTA reduction. A page whose slot 0 is written by this call
// restarts its summary from the new keys (fresh page / recycled slot).
// With E4M3 summaries (fp16 keys only) the old codes decode exactly into
// fp16, the fold runs as usual, and the result is rounded out again (min
// toward -inf, max toward +inf): rounding is monotone, so this equals the
// rounding of the exact summary (Quest page §1.2: min/max kept in the
// quantized domain; §3: directed rounding keeps the box conservative).
#include "common.cuh"
#include "internal.h"

namespace quest {
namespace {

constexpr int kAppendThreads = 256;

// Finds which (request, page-of-request) segment CTA `seg` handles. Returns
// false when `seg` is past the last segment. Warp 0 scans the requests.
__device__ bool find_segment(const AppendArgs& a, int seg, int* r_out, int* j_out) {
  __shared__ int s_r, s_j;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int base = 0;
    int found_r = -1, found_j = 0;
    for (int r0 = 0; r0 < a.batch && found_r < 0; r0 += 32) {
      int r = r0 + lane;
      int cnt = 0;
      if (r < a.batch) {
        int n = a.append_indptr[r + 1] - a.append_indptr[r];
        if (n > 0) {
          int p0 = a.seq_lens_before[r];
          cnt = (p0 + n - 1) / a.page_size - p0 / a.page_size + 1;
        }
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += t;
      }
      int excl = incl - cnt;
      unsigned hit = __ballot_sync(FULL, cnt > 0 && seg >= base + excl && seg < base + incl);
      if (hit) {
        int src = __ffs(hit) - 1;
        found_r = r0 + src;
        found_j = seg - base - __shfl_sync(FULL, excl, src);
      }
      base += __shfl_sync(FULL, incl, 31);
    }
    if (lane == 0) { s_r = found_r; s_j = found_j; }
  }
  __syncthreads();
  *r_out = s_r;
  *j_out = s_j;
  return s_r >= 0;
}

template <typename T, int D, bool F8>
__global__ void __launch_bounds__(kAppendThreads)
append_kernel(const AppendArgs a) {
  static_assert(!F8 || sizeof(T) == 2, "E4M3 summaries take fp16 keys");
  using K = KeyOps<T>;
  constexpr int VEC = Elem<T>::kVec;   // elements per 16 B
  constexpr int CH = D / VEC;          // 16-byte chunks per row

  int r, j;
  if (!find_segment(a, blockIdx.x, &r, &j)) return;

  const int S = a.page_size;
  const int n_r = a.append_indptr[r + 1] - a.append_indptr[r];
  const int pos0 = a.seq_lens_before[r];
  const int lp = pos0 / S + j;
  const int t_begin = max(pos0, lp * S);
  const int t_end = min(pos0 + n_r, (lp + 1) * S);
  const bool fresh = (t_begin == lp * S);
  const int table_pages = a.page_indptr[r + 1] - a.page_indptr[r];
  if (lp >= table_pages) {
    if (threadIdx.x == 0) report(a.err, QUEST_DEVERR_TABLE_RANGE);
    return;
  }
  const int pp = a.page_indices[a.page_indptr[r] + lp];
  if (pp < 0 || pp >= a.n_phys) {
    if (threadIdx.x == 0) report(a.err, QUEST_DEVERR_PAGE_RANGE);
    return;
  }
  const int row0 = a.append_indptr[r] + (t_begin - pos0);
  const int ntok = t_end - t_begin;
  const int slot0 = t_begin - lp * S;

  const size_t row_stride = (size_t)a.h_kv * D;               // elements per token
  const T* kn = static_cast<const T*>(a.k_new) + (size_t)row0 * row_stride;
  const T* vn = static_cast<const T*>(a.v_new) + (size_t)row0 * row_stride;
  T* kp = static_cast<T*>(a.k_pool) + (size_t)pp * a.h_kv * S * D;
  T* vp = static_cast<T*>(a.v_pool) + (size_t)pp * a.h_kv * S * D;
  T* sm = static_cast<T*>(a.summary) + (size_t)pp * a.h_kv * 2 * D;
  uint8_t* sm8 = static_cast<uint8_t*>(a.summary) + (size_t)pp * a.h_kv * 2 * D;
  bool ovf = false;

  for (int item = threadIdx.x; item < a.h_kv * CH; item += blockDim.x) {
    const int g = item / CH;
    const int c = item % CH;
    uint4 mn, mx;
    if (fresh) {
      mn = make_uint4(K::kMinInit, K::kMinInit, K::kMinInit, K::kMinInit);
      mx = make_uint4(K::kMaxInit, K::kMaxInit, K::kMaxInit, K::kMaxInit);
    } else {
      uint4 om, oM;
      if constexpr (F8) {        // VEC codes -> VEC exact fp16 values
        const uint2 cm = *reinterpret_cast<const uint2*>(sm8 + ((size_t)g * 2 + 0) * D + c * VEC);
        const uint2 cM = *reinterpret_cast<const uint2*>(sm8 + ((size_t)g * 2 + 1) * D + c * VEC);
        om = make_uint4(e4m3x4_lo_h2(cm.x), e4m3x4_hi_h2(cm.x), e4m3x4_lo_h2(cm.y), e4m3x4_hi_h2(cm.y));
        oM = make_uint4(e4m3x4_lo_h2(cM.x), e4m3x4_hi_h2(cM.x), e4m3x4_lo_h2(cM.y), e4m3x4_hi_h2(cM.y));
      } else {
        om = ld_v4(sm + ((size_t)g * 2 + 0) * D + c * VEC);
        oM = ld_v4(sm + ((size_t)g * 2 + 1) * D + c * VEC);
      }
      mn = make_uint4(K::to_key(om.x), K::to_key(om.y), K::to_key(om.z), K::to_key(om.w));
      mx = make_uint4(K::to_key(oM.x), K::to_key(oM.y), K::to_key(oM.z), K::to_key(oM.w));
    }
    const size_t src_off = (size_t)g * D + c * VEC;
    const size_t dst_off = ((size_t)g * S + slot0) * D + c * VEC;
#pragma unroll 4
    for (int t = 0; t < ntok; ++t) {
      uint4 kv = ld_stream_v4(kn + (size_t)t * row_stride + src_off);
      uint4 vv = ld_stream_v4(vn + (size_t)t * row_stride + src_off);
      st_v4(kp + dst_off + (size_t)t * D, kv);
      st_v4(vp + dst_off + (size_t)t * D, vv);
      mn.x = K::kmin(mn.x, K::to_key(kv.x)); mx.x = K::kmax(mx.x, K::to_key(kv.x));
      mn.y = K::kmin(mn.y, K::to_key(kv.y)); mx.y = K::kmax(mx.y, K::to_key(kv.y));
      mn.z = K::kmin(mn.z, K::to_key(kv.z)); mx.z = K::kmax(mx.z, K::to_key(kv.z));
      mn.w = K::kmin(mn.w, K::to_key(kv.w)); mx.w = K::kmax(mx.w, K::to_key(kv.w));
    }
    const uint4 vm = make_uint4(K::from_key(mn.x), K::from_key(mn.y), K::from_key(mn.z), K::from_key(mn.w));
    const uint4 vM = make_uint4(K::from_key(mx.x), K::from_key(mx.y), K::from_key(mx.z), K::from_key(mx.w));
    if constexpr (F8) {
      *reinterpret_cast<uint2*>(sm8 + ((size_t)g * 2 + 0) * D + c * VEC) =
          make_uint2(e4m3x4_floor_h(vm.x, vm.y, ovf), e4m3x4_floor_h(vm.z, vm.w, ovf));
      *reinterpret_cast<uint2*>(sm8 + ((size_t)g * 2 + 1) * D + c * VEC) =
          make_uint2(e4m3x4_ceil_h(vM.x, vM.y, ovf), e4m3x4_ceil_h(vM.z, vM.w, ovf));
    } else {
      st_v4(sm + ((size_t)g * 2 + 0) * D + c * VEC, vm);
      st_v4(sm + ((size_t)g * 2 + 1) * D + c * VEC, vM);
    }
  }
  if (F8 && ovf) report(a.err, QUEST_DEVERR_FP8_RANGE);
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
  if (a.batch == 0 || a.n_new == 0) return cudaSuccess;
  // A request with n new tokens touches at most ceil(n / S) + 1 pages, and
  // sum_r ceil(n_r / S) < n_new / S + batch, so this bounds the segment count.
  const long long segs = (long long)(a.n_new + a.page_size - 1) / a.page_size + 2LL * a.batch;
  dim3 grid((unsigned)segs);
  if (a.dtype == QUEST_F16 && a.summary_fp8) {
    if (a.head_dim == 128) append_kernel<__half, 128, true><<<grid, kAppendThreads, 0, s>>>(a);
    else append_kernel<__half, 64, true><<<grid, kAppendThreads, 0, s>>>(a);
  } else if (a.dtype == QUEST_F16) {
    if (a.head_dim == 128) append_kernel<__half, 128, false><<<grid, kAppendThreads, 0, s>>>(a);
    else append_kernel<__half, 64, false><<<grid, kAppendThreads, 0, s>>>(a);
  } else {
    if (a.head_dim == 128) append_kernel<float, 128, false><<<grid, kAppendThreads, 0, s>>>(a);
    else append_kernel<float, 64, false><<<grid, kAppendThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace quest
