// a4 + a5: attention over the selected pages only, read in place from the
// paged pool (Quest page Fig. 1 and §2.1; token set and 1/sqrt(d) scale of
// PageWeaver notes §2 eq (1)-(2)), split over chunks of pages, then merged
// by log-sum-exp (Quest page §2.1: one row-global max and sum, never a
// per-page softmax average).
//
// Split-K kernel: one CTA per (request, KV head, chunk of pages), NW warps.
// Each warp owns a ring of NST shared-memory slots; its lane 0 streams the
// warp's pages in with 1-D bulk async copies (cp.async.bulk, completion on
// an mbarrier): one (page, head) K block and V block are each S*d contiguous
// elements of the pool. QK runs on FMA with lanes over d and a transposed
// shuffle reduction over tokens; online softmax in fp32 (base-2 exponent);
// AV accumulates in registers. The CTA merges its warps and writes one
// partial (o, max, sum) per query head; the combine kernel merges chunks.
// Decode attention is a matrix-vector product per query head (G <= 8 rows
// share a KV head), too thin for a tensor-core tile, so it stays on FMA.
#include "common.cuh"
#include "internal.h"

namespace quest {
namespace {

constexpr int kNW = 4;        // warps per CTA
constexpr int kNST = 2;       // bulk-copy slots per warp
constexpr int kMaxWarpPages = 32;

template <typename T, int D, int S, int G>
struct AttnShape {
  static constexpr int VD = D / 32;                        // dims per lane
  static constexpr int TT = (G * S <= 64) ? S : 64 / G;    // tokens per tile
  static constexpr int NV = G * TT;                        // logits per tile
  static constexpr int BLOCK_BYTES = S * D * (int)sizeof(T);  // one K (or V) page block
  static constexpr int STAGE_BYTES = kNW * kNST * 2 * BLOCK_BYTES;
  static constexpr int BAR_OFF = STAGE_BYTES;
  static constexpr int LOGIT_OFF = BAR_OFF + kNW * kNST * 8;
  static constexpr int DESC_OFF = LOGIT_OFF + kNW * NV * 4;
  static constexpr int SMEM = DESC_OFF + kNW * kMaxWarpPages * 8;
  static_assert(kNW * G * (D + 2) * 4 <= STAGE_BYTES, "merge buffer must fit in the stage area");
};

// Load VD consecutive elements of T from shared memory as fp32.
template <typename T, int VD>
__device__ __forceinline__ void lds_row(const T* p, float (&out)[VD]);
template <> __device__ __forceinline__ void lds_row<__half, 4>(const __half* p, float (&o)[4]) {
  uint2 w = *reinterpret_cast<const uint2*>(p);
  float2 a = __half22float2(*reinterpret_cast<__half2*>(&w.x));
  float2 b = __half22float2(*reinterpret_cast<__half2*>(&w.y));
  o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
}
template <> __device__ __forceinline__ void lds_row<__half, 2>(const __half* p, float (&o)[2]) {
  float2 a = __half22float2(*reinterpret_cast<const __half2*>(p));
  o[0] = a.x; o[1] = a.y;
}
template <> __device__ __forceinline__ void lds_row<float, 4>(const float* p, float (&o)[4]) {
  float4 a = *reinterpret_cast<const float4*>(p);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
}
template <> __device__ __forceinline__ void lds_row<float, 2>(const float* p, float (&o)[2]) {
  float2 a = *reinterpret_cast<const float2*>(p);
  o[0] = a.x; o[1] = a.y;
}

template <typename T, int VD>
__device__ __forceinline__ void ldg_row(const T* p, float (&out)[VD]) {
#pragma unroll
  for (int v = 0; v < VD; ++v) out[v] = Elem<T>::to_f(p[v]);
}

// One halving step of the transposed butterfly: lanes with bit `o` set keep
// the upper half of the N live values, the others the lower half; each adds
// its partner's copy of the half it keeps.
template <int N>
__device__ __forceinline__ void tr_step(float* v, int lane, int o) {
  constexpr int H = N / 2;
  const bool up = (lane & o) != 0;
#pragma unroll
  for (int i = 0; i < H; ++i) {
    const float send = up ? v[i] : v[i + H];
    const float keep = up ? v[i + H] : v[i];
    v[i] = keep + __shfl_xor_sync(FULL, send, o);
  }
}

// Sum each of NV per-lane partial values over the 32 lanes. Afterwards, for
// NV >= 32 lane l holds the sums of indices l*(NV/32) + i in v[i]; for
// NV < 32 lane l holds the sum of index l >> (5 - log2(NV)) in v[0].
template <int NV>
__device__ __forceinline__ void transpose_reduce(float (&v)[NV], int lane) {
  if constexpr (NV >= 2) tr_step<NV>(v, lane, 16);
  if constexpr (NV >= 4) tr_step<NV / 2>(v, lane, 8);
  if constexpr (NV >= 8) tr_step<NV / 4>(v, lane, 4);
  if constexpr (NV >= 16) tr_step<NV / 8>(v, lane, 2);
  if constexpr (NV >= 32) tr_step<NV / 16>(v, lane, 1);
  if constexpr (NV < 32) {
#pragma unroll
    for (int o = 16 / NV; o >= 1; o >>= 1) v[0] += __shfl_xor_sync(FULL, v[0], o);
  }
}

template <int NV>
struct Log2 { static constexpr int value = NV <= 1 ? 0 : 1 + Log2<NV / 2>::value; };
template <> struct Log2<1> { static constexpr int value = 0; };

template <typename T, int D, int S, int G>
__global__ void __launch_bounds__(kNW * 32)
attn_split_kernel(const AttnArgs a) {
  using Sh = AttnShape<T, D, S, G>;
  constexpr int VD = Sh::VD, TT = Sh::TT, NV = Sh::NV;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::BAR_OFF);
  float* logits_all = reinterpret_cast<float*>(smem + Sh::LOGIT_OFF);
  int2* desc_all = reinterpret_cast<int2*>(smem + Sh::DESC_OFF);

  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c = blockIdx.x % a.n_chunks;
  const int unit = blockIdx.x / a.n_chunks;     // r * h_kv + g
  const int g = unit % a.h_kv, r = unit / a.h_kv;
  const int h_q = a.h_kv * G;
  const int L = a.seq_lens[r];
  const size_t sel_base = (size_t)unit * a.k;

  uint64_t* my_bars = bars + w * kNST;
  float* lg = logits_all + w * NV;
  int2* desc = desc_all + w * kMaxWarpPages;
  T* my_stage = reinterpret_cast<T*>(smem) + (size_t)w * kNST * 2 * S * D;

  // This warp's pages: j = c*cp + w + NW*i, i < nmine.
  const int jc0 = c * a.chunk_pages;
  const int jc1 = min(a.k, jc0 + a.chunk_pages);
  const int j0 = jc0 + w;
  const int nmine = j0 < jc1 ? (jc1 - j0 + kNW - 1) / kNW : 0;
  int my_pp = -1, my_valid = 0;
  if (lane < nmine) {
    const int j = j0 + lane * kNW;
    const int lp = __ldg(a.sel_logical + sel_base + j);
    const int pp = __ldg(a.sel_phys + sel_base + j);
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
  if (lane == 0) {
    for (int s = 0; s < kNST; ++s) mbar_init(my_bars + s, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const size_t head_block = (size_t)S * D;                 // elements per (page, head)
  const T* kbase = static_cast<const T*>(a.k_pool) + (size_t)g * head_block;
  const T* vbase = static_cast<const T*>(a.v_pool) + (size_t)g * head_block;
  const size_t page_stride = (size_t)a.h_kv * head_block;

  auto issue = [&](int n) {
    const int slot = n % kNST;
    const int pp = desc[n].x;
    T* dst = my_stage + (size_t)slot * 2 * head_block;
    mbar_expect_tx(my_bars + slot, 2 * Sh::BLOCK_BYTES);
    bulk_g2s(dst, kbase + (size_t)pp * page_stride, Sh::BLOCK_BYTES, my_bars + slot);
    bulk_g2s(dst + head_block, vbase + (size_t)pp * page_stride, Sh::BLOCK_BYTES, my_bars + slot);
  };
  if (lane == 0)
    for (int n = 0; n < min(kNST, nv); ++n) issue(n);

  // Queries of the group, pre-scaled so that exp2 gives e^(scale * q.k).
  float q[G][VD];
#pragma unroll
  for (int gi = 0; gi < G; ++gi) {
    ldg_row<T, VD>(static_cast<const T*>(a.q) + ((size_t)r * h_q + g * G + gi) * D + lane * VD, q[gi]);
#pragma unroll
    for (int v = 0; v < VD; ++v) q[gi][v] *= a.scale_log2;
  }
  float m_run[G], l_run[G], acc[G][VD];
#pragma unroll
  for (int gi = 0; gi < G; ++gi) {
    m_run[gi] = -INFINITY;
    l_run[gi] = 0.f;
#pragma unroll
    for (int v = 0; v < VD; ++v) acc[gi][v] = 0.f;
  }

  for (int n = 0; n < nv; ++n) {
    const int slot = n % kNST;
    const int valid = desc[n].y;
    const bool ok = mbar_wait_bounded(my_bars + slot, (n / kNST) & 1);
    if (!ok) {
      if (lane == 0) report(a.err, QUEST_DEVERR_WAIT_TIMEOUT);
    } else {
      const T* Kb = my_stage + (size_t)slot * 2 * head_block;
      const T* Vb = Kb + head_block;
      for (int t0 = 0; t0 < valid; t0 += TT) {
        float part[NV];
#pragma unroll
        for (int tt = 0; tt < TT; ++tt) {
          float kr[VD];
          lds_row<T, VD>(Kb + (size_t)(t0 + tt) * D + lane * VD, kr);
#pragma unroll
          for (int gi = 0; gi < G; ++gi) {
            float s = 0.f;
#pragma unroll
            for (int v = 0; v < VD; ++v) s = fmaf(q[gi][v], kr[v], s);
            part[gi * TT + tt] = s;
          }
        }
        transpose_reduce<NV>(part, lane);
        if constexpr (NV >= 32) {
#pragma unroll
          for (int i = 0; i < NV / 32; ++i) {
            const int vi = lane * (NV / 32) + i;
            lg[vi] = (t0 + vi % TT < valid) ? part[i] : -INFINITY;
          }
        } else {
          constexpr int SH = 5 - Log2<NV>::value;
          if ((lane & ((1 << SH) - 1)) == 0) {
            const int vi = lane >> SH;
            lg[vi] = (t0 + vi % TT < valid) ? part[0] : -INFINITY;
          }
        }
        __syncwarp();
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
          const float x = lg[gi * TT + (lane % TT)];
          const float mt = warp_max(x);
          const float m_new = fmaxf(m_run[gi], mt);
          const float alpha = exp2f(m_run[gi] - m_new);
          const float p = exp2f(x - m_new);
          const float psum = warp_sum(lane < TT ? p : 0.f);
          l_run[gi] = l_run[gi] * alpha + psum;
          m_run[gi] = m_new;
#pragma unroll
          for (int v = 0; v < VD; ++v) acc[gi][v] *= alpha;
          __syncwarp();
          if (lane < TT) lg[gi * TT + lane] = p;
        }
        __syncwarp();
        const int tv = min(TT, valid - t0);
        for (int tt = 0; tt < tv; ++tt) {
          float vr[VD];
          lds_row<T, VD>(Vb + (size_t)(t0 + tt) * D + lane * VD, vr);
#pragma unroll
          for (int gi = 0; gi < G; ++gi) {
            const float p = lg[gi * TT + tt];
#pragma unroll
            for (int v = 0; v < VD; ++v) acc[gi][v] = fmaf(p, vr[v], acc[gi][v]);
          }
        }
        __syncwarp();
      }
    }
    __syncwarp();
    if (lane == 0 && n + kNST < nv) {
      fence_proxy_async_smem();
      issue(n + kNST);
    }
  }

  // Merge the warps of this CTA (stage area reused once every warp is done).
  __syncthreads();
  float* mo = reinterpret_cast<float*>(smem);                 // [NW][G][D]
  float* ml = mo + kNW * G * D;                               // [NW][G][2]
#pragma unroll
  for (int gi = 0; gi < G; ++gi) {
#pragma unroll
    for (int v = 0; v < VD; ++v) mo[(w * G + gi) * D + lane * VD + v] = acc[gi][v];
    if (lane == 0) {
      ml[(w * G + gi) * 2 + 0] = m_run[gi];
      ml[(w * G + gi) * 2 + 1] = l_run[gi];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += kNW * 32) {
    const int gi = idx / D, col = idx % D;
    float mx = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kNW; ++ww) mx = fmaxf(mx, ml[(ww * G + gi) * 2]);
    float o = 0.f, l = 0.f;
    if (mx != -INFINITY) {
#pragma unroll
      for (int ww = 0; ww < kNW; ++ww) {
        const float sc = exp2f(ml[(ww * G + gi) * 2] - mx);
        o = fmaf(sc, mo[(ww * G + gi) * D + col], o);
        l = fmaf(sc, ml[(ww * G + gi) * 2 + 1], l);
      }
    }
    const size_t row = ((size_t)r * h_q + g * G + gi) * a.n_chunks + c;
    a.part_o[row * D + col] = o;
    if (col == 0) {
      a.part_ml[row * 2 + 0] = mx;
      a.part_ml[row * 2 + 1] = l;
    }
  }
}

// One warp per (request, query head): LSE merge of the chunk partials.
template <int D>
__global__ void __launch_bounds__(128)
attn_combine_kernel(const AttnArgs a) {
  constexpr int VD = D / 32;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);       // r * h_q + h
  const int h_q = a.h_kv * a.group;
  if (row >= a.batch * h_q) return;
  const float* pml = a.part_ml + (size_t)row * a.n_chunks * 2;
  const float* po = a.part_o + (size_t)row * a.n_chunks * D;
  float mx = -INFINITY;
  for (int c = lane; c < a.n_chunks; c += 32) mx = fmaxf(mx, pml[c * 2]);
  mx = warp_max(mx);
  float o[VD];
#pragma unroll
  for (int v = 0; v < VD; ++v) o[v] = 0.f;
  float l = 0.f;
  if (mx != -INFINITY) {
    for (int c = 0; c < a.n_chunks; ++c) {
      const float mc = pml[c * 2];
      if (mc == -INFINITY) continue;
      const float sc = exp2f(mc - mx);
      l = fmaf(sc, pml[c * 2 + 1], l);
#pragma unroll
      for (int v = 0; v < VD; ++v) o[v] = fmaf(sc, po[(size_t)c * D + lane * VD + v], o[v]);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int v = 0; v < VD; ++v) a.out[(size_t)row * D + lane * VD + v] = o[v] * inv;
  if (a.lse && lane == 0) a.lse[row] = l > 0.f ? (mx + log2f(l)) * LN2 : -INFINITY;
}

template <typename T, int D, int S, int G>
cudaError_t launch_split(const AttnArgs& a, cudaStream_t s) {
  using Sh = AttnShape<T, D, S, G>;
  auto kern = attn_split_kernel<T, D, S, G>;
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_done[64] = {};   // per device; racing setters write the same value
  if (dev >= 64 || !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_done[dev] = true;
  }
  const unsigned grid = (unsigned)a.batch * a.h_kv * a.n_chunks;
  kern<<<grid, kNW * 32, Sh::SMEM, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned rows = (unsigned)a.batch * a.h_kv * a.group;
  attn_combine_kernel<D><<<(rows + 3) / 4, 128, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T, int D, int S>
cudaError_t launch_g(const AttnArgs& a, cudaStream_t s) {
  switch (a.group) {
    case 1: return launch_split<T, D, S, 1>(a, s);
    case 2: return launch_split<T, D, S, 2>(a, s);
    case 4: return launch_split<T, D, S, 4>(a, s);
    case 8: return launch_split<T, D, S, 8>(a, s);
  }
  return cudaErrorInvalidValue;
}

template <typename T, int D>
cudaError_t launch_s(const AttnArgs& a, cudaStream_t s) {
  return a.page_size == 16 ? launch_g<T, D, 16>(a, s) : launch_g<T, D, 32>(a, s);
}

int smem_for(int dtype, int head_dim, int page_size, int group) {
  const int esz = dtype == QUEST_F16 ? 2 : 4;
  const int block = page_size * head_dim * esz;
  const int tt = (group * page_size <= 64) ? page_size : 64 / group;
  return kNW * kNST * 2 * block + kNW * kNST * 8 + kNW * group * tt * 4 + kNW * kMaxWarpPages * 8;
}

}  // namespace

bool attn_supported(int32_t dtype, int32_t head_dim, int32_t page_size, int32_t group) {
  return (dtype == QUEST_F16 || dtype == QUEST_F32) && (head_dim == 64 || head_dim == 128) &&
         (page_size == 16 || page_size == 32) &&
         (group == 1 || group == 2 || group == 4 || group == 8) &&
         smem_for(dtype, head_dim, page_size, group) <= 227 * 1024;   // per-CTA limit
}

AttnPlan plan_attn(int32_t batch, int32_t h_kv, int32_t group, int32_t head_dim,
                   int32_t page_size, int32_t dtype, int32_t k) {
  int dev = 0, sms = 148, smem_sm = 228 * 1024;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  }
  cudaGetLastError();
  const int smem = smem_for(dtype, head_dim, page_size, group) + 1024;   // + per-CTA reserve
  const int per_sm = smem_sm / smem > 0 ? smem_sm / smem : 1;
  const long long target = (long long)sms * per_sm;
  const long long total = (long long)batch * h_kv * k;
  long long cp = (total + target * kNW - 1) / (target * kNW) * kNW;       // pages per chunk
  if (cp < kNW) cp = kNW;
  if (cp > kNW * kMaxWarpPages) cp = kNW * kMaxWarpPages;
  AttnPlan p;
  p.chunk_pages = (int32_t)cp;
  p.n_chunks = (int32_t)((k + cp - 1) / cp);
  const size_t rows = (size_t)batch * h_kv * group * p.n_chunks;
  p.workspace_bytes = rows * head_dim * sizeof(float) + rows * 2 * sizeof(float);
  p.workspace_bytes = (p.workspace_bytes + 255) & ~(size_t)255;
  return p;
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s) {
  if (a.batch == 0 || a.h_kv == 0) return cudaSuccess;
  if (a.dtype == QUEST_F16)
    return a.head_dim == 128 ? launch_s<__half, 128>(a, s) : launch_s<__half, 64>(a, s);
  return a.head_dim == 128 ? launch_s<float, 128>(a, s) : launch_s<float, 64>(a, s);
}

}  // namespace quest
