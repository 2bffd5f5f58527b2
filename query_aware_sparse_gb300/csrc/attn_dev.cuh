// Warp-level attention over one staged (page, KV head) block: QK for the G
// query heads of the group, online softmax in fp32 with base-2 exponents, AV
// accumulation (Quest page Fig. 1 candidate attention; the softmax merge over
// pages keeps one running max and sum per row, Quest page §2.1).
//
// Lanes own D/32 consecutive dims; the QK partial sums of a tile of tokens
// are summed across lanes with a transposed butterfly (each halving step
// trades half of the live values), so G*TT dot products cost G*TT - 1
// shuffles instead of 5 per dot product.
#pragma once

#include "common.cuh"

namespace quest {

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

// Sum each of NV per-lane values over the 32 lanes. Afterwards, for NV >= 32
// lane l holds the sums of indices l*(NV/32) + i in v[i]; for NV < 32 lane l
// holds the sum of index l >> (5 - log2(NV)) in v[0].
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

template <int N>
struct ILog2 { static constexpr int value = 1 + ILog2<N / 2>::value; };
template <> struct ILog2<1> { static constexpr int value = 0; };

template <typename T, int D, int S, int G>
struct WarpAttn {
  static constexpr int VD = D / 32;                        // dims per lane
  static constexpr int TT = (G * S <= 64) ? S : 64 / G;    // tokens per tile
  static constexpr int NV = G * TT;                        // logits per tile
  static constexpr int BLOCK_BYTES = S * D * (int)sizeof(T);

  float q[G][VD];
  float m[G], l[G], acc[G][VD];

  // q rows of the G heads of the group (contiguous rows of D), pre-scaled so
  // that exp2 of the scaled dot product equals e^(sm_scale * q.k).
  __device__ __forceinline__ void init(const T* qrows, float scale_log2, int lane) {
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
#pragma unroll
      for (int v = 0; v < VD; ++v)
        q[gi][v] = Elem<T>::to_f(qrows[(size_t)gi * D + lane * VD + v]) * scale_log2;
      m[gi] = -INFINITY;
      l[gi] = 0.f;
#pragma unroll
      for (int v = 0; v < VD; ++v) acc[gi][v] = 0.f;
    }
  }

  // Fold one staged page (K block Kb, V block Vb, `valid` leading tokens) into
  // the running state. `lg` is this warp's NV-float shared scratch. Heads
  // whose bit of `hmask` is clear did not choose the page and skip it.
  __device__ __forceinline__ void page(const T* Kb, const T* Vb, int valid, float* lg, int lane,
                                       unsigned hmask = ~0u) {
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
        constexpr int SH = 5 - ILog2<NV>::value;
        if ((lane & ((1 << SH) - 1)) == 0) {
          const int vi = lane >> SH;
          lg[vi] = (t0 + vi % TT < valid) ? part[0] : -INFINITY;
        }
      }
      __syncwarp();
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        if (!((hmask >> gi) & 1u)) {         // not this head's page: weight 0
          if (lane < TT) lg[gi * TT + lane] = 0.f;
          continue;
        }
        const float x = lg[gi * TT + (lane % TT)];
        const float mt = warp_max(x);
        const float m_new = fmaxf(m[gi], mt);
        const float alpha = exp2f(m[gi] - m_new);
        const float p = exp2f(x - m_new);
        const float psum = warp_sum(lane < TT ? p : 0.f);
        l[gi] = l[gi] * alpha + psum;
        m[gi] = m_new;
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

  // page() in two halves, for pages of one tile (TT == S): qk() folds the
  // logits of the K block into the running max and sum and leaves the
  // probabilities in `lg`; av() then accumulates the V block with them. The
  // K block is not read after qk() returns, so its buffer may be refilled
  // while av() runs.
  __device__ __forceinline__ void qk(const T* Kb, int valid, float* lg, int lane) {
    static_assert(TT == S, "one tile per page");
    float part[NV];
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
      float kr[VD];
      lds_row<T, VD>(Kb + (size_t)tt * D + lane * VD, kr);
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
        lg[vi] = (vi % TT < valid) ? part[i] : -INFINITY;
      }
    } else {
      constexpr int SH = 5 - ILog2<NV>::value;
      if ((lane & ((1 << SH) - 1)) == 0) {
        const int vi = lane >> SH;
        lg[vi] = (vi % TT < valid) ? part[0] : -INFINITY;
      }
    }
    __syncwarp();
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      const float x = lg[gi * TT + (lane % TT)];
      const float mt = warp_max(x);
      const float m_new = fmaxf(m[gi], mt);
      const float alpha = exp2f(m[gi] - m_new);
      const float p = exp2f(x - m_new);
      const float psum = warp_sum(lane < TT ? p : 0.f);
      l[gi] = l[gi] * alpha + psum;
      m[gi] = m_new;
#pragma unroll
      for (int v = 0; v < VD; ++v) acc[gi][v] *= alpha;
      __syncwarp();
      if (lane < TT) lg[gi * TT + lane] = p;
    }
    __syncwarp();
  }
  __device__ __forceinline__ void av(const T* Vb, int valid, const float* lg, int lane) {
    for (int tt = 0; tt < valid; ++tt) {
      float vr[VD];
      lds_row<T, VD>(Vb + (size_t)tt * D + lane * VD, vr);
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        const float p = lg[gi * TT + tt];
#pragma unroll
        for (int v = 0; v < VD; ++v) acc[gi][v] = fmaf(p, vr[v], acc[gi][v]);
      }
    }
    __syncwarp();
  }

  // Store this warp's state in shared memory: mo[w][gi][D], ml[w][gi][2].
  __device__ __forceinline__ void stash(float* mo, float* ml, int w, int lane) const {
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
#pragma unroll
      for (int v = 0; v < VD; ++v) mo[(w * G + gi) * D + lane * VD + v] = acc[gi][v];
      if (lane == 0) {
        ml[(w * G + gi) * 2 + 0] = m[gi];
        ml[(w * G + gi) * 2 + 1] = l[gi];
      }
    }
  }
};

// Merge NW stashed warp states of a CTA into one (o, max, sum) per query head
// and write them through `put(gi, col, o)` and `put_ml(gi, max, sum)`.
template <int D, int G, int NW, int NT, typename PutO, typename PutML>
__device__ __forceinline__ void merge_warps(const float* mo, const float* ml, PutO put,
                                            PutML put_ml) {
  for (int idx = threadIdx.x; idx < G * D; idx += NT) {
    const int gi = idx / D, col = idx % D;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) mx = fmaxf(mx, ml[(w * G + gi) * 2]);
    float o = 0.f, l = 0.f;
    if (mx != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float sc = exp2f(ml[(w * G + gi) * 2] - mx);
        o = fmaf(sc, mo[(w * G + gi) * D + col], o);
        l = fmaf(sc, ml[(w * G + gi) * 2 + 1], l);
      }
    }
    put(gi, col, o);
    if (col == 0) put_ml(gi, mx, l);
  }
}

}  // namespace quest
