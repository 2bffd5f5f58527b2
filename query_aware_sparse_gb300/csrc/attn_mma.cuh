// Warp-level attention for the G >= 4 query heads of one KV head (GQA), fp16
// pages of 16 tokens, on the warp MMA (mma.sync m16n8k16: fp16 in, fp32
// accumulate). Quest page Fig. 1 candidate attention; the online softmax over
// pages keeps one running max and sum per head (Quest page §2.1).
//
// Per page:  S^T = K Q^T     (16 tokens x 8 heads: the group's G heads, the
//                              rest of the 8 columns zero), k = head dims;
//            O^T += V^T P^T  (16 dims per m-tile x 8 heads), k = tokens.
// The dims are a sum index of S and a row index of O, so each side may take
// them in any order it likes as long as A and B agree: lanes load K and V
// rows straight from global memory in 16-byte pieces that are contiguous
// across the lanes of a warp instruction (no shared-memory staging, no bank
// conflicts), and the fragments are taken from those registers as they are.
//
// Register layout (gid = lane / 4, t = lane % 4):
//   K: rows gid and gid + 8, 16-byte vectors i < D/32 at dims 32 i + 8 t;
//      k-tile j of QK takes vector j / 2, words 2 (j % 2) and 2 (j % 2) + 1.
//   q: head gid (zero for gid >= G), the same dims as K.
//   V: token rows 2t, 2t+1, 2t+8, 2t+9, vectors i < D/64 at dims 64 i + 8 gid;
//      m-tile mt of AV takes word mt % 4 of vector mt / 4 (dims d, d + 1 with
//      d = 64 (mt / 4) + 8 gid + 2 (mt % 4)), interleaved by token pair.
//   O: acc[mt] = O[2t][d], O[2t+1][d], O[2t][d+1], O[2t+1][d+1].
#pragma once

#include "common.cuh"

namespace quest {

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte load through L2 only (coherent with this kernel's own writes: the
// appended rows), marked evict-first: pages are read once.
__device__ __forceinline__ uint4 ld_cg_v4_hint(const void* p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.cg.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p), "l"(pol));
  return r;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int w) {
  return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

template <int D, int G>
struct WarpAttnMma {
  static_assert(G >= 1 && G <= 8, "the heads of a group fill at most the 8 MMA columns");
  static_assert(D % 64 == 0, "head dim: a multiple of 64");
  static constexpr int S = 16;              // tokens per page
  static constexpr int KVEC = D / 32;       // K vectors per row per lane
  static constexpr int VVEC = D / 64;       // V vectors per row per lane
  static constexpr int KT = D / 16;         // k-tiles of QK; m-tiles of AV

  struct Page {
    uint4 k[2][KVEC];                       // rows gid, gid + 8
    uint4 v[4][VVEC];                       // rows 2t, 2t+1, 2t+8, 2t+9
  };

  uint4 q[KVEC];
  float m[2], l[2];                         // heads 2t, 2t+1 (base-2 logits)
  float acc[KT][4];
  float scale_log2;

  __device__ __forceinline__ void init(const __half* qrows, float sl2, int lane) {
    const int gid = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < KVEC; ++i)
      q[i] = gid < G ? *reinterpret_cast<const uint4*>(qrows + (size_t)gid * D + 32 * i + 8 * t)
                     : make_uint4(0u, 0u, 0u, 0u);
    scale_log2 = sl2;
#pragma unroll
    for (int h = 0; h < 2; ++h) { m[h] = -INFINITY; l[h] = 0.f; }
#pragma unroll
    for (int mt = 0; mt < KT; ++mt)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[mt][c] = 0.f;
  }

  // Issue the loads of one page's K and V blocks ([16][D] each).
  __device__ __forceinline__ static void load(const __half* kb, const __half* vb, int lane,
                                              uint64_t pol, Page& p) {
    const int gid = lane >> 2, t = lane & 3;
#pragma unroll
    for (int i = 0; i < KVEC; ++i) {
      p.k[0][i] = ld_cg_v4_hint(kb + (size_t)gid * D + 32 * i + 8 * t, pol);
      p.k[1][i] = ld_cg_v4_hint(kb + (size_t)(gid + 8) * D + 32 * i + 8 * t, pol);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int tok = 2 * t + (r & 1) + 8 * (r >> 1);
#pragma unroll
      for (int i = 0; i < VVEC; ++i)
        p.v[r][i] = ld_cg_v4_hint(vb + (size_t)tok * D + 64 * i + 8 * gid, pol);
    }
  }

  // Fold one page (`valid` leading tokens) into the running state. `ps` is
  // this warp's 256-byte scratch for the P tile (8 heads x 16 tokens, fp16).
  __device__ __forceinline__ void page(Page& p, int valid, float* ps, int lane) {
    const int gid = lane >> 2, t = lane & 3;
    // S^T = K Q^T
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      const int i = j >> 1, w = 2 * (j & 1);
      mma_f16_16816(s, word_of(p.k[0][i], w), word_of(p.k[1][i], w), word_of(p.k[0][i], w + 1),
                    word_of(p.k[1][i], w + 1), word_of(q[i], w), word_of(q[i], w + 1));
    }
    // tokens gid (s0: head 2t, s1: head 2t+1) and gid + 8 (s2, s3)
    const bool v0 = gid < valid, v1 = gid + 8 < valid;
    float x[4] = {v0 ? s[0] * scale_log2 : -INFINITY, v0 ? s[1] * scale_log2 : -INFINITY,
                  v1 ? s[2] * scale_log2 : -INFINITY, v1 ? s[3] * scale_log2 : -INFINITY};
    float alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mx = fmaxf(x[h], x[h + 2]);
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 16));
      const float mn = fmaxf(m[h], mx);
      alpha[h] = exp2f(m[h] - mn);
      m[h] = mn;
      // p rounded to fp16 (the MMA's input); the sum takes the rounded values
      const __half pa = __float2half_rn(exp2f(x[h] - mn));
      const __half pb = __float2half_rn(exp2f(x[h + 2] - mn));
      float sum = __half2float(pa) + __half2float(pb);
      sum += __shfl_xor_sync(FULL, sum, 4);
      sum += __shfl_xor_sync(FULL, sum, 8);
      sum += __shfl_xor_sync(FULL, sum, 16);
      l[h] = l[h] * alpha[h] + sum;
      __half* pt = reinterpret_cast<__half*>(ps);      // [8 heads][16 tokens]
      pt[(2 * t + h) * 16 + gid] = pa;
      pt[(2 * t + h) * 16 + gid + 8] = pb;
    }
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      acc[mt][0] *= alpha[0]; acc[mt][1] *= alpha[1];
      acc[mt][2] *= alpha[0]; acc[mt][3] *= alpha[1];
    }
    // B = P^T: P[head gid][tokens 2t, 2t+1] and [2t+8, 2t+9]
    const uint32_t* pw = reinterpret_cast<const uint32_t*>(ps);
    const uint32_t b0 = pw[gid * 8 + t], b1 = pw[gid * 8 + 4 + t];
    __syncwarp();                                       // scratch free for the next page
    // tokens past `valid` hold anything (a NaN times p = 0 is still NaN):
    // their V rows are zeroed
    const int tok0 = 2 * t, tok8 = 2 * t + 8;
    const uint32_t z0 = tok0 < valid ? 0xffffffffu : 0u, z1 = tok0 + 1 < valid ? 0xffffffffu : 0u;
    const uint32_t z2 = tok8 < valid ? 0xffffffffu : 0u, z3 = tok8 + 1 < valid ? 0xffffffffu : 0u;
    // O^T += V^T P^T
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      const int i = mt >> 2, w = mt & 3;
      const uint32_t r0 = word_of(p.v[0][i], w) & z0, r1 = word_of(p.v[1][i], w) & z1;
      const uint32_t r2 = word_of(p.v[2][i], w) & z2, r3 = word_of(p.v[3][i], w) & z3;
      // (V[tok][d], V[tok + 1][d]) and (V[tok][d + 1], V[tok + 1][d + 1])
      mma_f16_16816(acc[mt], __byte_perm(r0, r1, 0x5410), __byte_perm(r0, r1, 0x7632),
                    __byte_perm(r2, r3, 0x5410), __byte_perm(r2, r3, 0x7632), b0, b1);
    }
  }

  // Store this warp's state for the CTA merge: mo[w][gi][D], ml[w][gi][2].
  __device__ __forceinline__ void stash(float* mo, float* ml, int w, int lane) const {
    const int gid = lane >> 2, t = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int gi = 2 * t + h;
      if (gi >= G) continue;
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        const int d = 64 * (mt >> 2) + 8 * gid + 2 * (mt & 3);
        mo[(size_t)(w * G + gi) * D + d] = acc[mt][h];
        mo[(size_t)(w * G + gi) * D + d + 1] = acc[mt][h + 2];
      }
      if (gid == 0) {
        ml[(w * G + gi) * 2 + 0] = m[h];
        ml[(w * G + gi) * 2 + 1] = l[h];
      }
    }
  }
};

}  // namespace quest

namespace quest {

// The same attention for the G >= 4 query heads of a KV head, with the K and
// V blocks of 16-token tiles staged in shared memory in rows of D halves whose
// 16-byte units are XOR-swizzled by the row (unit u of row r at u ^ (r & 7)),
// so that ldmatrix reads eight rows without bank conflicts:
//   S^T = K Q^T   A = K tile (ldmatrix.x4), B = the group's queries
//                 (registers; head gid, the rest of the 8 columns zero)
//   O^T += V^T P^T   A = V tile transposed (ldmatrix.x4.trans), B = P^T
//                 staged through a 256-byte warp scratch
// Accumulators: acc[mt] = O^T[16 mt + gid][2t], [..][2t+1], [16 mt + gid + 8][2t], [..][2t+1].
template <int D, int G>
struct WarpAttnMmaS {
  static_assert(G >= 1 && G <= 8 && D % 64 == 0, "at most 8 heads, D a multiple of 64");
  static constexpr int KT = D / 16;         // k-steps of QK; m-tiles of AV
  static constexpr int RB = D * 2;          // bytes of a K or V row

  uint32_t qb[KT][2];                       // B fragments of Q^T
  float m[2], l[2];                         // heads 2t, 2t+1 (base-2 logits)
  float acc[KT][4];
  float scale_log2;

  __device__ __forceinline__ static int sw(int row, int unit) {
    return row * RB + (((unit ^ (row & 7)) & (RB / 16 - 1)) << 4);
  }

  __device__ __forceinline__ void init(const __half* qrows, float sl2, int lane) {
    const int gid = lane >> 2, t = lane & 3;
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      if (gid < G) {
        qb[kk][0] = *reinterpret_cast<const uint32_t*>(qrows + (size_t)gid * D + 16 * kk + 2 * t);
        qb[kk][1] = *reinterpret_cast<const uint32_t*>(qrows + (size_t)gid * D + 16 * kk + 2 * t + 8);
      } else {
        qb[kk][0] = 0u;
        qb[kk][1] = 0u;
      }
    }
    scale_log2 = sl2;
#pragma unroll
    for (int h = 0; h < 2; ++h) { m[h] = -INFINITY; l[h] = 0.f; }
#pragma unroll
    for (int mt = 0; mt < KT; ++mt)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[mt][c] = 0.f;
  }

  // One tile of 16 tokens (`valid` of them real), in two halves: qk() folds
  // the K tile (shared-memory byte address kb, swizzled rows) into the running
  // max and sum and leaves P in ps (this warp's 256-byte scratch); av() then
  // accumulates the V tile (vb). The K tile is not read after qk() returns.
  // Heads whose bit of `hmask` is clear did not choose the page: weight 0.
  __device__ __forceinline__ void qk(uint32_t kb, int valid, __half* ps, int lane, unsigned hmask = ~0u) {
    const int gid = lane >> 2, t = lane & 3;
    const int q4 = lane >> 3, r8 = lane & 7;  // ldmatrix: matrix q4, row r8 of this lane's address
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      // matrices: (tokens 0-7, dims 16kk..+7), (8-15, same), (0-7, +8..+15), (8-15, +8..+15)
      const int row = r8 + 8 * (q4 & 1), unit = 2 * kk + (q4 >> 1);
      uint32_t a0, a1, a2, a3;
      asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                   : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(kb + sw(row, unit)));
      if (kk & 1) mma_f16_16816(s1, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
      else mma_f16_16816(s0, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
    }
    // tokens gid (s: head 2t, 2t+1) and gid + 8
    const bool v0 = gid < valid, v1 = gid + 8 < valid;
    const bool ha = (hmask >> (2 * t)) & 1u, hb = (hmask >> (2 * t + 1)) & 1u;
    const float x[4] = {v0 && ha ? (s0[0] + s1[0]) * scale_log2 : -INFINITY,
                        v0 && hb ? (s0[1] + s1[1]) * scale_log2 : -INFINITY,
                        v1 && ha ? (s0[2] + s1[2]) * scale_log2 : -INFINITY,
                        v1 && hb ? (s0[3] + s1[3]) * scale_log2 : -INFINITY};
    float alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mx = fmaxf(x[h], x[h + 2]);
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 16));
      const float mn = fmaxf(m[h], mx);
      alpha[h] = mn == -INFINITY ? 1.f : exp2f(m[h] - mn);
      m[h] = mn;
      // p rounded to fp16 (the MMA's input); the sum takes the rounded values
      const __half pa = __float2half_rn(mn == -INFINITY ? 0.f : exp2f(x[h] - mn));
      const __half pb = __float2half_rn(mn == -INFINITY ? 0.f : exp2f(x[h + 2] - mn));
      float sum = __half2float(pa) + __half2float(pb);
      sum += __shfl_xor_sync(FULL, sum, 4);
      sum += __shfl_xor_sync(FULL, sum, 8);
      sum += __shfl_xor_sync(FULL, sum, 16);
      l[h] = l[h] * alpha[h] + sum;
      ps[(2 * t + h) * 16 + gid] = pa;       // P[head][token]
      ps[(2 * t + h) * 16 + gid + 8] = pb;
    }
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      acc[mt][0] *= alpha[0]; acc[mt][1] *= alpha[1];
      acc[mt][2] *= alpha[0]; acc[mt][3] *= alpha[1];
    }
    __syncwarp();
  }

  __device__ __forceinline__ void av(uint32_t vb, int valid, const __half* ps, int lane) {
    const int gid = lane >> 2, t = lane & 3;
    const int q4 = lane >> 3, r8 = lane & 7;
    // B = P^T: P[head gid][tokens 2t, 2t+1] and [2t+8, 2t+9]
    const uint32_t* pw = reinterpret_cast<const uint32_t*>(ps);
    const uint32_t b0 = pw[gid * 8 + t], b1 = pw[gid * 8 + 4 + t];
    __syncwarp();                                        // scratch free for the next tile
    // tokens past `valid` may hold anything (a NaN times p = 0 is NaN): their
    // V entries are zeroed. A = V^T: a0 (dims gid, tokens 2t, 2t+1), a1 (dims
    // gid + 8, same), a2 (dims gid, tokens 2t+8, 2t+9), a3 (dims gid + 8, same)
    const uint32_t z02 = (2 * t < valid ? 0xffffu : 0u) | (2 * t + 1 < valid ? 0xffff0000u : 0u);
    const uint32_t z13 = (2 * t + 8 < valid ? 0xffffu : 0u) | (2 * t + 9 < valid ? 0xffff0000u : 0u);
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      // matrices (transposed): (tokens 0-7, dims 16mt..+7), (tokens 0-7, +8..+15),
      // (tokens 8-15, dims 16mt..+7), (tokens 8-15, +8..+15)
      const int row = r8 + 8 * (q4 >> 1), unit = 2 * mt + (q4 & 1);
      uint32_t a0, a1, a2, a3;
      asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                   : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(vb + sw(row, unit)));
      mma_f16_16816(acc[mt], a0 & z02, a1 & z02, a2 & z13, a3 & z13, b0, b1);
    }
  }

  // Store this warp's state for the CTA merge: mo[w][gi][D], ml[w][gi][2].
  __device__ __forceinline__ void stash(float* mo, float* ml, int w, int lane) const {
    const int gid = lane >> 2, t = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int gi = 2 * t + h;
      if (gi >= G) continue;
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        mo[(size_t)(w * G + gi) * D + 16 * mt + gid] = acc[mt][h];
        mo[(size_t)(w * G + gi) * D + 16 * mt + gid + 8] = acc[mt][h + 2];
      }
      if (gid == 0) {
        ml[(w * G + gi) * 2 + 0] = m[h];
        ml[(w * G + gi) * 2 + 1] = l[h];
      }
    }
  }
};

}  // namespace quest
