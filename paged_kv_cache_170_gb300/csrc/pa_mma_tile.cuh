// pa_mma_tile.cuh -- one K/V tile of decode attention on the tensor cores,
// for one warp and up to 8 query rows: the step both tensor-core decode
// kernels repeat for every tile they consume.
//
// * QK, transposed: S^T = K * Q^T with one mma.m16n8k16 per 16 tokens x 16
//   dims (M = tokens, N = the warp's <= 8 query rows, K = dims).  K fragments
//   come from ldmatrix on the 128-byte-swizzled tile; the q fragment `qf`
//   stays in registers.  Products of two 16-bit inputs are exact and summed
//   in fp32; the fp32 score is then scaled by scale*log2(e).
// * Online softmax in registers, base 2: each lane holds 2 rows x 2 tokens of
//   every 16-token sub-tile; row maxima come from 3 xor-shuffles.
// * PV, transposed: O^T += V^T * P^T (M = dims, N = rows, K = tokens), V^T
//   from ldmatrix.trans.  The accumulator layout of S^T is the transpose of
//   the operand layout P^T needs; one 8x8 movmatrix.trans per half turns one
//   into the other.  P is fed as two 16-bit terms (P = P_hi + P_lo, each
//   rounded to the input type), so the weights carry ~16 significant bits
//   and PV stays close to an fp32 product.
//
// Lane (g = lane / 4, c4 = lane % 4) owns rows h0 = 2*c4 and h1 = 2*c4 + 1:
// m0/l0 and m1/l1, and o[mt][0] (h0, dim 16mt + g), o[mt][1] (h1, 16mt + g),
// o[mt][2] (h0, 16mt + g + 8), o[mt][3] (h1, 16mt + g + 8).  l0/l1 are
// per-lane partial sums (over the lane's tokens); reduce them over g before
// use.  V rows nv .. 16*ceil(nv/16) - 1 must hold zeros (or any finite data).
#pragma once

#include <math_constants.h>

#include "pa_common.cuh"

namespace pagedkv {

// Shared-memory address of (row, 16-byte logical chunk) in a swizzled tile
// laid out as [D/64 halves][B rows][128 bytes].
__device__ __forceinline__ uint32_t swz(uint32_t tile, int B, int half, int row, int chunk) {
  return tile + uint32_t(half * B * 128 + row * 128 + ((chunk ^ (row & 7)) << 4));
}

// `a` only serves the debug-build bound checks (its err word); [lo, hi) is
// the shared-memory window the tile must lie in.
template <typename T, int D, class Args>
__device__ __forceinline__ void mma_tile(const Args &a, uint32_t kt, uint32_t vt, int B, int nv,
                                         const uint32_t (&qf)[D / 16][2], float qscale, float &m0, float &m1,
                                         float &l0, float &l1, float (&o)[D / 16][4], int lane, uint32_t lo,
                                         uint32_t hi) {
  constexpr int KS = D / 16;
  (void)a;
  (void)lo;
  (void)hi;
  const int g = lane >> 2;
  const int mj = lane >> 3;  // ldmatrix: which 8x8 matrix this lane addresses
  const int mr = lane & 7;   // ldmatrix: which row of it
  const int nsub = (nv + 15) >> 4;

  // ---- QK: scores of up to 4 sub-tiles of 16 tokens
  float sc[4][4];
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    sc[st][0] = sc[st][1] = sc[st][2] = sc[st][3] = -CUDART_INF_F;
    if (st < nsub) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      const int row = st * 16 + (mj & 1) * 8 + mr;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t af[4];
        uint32_t ad = swz(kt, B, ks >> 2, row, (ks & 3) * 2 + (mj >> 1));
        PA_DBG_FIX(ad >= lo && ad + 16 <= hi && (ad & 15u) == 0, kDbgSmem, ad = lo);
        ldmatrix_x4(af, ad);
        Mma<T>::run(c, af, qf[ks][0], qf[ks][1]);
      }
      const int t0 = st * 16 + g;
      sc[st][0] = t0 < nv ? c[0] * qscale : -CUDART_INF_F;
      sc[st][1] = t0 < nv ? c[1] * qscale : -CUDART_INF_F;
      sc[st][2] = t0 + 8 < nv ? c[2] * qscale : -CUDART_INF_F;
      sc[st][3] = t0 + 8 < nv ? c[3] * qscale : -CUDART_INF_F;
    }
  }
  // ---- online softmax (base 2), rows h0 / h1 of this lane
  float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    mx0 = fmaxf(mx0, fmaxf(sc[st][0], sc[st][2]));
    mx1 = fmaxf(mx1, fmaxf(sc[st][1], sc[st][3]));
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, off));
  }
  const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
  const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
  m0 = mn0;
  m1 = mn1;
  l0 *= al0;
  l1 *= al1;
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    sc[st][0] = fast_exp2(sc[st][0] - mn0);
    sc[st][1] = fast_exp2(sc[st][1] - mn1);
    sc[st][2] = fast_exp2(sc[st][2] - mn0);
    sc[st][3] = fast_exp2(sc[st][3] - mn1);
    l0 += sc[st][0] + sc[st][2];
    l1 += sc[st][1] + sc[st][3];
  }
  if (__any_sync(kFullMask, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      o[mt][0] *= al0;
      o[mt][1] *= al1;
      o[mt][2] *= al0;
      o[mt][3] *= al1;
    }
  }

  // ---- PV
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    if (st < nsub) {
      const uint32_t hi0 = Mma<T>::pack(sc[st][0], sc[st][1]);  // token g
      const uint32_t hi1 = Mma<T>::pack(sc[st][2], sc[st][3]);  // token g + 8
      const float2 f0 = Mma<T>::unpack(hi0), f1 = Mma<T>::unpack(hi1);
      const uint32_t lo0 = Mma<T>::pack(sc[st][0] - f0.x, sc[st][1] - f0.y);
      const uint32_t lo1 = Mma<T>::pack(sc[st][2] - f1.x, sc[st][3] - f1.y);
      const uint32_t bh0 = movmatrix_trans(hi0), bh1 = movmatrix_trans(hi1);
      const uint32_t bl0 = movmatrix_trans(lo0), bl1 = movmatrix_trans(lo1);
      const int row = st * 16 + (mj >> 1) * 8 + mr;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int chunk = 2 * mt + (mj & 1);
        uint32_t af[4];
        uint32_t ad = swz(vt, B, chunk >> 3, row, chunk & 7);
        PA_DBG_FIX(ad >= lo && ad + 16 <= hi && (ad & 15u) == 0, kDbgSmem, ad = lo);
        ldmatrix_x4_trans(af, ad);
        Mma<T>::run(o[mt], af, bh0, bh1);
        Mma<T>::run(o[mt], af, bl0, bl1);
      }
    }
  }
}

}  // namespace pagedkv
