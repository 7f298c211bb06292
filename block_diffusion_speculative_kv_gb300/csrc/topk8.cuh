// Merging of top-8 lists kept in registers (value desc, id asc) and of
// (max, sum of exp(x - max)) pairs, shared by the top-K passes: a merge of two
// sorted 8-lists is one bitonic step, so a warp, or any power-of-two group of
// lanes, merges its lanes' lists in log2(group) shuffle rounds.
#pragma once

#include <math_constants.h>

namespace dfl {

// (v, i) ranks above (ov, oi): value desc, then token id asc.
__device__ __forceinline__ bool tk_better(float v, int i, float ov, int oi) {
  return v > ov || (v == ov && i < oi);
}

// Merge of two (max, sum of exp(x - max)) pairs.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  s = (M == -CUDART_INF_F) ? 0.f
      : (m == -CUDART_INF_F ? 0.f : s * exp2f((m - M) * 1.4426950408889634f)) +
            (m2 == -CUDART_INF_F ? 0.f : s2 * exp2f((m2 - M) * 1.4426950408889634f));
  m = M;
}

// a := the 8 best of a and b, both sorted by (value desc, id asc).  The better
// of a[q] and b[7-q] at every q is the top half of the union as a bitonic
// sequence; three half-cleaner stages sort it.
__device__ __forceinline__ void tk_merge8(float (&a)[8], int (&ai)[8], const float (&b)[8],
                                          const int (&bi)[8]) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    if (tk_better(b[7 - q], bi[7 - q], a[q], ai[q])) { a[q] = b[7 - q]; ai[q] = bi[7 - q]; }
#pragma unroll
  for (int j = 4; j > 0; j >>= 1) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if ((q & j) == 0 && tk_better(a[q + j], ai[q + j], a[q], ai[q])) {
        const float tv = a[q];
        const int ti = ai[q];
        a[q] = a[q + j];
        ai[q] = ai[q + j];
        a[q + j] = tv;
        ai[q + j] = ti;
      }
    }
  }
}

// Butterfly over lane groups: after the offsets lo..hi (powers of two, xor),
// every lane of a group holds the group's merged list and (max, sum).
__device__ __forceinline__ void tk_lane_merge(float (&tv)[8], int (&ti)[8], float& m, float& s,
                                              int off_lo, int off_hi) {
  for (int off = off_lo; off <= off_hi; off <<= 1) {
    float ov[8];
    int oi[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      ov[q] = __shfl_xor_sync(0xffffffffu, tv[q], off);
      oi[q] = __shfl_xor_sync(0xffffffffu, ti[q], off);
    }
    lse_merge(m, s, __shfl_xor_sync(0xffffffffu, m, off), __shfl_xor_sync(0xffffffffu, s, off));
    tk_merge8(tv, ti, ov, oi);
  }
}

}  // namespace dfl
