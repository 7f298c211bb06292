// Vocabulary-wide log-softmax and top-K (step a6).
//
// "Accelerating Speculative Decoding with Block Diffusion Draft Trees",
// section 3.4.2 (q_i = softmax(l_i)) and section 3.4.4 (Lemma 1: only the
// top-K tokens of each depth are needed, ranked by descending probability).
//
// This file serves temperature sampling and 8 < K <= 32; the plain top-K
// with K <= 8 on 16-byte aligned rows takes the streamed pass of
// topk_stream.cu (launch_topk dispatches).
//
// Design (HBM-bound): each row of logits is split into `splits` contiguous
// chunks, one CTA per chunk.  A CTA streams its chunk once with 16-byte loads
// (8 bf16 or 4 fp32 per load), keeping per thread a running (max, sum of exp)
// pair and a sorted register list of its K best (value desc, id asc).  The
// 256 lists are merged by warp tournaments into the CTA's list.  With one
// split the CTA finishes the row; otherwise it writes a partial record and the
// last CTA to arrive for the row (an atomic arrival counter, no waiting)
// merges the partial records in split order and writes the result.
//
// With temperature sampling (DFlash page, 3.4.4) the lists rank Gumbel scores
// l / T + G instead of logits, so the first entry is a sample from
// softmax(l / T) and the K entries a draw without replacement; the running
// (max, sum of exp) pair still covers the logits, and the log-probability
// written for an entry is its logit (recovered from the score) minus lse.
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "sampling.cuh"
#include "topk8.cuh"

#include <math_constants.h>

namespace dfl {

namespace {

constexpr int kTopkThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

struct TopkPart {
  // [rows][splits] records of: m, s, vals[KMAX], ids[KMAX]
  float* base;
  int stride;  // floats per record = 2 + 2*KMAX
};

__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2) {
  float M = fmaxf(m, m2);
  if (M == -CUDART_INF_F) { m = M; s = 0.f; return; }
  float a = (m == -CUDART_INF_F) ? 0.f : s * exp2f((m - M) * kLog2e);
  float b = (m2 == -CUDART_INF_F) ? 0.f : s2 * exp2f((m2 - M) * kLog2e);
  m = M;
  s = a + b;
}

// (v, i) is better than (ov, oi) under (value desc, id asc).
__device__ __forceinline__ bool better(float v, int i, float ov, int oi) {
  return v > ov || (v == ov && i < oi);
}

__device__ __forceinline__ void warp_best(float& v, int& i) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, off);
    int oi = __shfl_xor_sync(0xffffffffu, i, off);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

template <int KMAX>
__device__ __forceinline__ void list_insert(float (&tv)[KMAX], int (&ti)[KMAX], int K,
                                            float x, int id, float& thr) {
#pragma unroll
  for (int j = KMAX - 1; j >= 0; --j) {
    if (j < K) {
      float pv = (j > 0) ? tv[j > 0 ? j - 1 : 0] : CUDART_INF_F;
      int pi = (j > 0) ? ti[j > 0 ? j - 1 : 0] : 0;
      if (x > pv) { tv[j] = pv; ti[j] = pi; }
      else if (x > tv[j]) { tv[j] = x; ti[j] = id; }
    }
  }
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
    if (j == K - 1) thr = tv[j];
}

template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<__nv_bfloat16> { static constexpr int N = 8; };

template <typename T, int N>
__device__ __forceinline__ void load_vec(const T* p, float (&x)[N]) {
  uint4 raw = __ldcs(reinterpret_cast<const uint4*>(p));
  if constexpr (sizeof(T) == 4) {
    x[0] = __uint_as_float(raw.x); x[1] = __uint_as_float(raw.y);
    x[2] = __uint_as_float(raw.z); x[3] = __uint_as_float(raw.w);
  } else {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __uint_as_float(w[k] << 16);
      x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
}

struct TopkSample {
  float inv_t, t;      // 1/T and T (inv_t == 0: plain top-K)
  uint64_t seed;
  long long row0;      // counter row of logits row 0
};

template <bool SAMPLE>
__device__ __forceinline__ float out_logp(float v, int id, int row, float lse,
                                          const TopkSample& smp) {
  if constexpr (SAMPLE) return sampled_logq(v, smp.t, smp.seed, smp.row0 + row, id, lse);
  else return v - lse;
}

template <typename T, int KMAX, bool VECTOR, bool SAMPLE>
__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const T* __restrict__ logits, int rows, int vocab, long long ld, int K,
            int splits, int chunk, TopkPart part, int* __restrict__ counters,
            int32_t* __restrict__ ids_out, float* __restrict__ logp_out, TopkSample smp) {
  constexpr int VN = VECTOR ? Vec<T>::N : 1;
  __shared__ float s_v[KMAX];
  __shared__ int s_i[KMAX];
  __shared__ float s_wv[kTopkThreads / kWarp][KMAX];
  __shared__ int s_wi[kTopkThreads / kWarp][KMAX];
  __shared__ float s_m[kTopkThreads / kWarp], s_s[kTopkThreads / kWarp];
  __shared__ int s_last;

  const int row = blockIdx.x / splits;
  const int split = blockIdx.x % splits;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int v0 = split * chunk;
  const int v1 = min(vocab, v0 + chunk);
  const T* rp = logits + (long long)row * ld;
  pdl_wait();
  pdl_trigger();

  float m = -CUDART_INF_F, s = 0.f, thr = -CUDART_INF_F;
  float tv[KMAX];
  int ti[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) { tv[j] = -CUDART_INF_F; ti[j] = 0x7fffffff; }

  // wthr: the largest per-lane K-th value in the warp.  That lane holds K values
  // at or above it, so anything strictly below cannot be in the row's top-K;
  // it is refreshed after every step of the warp-uniform main loop.
  float wthr = -CUDART_INF_F;
  // x: logits (for the log-sum-exp), y: the values ranked (logits or scores)
  auto consume = [&](const float* x, const float* y, int n, int id0) {
    float vmax = x[0];
#pragma unroll
    for (int e = 1; e < VN; ++e) if (e < n) vmax = fmaxf(vmax, x[e]);
    if (vmax > m) {
      s = (m == -CUDART_INF_F) ? 0.f : s * exp2f((m - vmax) * kLog2e);
      m = vmax;
    }
    if (m != -CUDART_INF_F) {
#pragma unroll
      for (int e = 0; e < VN; ++e) if (e < n) s += exp2f((x[e] - m) * kLog2e);
    }
#pragma unroll
    for (int e = 0; e < VN; ++e)
      if (e < n && y[e] > thr && y[e] >= wthr) list_insert<KMAX>(tv, ti, K, y[e], id0 + e, thr);
  };
  auto rank_values = [&](const float* x, float* y, int n, int id0) {
#pragma unroll
    for (int e = 0; e < VN; ++e) {
      if constexpr (SAMPLE)
        y[e] = (e < n && x[e] != -CUDART_INF_F)
                   ? gumbel_score(x[e], smp.inv_t, smp.seed, smp.row0 + row, id0 + e)
                   : -CUDART_INF_F;
      else
        y[e] = x[e];
    }
  };

  if (v1 > v0) {
    const int nvec = (v1 - v0) / VN;
    constexpr int U = 4;
    // warp-uniform loop: a warp step covers U*32 consecutive vectors, lane-major
    bool first = true;
    for (int kb = warp * 32 * U; kb < nvec; kb += (kTopkThreads / kWarp) * 32 * U) {
      float x[U][VN];
      bool ok[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int idx = kb + u * 32 + lane;
        ok[u] = idx < nvec;
        if (ok[u]) {
          const T* p = rp + v0 + (size_t)idx * VN;
          if constexpr (VECTOR) load_vec<T, VN>(p, x[u]);
          else x[u][0] = to_f32<T>(p[0]);
        } else {
#pragma unroll
          for (int e = 0; e < VN; ++e) x[u][e] = -CUDART_INF_F;
        }
      }
      float y[U][VN];
#pragma unroll
      for (int u = 0; u < U; ++u) rank_values(x[u], y[u], VN, v0 + (kb + u * 32 + lane) * VN);
      if (first) {
        // seed: the K-th largest of the lanes' maxima over this first step is
        // met or beaten by K distinct values, so it bounds the row's K-th value
        float lm = -CUDART_INF_F;
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int e = 0; e < VN; ++e) lm = fmaxf(lm, y[u][e]);
        float seed = -CUDART_INF_F;
        for (int r = 0; r < K; ++r) {
          const uint32_t mb = __reduce_max_sync(0xffffffffu, ordered_bits(lm));
          seed = from_ordered_bits(mb);
          const unsigned holders = __ballot_sync(0xffffffffu, ordered_bits(lm) == mb);
          if (lane == __ffs(holders) - 1) lm = -CUDART_INF_F;
        }
        wthr = seed;
        first = false;
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (ok[u]) consume(x[u], y[u], VN, v0 + (kb + u * 32 + lane) * VN);
      wthr = fmaxf(wthr, from_ordered_bits(__reduce_max_sync(0xffffffffu, ordered_bits(thr))));
    }
    const int tail0 = v0 + nvec * VN;
    if (tail0 + tid < v1) {
      float x[VN];
      x[0] = to_f32<T>(rp[tail0 + tid]);
#pragma unroll
      for (int e = 1; e < VN; ++e) x[e] = -CUDART_INF_F;
      float y[VN];
      rank_values(x, y, 1, tail0 + tid);
      consume(x, y, 1, tail0 + tid);
    }
  }

  if constexpr (KMAX == 8) {
    // ---- K <= 8: butterfly merges of the register lists ----
    tk_lane_merge(tv, ti, m, s, 1, 16);   // every lane: the warp's list
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < 8; ++q) { s_wv[warp][q] = tv[q]; s_wi[warp][q] = ti[q]; }
      s_m[warp] = m;
      s_s[warp] = s;
    }
    __syncthreads();
    if (warp != 0) return;
    constexpr int kWarps = kTopkThreads / kWarp;   // 8: lanes 0..7 take one warp each
    const bool own = lane < kWarps;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      tv[q] = own ? s_wv[own ? lane : 0][q] : -CUDART_INF_F;
      ti[q] = own ? s_wi[own ? lane : 0][q] : 0x7fffffff;
    }
    m = own ? s_m[lane] : -CUDART_INF_F;
    s = own ? s_s[lane] : 0.f;
    tk_lane_merge(tv, ti, m, s, 1, kWarps / 2);   // lanes 0..7: the CTA's list
    if (splits == 1) {
      if (lane == 0) {
        const float lse = m + logf(s);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q < K) {
            ids_out[(long long)row * K + q] = ti[q];
            logp_out[(long long)row * K + q] = out_logp<SAMPLE>(tv[q], ti[q], row, lse, smp);
          }
      }
      return;
    }
    float* rec = part.base + ((long long)row * splits + split) * part.stride;
    if (lane == 0) {
      rec[0] = m;
      rec[1] = s;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        rec[2 + q] = tv[q];
        rec[2 + KMAX + q] = __int_as_float(ti[q]);
      }
      __threadfence();
      s_last = atomicAdd(&counters[row], 1) == splits - 1;
    }
    __syncwarp();
    if (!s_last) return;
    __threadfence();
    // the last CTA of the row: lane sp takes split sp's record (splits <= 32)
    const bool has = lane < splits;
    const float* my = part.base + ((long long)row * splits + (has ? lane : 0)) * part.stride;
    m = has ? __ldcg(my) : -CUDART_INF_F;
    s = has ? __ldcg(my + 1) : 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      tv[q] = has ? __ldcg(my + 2 + q) : -CUDART_INF_F;
      ti[q] = has ? __float_as_int(__ldcg(my + 2 + KMAX + q)) : 0x7fffffff;
    }
    tk_lane_merge(tv, ti, m, s, 1, 16);
    if (lane == 0) {
      const float lse = m + logf(s);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < K) {
          ids_out[(long long)row * K + q] = ti[q];
          logp_out[(long long)row * K + q] = out_logp<SAMPLE>(tv[q], ti[q], row, lse, smp);
        }
      counters[row] = 0;
    }
  } else {
    // ---- CTA merge: (m, s) and the K best of 256 sorted lists ----
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float m2 = __shfl_xor_sync(0xffffffffu, m, off);
      float s2 = __shfl_xor_sync(0xffffffffu, s, off);
      merge_ms(m, s, m2, s2);
    }
    if (lane == 0) { s_m[warp] = m; s_s[warp] = s; }
    // warp tournament: every lane offers the head of its sorted list; the winner
    // shifts its list by one, so the head always sits in register slot 0
    for (int r = 0; r < K; ++r) {
      float bv = tv[0]; int bi = ti[0];
      warp_best(bv, bi);
      if (bv == tv[0] && bi == ti[0]) {
#pragma unroll
        for (int j = 0; j < KMAX - 1; ++j) { tv[j] = tv[j + 1]; ti[j] = ti[j + 1]; }
        tv[KMAX - 1] = -CUDART_INF_F; ti[KMAX - 1] = 0x7fffffff;
      }
      if (lane == 0) { s_wv[warp][r] = bv; s_wi[warp][r] = bi; }
    }
    __syncthreads();

    float cm = -CUDART_INF_F, cs = 0.f;
    if (warp == 0) {
      for (int w = 0; w < kTopkThreads / kWarp; ++w) merge_ms(cm, cs, s_m[w], s_s[w]);
      int p = 0;
      for (int r = 0; r < K; ++r) {
        float v = (lane < kTopkThreads / kWarp && p < K) ? s_wv[lane][p] : -CUDART_INF_F;
        int i = (lane < kTopkThreads / kWarp && p < K) ? s_wi[lane][p] : 0x7fffffff;
        float bv = v; int bi = i;
        warp_best(bv, bi);
        if (lane < kTopkThreads / kWarp && p < K && bv == v && bi == i) ++p;
        if (lane == 0) { s_v[r] = bv; s_i[r] = bi; }
        __syncwarp();
      }
    }

    if (splits == 1) {
      if (warp == 0) {
        const float lse = cm + logf(cs);
        for (int r = lane; r < K; r += 32) {
          ids_out[(long long)row * K + r] = s_i[r];
          logp_out[(long long)row * K + r] = out_logp<SAMPLE>(s_v[r], s_i[r], row, lse, smp);
        }
      }
      return;
    }

    // ---- multi-split: publish the partial record, the last CTA of the row merges ----
    float* rec = part.base + ((long long)row * splits + split) * part.stride;
    if (warp == 0) {
      if (lane == 0) { rec[0] = cm; rec[1] = cs; }
      for (int r = lane; r < K; r += 32) {
        rec[2 + r] = s_v[r];
        rec[2 + KMAX + r] = __int_as_float(s_i[r]);
      }
      __threadfence();
      __syncwarp();
      if (lane == 0) {
        int prev = atomicAdd(&counters[row], 1);
        s_last = (prev == splits - 1);
      }
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (warp != 0) return;

    const float* recs = part.base + (long long)row * splits * part.stride;
    float M = -CUDART_INF_F, S = 0.f;
    for (int sp = 0; sp < splits; ++sp)
      merge_ms(M, S, __ldcg(recs + sp * part.stride), __ldcg(recs + sp * part.stride + 1));
    const float lse = M + logf(S);
    // splits <= 32 is enforced by the launcher: one split per lane
    {
      int p = 0;
      const bool own = lane < splits;
      const float* my = recs + (own ? lane : 0) * part.stride;
      for (int r = 0; r < K; ++r) {
        float v = (own && p < K) ? __ldcg(my + 2 + p) : -CUDART_INF_F;
        int i = (own && p < K) ? __float_as_int(__ldcg(my + 2 + KMAX + p)) : 0x7fffffff;
        float bv = v; int bi = i;
        warp_best(bv, bi);
        if (own && p < K && bv == v && bi == i) ++p;
        if (lane == 0) {
          ids_out[(long long)row * K + r] = bi;
          logp_out[(long long)row * K + r] = out_logp<SAMPLE>(bv, bi, row, lse, smp);
        }
      }
    }
    if (lane == 0) counters[row] = 0;
  }
}

template <typename T, int KMAX, bool SAMPLE>
void launch_topk_t(const TopkLaunch& a, cudaStream_t st) {
  const int VN = Vec<T>::N;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(a.logits) % 16) == 0) &&
                      ((a.ld * (long long)sizeof(T)) % 16 == 0);
  int chunk = ceil_div(a.vocab, a.splits);
  chunk = ceil_div(chunk, 8) * 8;
  TopkPart part{a.part, 2 + 2 * KMAX};
  TopkSample smp{a.inv_t, a.t, a.seed, a.row0};
  dim3 grid(a.rows * a.splits);
  TraceScope ts(SAMPLE ? "lse_sample" : "lse_topk", st);
  if (vec_ok) {
    launch_k(topk_kernel<T, KMAX, true, SAMPLE>, grid, dim3(kTopkThreads), 0, st,
             static_cast<const T*>(a.logits), a.rows, a.vocab, a.ld, a.K, a.splits, chunk, part,
             a.counters, a.ids, a.logp, smp);
  } else {
    launch_k(topk_kernel<T, KMAX, false, SAMPLE>, grid, dim3(kTopkThreads), 0, st,
             static_cast<const T*>(a.logits), a.rows, a.vocab, a.ld, a.K, a.splits, chunk, part,
             a.counters, a.ids, a.logp, smp);
  }
  (void)VN;
}

}  // namespace

// Pieces per row: one row per piece once the rows fill every worker of the
// streamed pass (a warp), else as many pieces as the workers take (at most 32
// per row, each at least a few thousand logits).
int topk_splits(int rows, int vocab) {
  if (rows <= 0) return 1;
  int s = topk_stream_workers() / rows;
  s = s < 1 ? 1 : (s > 32 ? 32 : s);
  while (s > 1 && vocab / s < 4096) --s;
  return s;
}

size_t topk_part_bytes(int rows, int splits) {
  if (splits <= 1) return 0;
  return (size_t)rows * splits * (2 + 2 * 32) * sizeof(float);
}

void launch_topk(const TopkLaunch& a, cudaStream_t st) {
  if (a.rows <= 0) return;
  if (topk_stream_supported(a)) {
    launch_topk_stream(a, st);
    return;
  }
  const bool k8 = a.K <= 8;
  const bool smp = a.inv_t > 0.f;
  if (a.dtype == DFLASH_BF16) {
    if (smp) {
      if (k8) launch_topk_t<__nv_bfloat16, 8, true>(a, st);
      else launch_topk_t<__nv_bfloat16, 32, true>(a, st);
    } else {
      if (k8) launch_topk_t<__nv_bfloat16, 8, false>(a, st);
      else launch_topk_t<__nv_bfloat16, 32, false>(a, st);
    }
  } else {
    if (smp) {
      if (k8) launch_topk_t<float, 8, true>(a, st);
      else launch_topk_t<float, 32, true>(a, st);
    } else {
      if (k8) launch_topk_t<float, 8, false>(a, st);
      else launch_topk_t<float, 32, false>(a, st);
    }
  }
}

}  // namespace dfl
