// Fused GEMM epilogues of the drafter pass.
//
// Every GEMM of the path computes acc[row][col] = sum_k X[row][k] W[col][k]
// (X: activations, W: a weight matrix in [out][in] layout) and then one of the
// operations below, applied to 16-row chunks of a 128-column tile that sit in
// shared memory (buf[r][c], r < 16, c < 128).  The thread with tile column f
// (0..127) handles column f of every row of the chunk.
//
//   STORE   out[row][col] = T(acc * s(row))                     (fusion, W_proj)
//   QKV     Q/K columns rotated (RoPE at the row's block position), V plain,
//           all scaled by the row's RMS factor s(row)             (W_q|W_k|W_v)
//   RESID   x[row][col] += acc;  xn[row][col] = T(x * gain[col]); per-tile
//           sum of x^2 of the row for the next RMSNorm            (W_o, W_down)
//   SWIGLU  h[row][col/2] = T(silu(g) * u), g = even col, u = odd col, both
//           scaled by s(row)                                       (W_gate|W_up)
//   KV      columns [layer][K|V][n_kv*hd]: K rotated at the row's cache
//           position, written to that layer's cache slot           (U_K|U_V)
//   LOGITS  logits[req][j-1][col] = acc * s(row) for block rows j >= 1 (LM head);
//           logits == nullptr skips the store.  With tk_part set the GEMM also
//           folds every value into a running top-K and log-sum-exp per row and
//           publishes one record per CTA and row (gemm_tc.cu)
//   STORE_F32  logits[row][col] = acc (fp32, plain dense product)
//
// s(row) = rsqrt(sum of the row's per-tile x^2 partials / d + eps) is the
// RMSNorm factor; the norm's gain is folded into xn when the residual is
// written, so (xn . W) * s = RMSNorm(x) . W.
#pragma once

#include "common.cuh"

namespace dfl {

enum EpiKind : int {
  EPI_STORE = 0,
  EPI_QKV = 1,
  EPI_RESID = 2,
  EPI_SWIGLU = 3,
  EPI_KV = 4,
  EPI_LOGITS = 5,
  EPI_STORE_F32 = 6
};

constexpr int kTileN = 128;   // weight rows (output columns) per tile
constexpr int kChunk = 16;    // activation rows per epilogue chunk
constexpr int kBufLd = 132;   // padded row stride of the chunk buffer (floats)

struct EpiParams {
  int kind;
  int M_rows;   // activation rows
  int N_feat;   // GEMM output columns
  // RMS row scale; ssq_in == nullptr means s = 1
  const float* ssq_in;
  int ssq_parts;
  float inv_d;
  float eps;
  // STORE / QKV / SWIGLU destination (type T)
  void* out;
  long long ldo;
  // RoPE table [M_rows][head_dim/2] of (cos, sin); columns < rope_cols rotate
  const float2* rope;
  int head_dim;
  int rope_cols;
  // RESID
  float* x;           // [M_rows][N_feat] fp32, updated in place
  void* xn;           // [M_rows][N_feat] T
  const void* gain;   // [N_feat] T
  float* ssq_out;     // [N_feat/128][M_rows]
  // KV
  void* cache_k[DFLASH_MAX_LAYERS];
  void* cache_v[DFLASH_MAX_LAYERS];
  int n_kv;
  int cap;
  int n_req;
  const int* row_off;  // [n_req+1]
  const int* pos0;     // [n_req]
  // LOGITS
  float* logits;
  int L;
  // fused top-K (K <= kTkMax) of the logits rows: per-CTA records
  // [grid][n_req*(L-1)][kTkStride]; LOGITS is the chain's last phase and the
  // last CTAs to publish their records merge them into ids / log-probabilities
  // [n_req*(L-1)][K]
  float* tk_part;
  int tk_K;
  int32_t* tk_ids;
  float* tk_logp;
  // temperature sampling (tk_inv_t > 0, K <= 8): the lists rank the Gumbel
  // scores l * tk_inv_t + G of counter row tk_row0 + output row, and the merge
  // writes log q of each drawn token (see sampling.cuh)
  float tk_inv_t, tk_t;
  uint64_t tk_seed;
  long long tk_row0;
};

// Record of a fused top-K: max, sum of exp(x - max), K values (desc), K ids.
constexpr int kTkMax = 8;
constexpr int kTkStride = 2 + 2 * kTkMax;

// An approximate reciprocal (rcp.approx, within about one ulp) instead of an
// IEEE division: the epilogue's rows are short dependent chains on one warp
// per scheduler, and the division's long sequence dominated them.
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float silu_f(float g) { return g * rcp_approx(1.f + __expf(-g)); }

// Row scales of the rows [row0, row0 + n) into s_scale (s = 1 without ssq).
// A row's partial sums are split over tpr threads of one warp (tpr a power of
// two), each adding every tpr-th part with several loads in flight, then
// folded with shuffles.  Every thread of the group must call this (nthreads a
// multiple of 32).
__device__ __forceinline__ void epi_row_scales(const EpiParams& e, int row0, int n,
                                               float* s_scale, int tid, int nthreads) {
  if (e.ssq_in == nullptr) {
    for (int r = tid; r < n; r += nthreads) s_scale[r] = 1.f;
    return;
  }
  int tpr = 1;
  while (tpr < 32 && tpr * 2 * n <= nthreads) tpr *= 2;
  const int per_pass = nthreads / tpr;
  const int q = tid % tpr;
  for (int rb = 0; rb < n; rb += per_pass) {
    const int r = rb + tid / tpr;
    const int row = row0 + r;
    const bool valid = r < n && row < e.M_rows;
    float acc = 0.f;
    if (valid) {
      const float* src = e.ssq_in + row;
      int p = q;
      for (; p + 3 * tpr < e.ssq_parts; p += 4 * tpr) {
        const float v0 = src[(size_t)p * e.M_rows];
        const float v1 = src[(size_t)(p + tpr) * e.M_rows];
        const float v2 = src[(size_t)(p + 2 * tpr) * e.M_rows];
        const float v3 = src[(size_t)(p + 3 * tpr) * e.M_rows];
        acc += (v0 + v1) + (v2 + v3);
      }
      for (; p < e.ssq_parts; p += tpr) acc += src[(size_t)p * e.M_rows];
    }
    for (int off = tpr >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (r < n && q == 0) s_scale[r] = valid ? rsqrtf(acc * e.inv_d + e.eps) : 1.f;
  }
}

// Request of a global activation row (row_off is a prefix-offset array).
__device__ __forceinline__ int row_request(const int* row_off, int n_req, int row) {
  int lo = 0, hi = n_req - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (row_off[mid] <= row) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// The global inputs of one chunk's epilogue that do not depend on the
// accumulator (RESID: residual rows and gain; QKV: RoPE rotation; KV: RoPE
// rotation and cache slot).  Loading them ahead of the accumulator lets the
// loads overlap the MMAs.
struct EpiPre {
  float a[kChunk];   // RESID: x; QKV / KV: cos
  float b[kChunk];   // QKV / KV: sin
  int s[kChunk];     // KV: (request * n_kv) * cap + position, or -1 outside the slab
  float g;           // RESID: gain of the column
};

template <typename T>
__device__ __forceinline__ void epi_preload(const EpiParams& e, int col0, int crow0, int nrows,
                                            int f, EpiPre& pre) {
  const int col = col0 + f;
  const bool cvalid = col < e.N_feat;
  switch (e.kind) {
    case EPI_RESID: {
#pragma unroll
      for (int r = 0; r < kChunk; ++r)
        pre.a[r] = (r < nrows && cvalid) ? e.x[(size_t)(crow0 + r) * e.N_feat + col] : 0.f;
      pre.g = cvalid ? to_f32<T>(static_cast<const T*>(e.gain)[col]) : 0.f;
      break;
    }
    case EPI_QKV: {
      const bool rot = col < e.rope_cols;
      const int half = e.head_dim >> 1;
      const int i = col % e.head_dim;
#pragma unroll
      for (int r = 0; r < kChunk; ++r) {
        const float2 cs = (rot && r < nrows) ? e.rope[(size_t)(crow0 + r) * half + (i % half)]
                                             : make_float2(1.f, 0.f);
        pre.a[r] = cs.x;
        pre.b[r] = cs.y;
      }
      break;
    }
    case EPI_KV: {
      if (!cvalid) break;
      const int kvd = e.n_kv * e.head_dim;
      const int kind = (col / kvd) & 1;
      const int i = (col % kvd) % e.head_dim;
      const int half = e.head_dim >> 1;
      const int n_used = e.row_off[e.n_req];   // rows past it are computed, not stored
#pragma unroll
      for (int r = 0; r < kChunk; ++r) {
        const int row = crow0 + (r < nrows ? r : 0);
        const int req = row_request(e.row_off, e.n_req, row);
        const int pos = e.pos0[req] + (row - e.row_off[req]);
        const float2 cs =
            (kind == 0) ? e.rope[(size_t)row * half + (i % half)] : make_float2(1.f, 0.f);
        pre.a[r] = cs.x;
        pre.b[r] = cs.y;
        pre.s[r] = (r >= nrows || row >= n_used || pos < 0 || pos >= e.cap)
                       ? -1
                       : (req * e.n_kv) * e.cap + pos;
      }
      break;
    }
    default:
      break;
  }
}

// L2 prefetch of the global inputs of a chunk's epilogue (what epi_preload
// reads), issued long before the chunk's accumulator exists.
__device__ __forceinline__ void prefetch_l2(const void* p);
template <typename T>
__device__ __forceinline__ void epi_prefetch_inputs(const EpiParams& e, int col0, int crow0,
                                                    int nrows, int f) {
  const int col = col0 + f;
  if (col >= e.N_feat) return;
  if (e.kind == EPI_RESID) {
#pragma unroll
    for (int r = 0; r < kChunk; ++r)
      if (r < nrows) prefetch_l2(e.x + (size_t)(crow0 + r) * e.N_feat + col);
  }
}

// Touch the first destination row of a chunk ahead of its stores.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
template <typename T>
__device__ __forceinline__ void epi_touch_out(const EpiParams& e, int col0, int crow0, int f) {
  const int col = min(col0 + f, e.N_feat - 1);
  switch (e.kind) {
    case EPI_STORE:
    case EPI_QKV:
      prefetch_l2(static_cast<const T*>(e.out) + (size_t)crow0 * e.ldo + col);
      break;
    case EPI_SWIGLU:
      prefetch_l2(static_cast<const T*>(e.out) + (size_t)crow0 * e.ldo + (col >> 1));
      break;
    case EPI_RESID:
      prefetch_l2(static_cast<const T*>(e.xn) + (size_t)crow0 * e.N_feat + col);
      prefetch_l2(e.ssq_out);
      break;
    case EPI_LOGITS:
      if (e.logits) prefetch_l2(e.logits + col);
      break;
    default:
      break;
  }
}

// Apply the epilogue to one chunk: rows [crow0, crow0 + nrows) (nrows <= 16)
// of the tile whose first column is col0.  buf[r * kBufLd + c] holds acc.  `f`
// is this thread's tile column; all 128 threads of the group call this
// together (warp-uniform control flow, shuffles inside).  s_scale is indexed by
// row - srow0; s_red[warp][row - srow0] accumulates RESID sums of squares.
// pre: epi_preload of the same chunk.
template <typename T>
__device__ __forceinline__ void epi_apply_chunk(const EpiParams& e, const float* buf, int col0,
                                                int crow0, int nrows, int f,
                                                const float* s_scale, int srow0,
                                                float* s_red, int s_red_ld, int ewarp,
                                                const EpiPre& pre) {
  const int col = col0 + f;
  const bool cvalid = col < e.N_feat;
  const int lane = f & 31;
  float a[kChunk];
#pragma unroll
  for (int r = 0; r < kChunk; ++r) a[r] = (r < nrows) ? buf[r * kBufLd + f] : 0.f;
  switch (e.kind) {
    case EPI_STORE: {
#pragma unroll
      for (int r = 0; r < kChunk; ++r)
        if (r < nrows && cvalid)
          static_cast<T*>(e.out)[(size_t)(crow0 + r) * e.ldo + col] =
              from_f32<T>(a[r] * s_scale[crow0 + r - srow0]);
      break;
    }
    case EPI_STORE_F32: {
#pragma unroll
      for (int r = 0; r < kChunk; ++r)
        if (r < nrows && cvalid) e.logits[(size_t)(crow0 + r) * e.ldo + col] = a[r];
      break;
    }
    case EPI_QKV: {
      const bool rot = col < e.rope_cols;
      const int half = e.head_dim >> 1;
      const int i = col % e.head_dim;
      const int pf = (i < half) ? f + half : f - half;
#pragma unroll
      for (int r = 0; r < kChunk; ++r) {
        if (r < nrows && cvalid) {
          const float s = s_scale[crow0 + r - srow0];
          float v = a[r] * s;
          if (rot) {
            const float pv = buf[r * kBufLd + pf] * s;
            v = (i < half) ? (v * pre.a[r] - pv * pre.b[r]) : (v * pre.a[r] + pv * pre.b[r]);
          }
          static_cast<T*>(e.out)[(size_t)(crow0 + r) * e.ldo + col] = from_f32<T>(v);
        }
      }
      break;
    }
    case EPI_RESID: {
      float xv[kChunk];
#pragma unroll
      for (int r = 0; r < kChunk; ++r) xv[r] = pre.a[r];
      const float g = pre.g;
#pragma unroll
      for (int r = 0; r < kChunk; ++r) {
        if (r < nrows && cvalid) {
          const size_t idx = (size_t)(crow0 + r) * e.N_feat + col;
          xv[r] += a[r];
          e.x[idx] = xv[r];
          static_cast<T*>(e.xn)[idx] = from_f32<T>(xv[r] * g);
        }
      }
      float sq[kChunk];
#pragma unroll
      for (int r = 0; r < kChunk; ++r) sq[r] = xv[r] * xv[r];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
        for (int r = 0; r < kChunk; ++r) sq[r] += __shfl_xor_sync(0xffffffffu, sq[r], off);
      }
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < kChunk; ++r)
          if (r < nrows) s_red[ewarp * s_red_ld + (crow0 + r - srow0)] += sq[r];
      }
      break;
    }
    case EPI_SWIGLU: {
#pragma unroll
      for (int r = 0; r < kChunk; ++r) {
        const float v = a[r] * ((r < nrows) ? s_scale[crow0 + r - srow0] : 0.f);
        const float other = __shfl_xor_sync(0xffffffffu, v, 1);
        if (r < nrows && (f & 1) == 0 && cvalid)
          static_cast<T*>(e.out)[(size_t)(crow0 + r) * e.ldo + (col >> 1)] =
              from_f32<T>(silu_f(v) * other);
      }
      break;
    }
    case EPI_KV: {
      if (!cvalid) break;
      const int kvd = e.n_kv * e.head_dim;
      const int layer = col / (2 * kvd);
      const int kind = (col / kvd) & 1;
      const int c = col % kvd;
      const int head = c / e.head_dim;
      const int i = c % e.head_dim;
      const int half = e.head_dim >> 1;
      const int pf = (i < half) ? f + half : f - half;
      T* dst = static_cast<T*>(kind == 0 ? e.cache_k[layer] : e.cache_v[layer]);
#pragma unroll
      for (int r = 0; r < kChunk; ++r) {
        if (pre.s[r] < 0) continue;  // outside the slab (or past nrows)
        float v = a[r];
        if (kind == 0) {
          const float pv = buf[r * kBufLd + pf];
          v = (i < half) ? (v * pre.a[r] - pv * pre.b[r]) : (v * pre.a[r] + pv * pre.b[r]);
        }
        // ((req * n_kv + head) * cap + pos) * head_dim + i
        dst[((size_t)pre.s[r] + (size_t)head * e.cap) * e.head_dim + i] = from_f32<T>(v);
      }
      break;
    }
    case EPI_LOGITS: {
#pragma unroll
      for (int r = 0; r < kChunk; ++r) {
        const int row = crow0 + r;
        const int rq = row / e.L;
        const int j = row - rq * e.L;
        if (r < nrows && j >= 1 && cvalid && e.logits)
          e.logits[((size_t)rq * (e.L - 1) + (j - 1)) * e.N_feat + col] =
              a[r] * s_scale[row - srow0];
      }
      break;
    }
    default:
      break;
  }
}

// RESID over one 16-row chunk with four consecutive columns per thread: warp
// w takes rows w, w + 4, w + 8, w + 12 and lane l columns 4l .. 4l + 3, so the
// residual rows are read and written as float4 and each row's sum of squares
// needs one warp reduction (instead of one per row and column thread).
// Needs N_feat % 4 == 0.  pre.a[4i + j]: x of row w + 4i, column 4l + j;
// pre.b[j]: gain of column 4l + j.
template <typename T>
__device__ __forceinline__ void epi_preload_resid4(const EpiParams& e, int col0, int crow0,
                                                   int nrows, int ew, int lane, EpiPre& pre) {
  const int col = col0 + 4 * lane;
  const bool cv = col < e.N_feat;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ew + 4 * i;
    const float4 v = (r < nrows && cv)
                         ? *reinterpret_cast<const float4*>(e.x + (size_t)(crow0 + r) * e.N_feat + col)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    pre.a[4 * i + 0] = v.x;
    pre.a[4 * i + 1] = v.y;
    pre.a[4 * i + 2] = v.z;
    pre.a[4 * i + 3] = v.w;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    pre.b[j] = cv ? to_f32<T>(static_cast<const T*>(e.gain)[col + j]) : 0.f;
}

template <typename T>
__device__ __forceinline__ void epi_apply_resid4(const EpiParams& e, const float* buf, int col0,
                                                 int crow0, int nrows, int ew, int lane,
                                                 int srow0, float* s_red, int s_red_ld,
                                                 const EpiPre& pre) {
  const int col = col0 + 4 * lane;
  const bool cv = col < e.N_feat;
  float ss[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ew + 4 * i;
    const float4 a = *reinterpret_cast<const float4*>(buf + r * kBufLd + 4 * lane);
    const float x0 = pre.a[4 * i + 0] + a.x, x1 = pre.a[4 * i + 1] + a.y;
    const float x2 = pre.a[4 * i + 2] + a.z, x3 = pre.a[4 * i + 3] + a.w;
    const bool live = r < nrows && cv;
    if (live) {
      const size_t idx = (size_t)(crow0 + r) * e.N_feat + col;
      *reinterpret_cast<float4*>(e.x + idx) = make_float4(x0, x1, x2, x3);
      T* xn = static_cast<T*>(e.xn) + idx;
      if constexpr (sizeof(T) == 2) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(x0 * pre.b[0], x1 * pre.b[1]);
        __nv_bfloat162 hi = __floats2bfloat162_rn(x2 * pre.b[2], x3 * pre.b[3]);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo);
        pk.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(xn) = pk;
      } else {
        *reinterpret_cast<float4*>(xn) =
            make_float4(x0 * pre.b[0], x1 * pre.b[1], x2 * pre.b[2], x3 * pre.b[3]);
      }
    }
    ss[i] = live ? (x0 * x0 + x1 * x1) + (x2 * x2 + x3 * x3) : 0.f;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], off);
  }
  if (lane < 4) {
    float v = ss[0];
#pragma unroll
    for (int i = 1; i < 4; ++i)
      if (lane == i) v = ss[i];
    const int r = ew + 4 * lane;
    if (r < nrows) s_red[ew * s_red_ld + (crow0 + r - srow0)] += v;
  }
}

// QKV (and STORE, no rotation) over one 16-row chunk, same mapping as
// epi_apply_resid4 (warp w: rows w + 4i; lane l: columns 4l .. 4l + 3, which
// lie in one half of a head, so their RoPE partners are four consecutive
// columns too).  Needs head_dim % 8 == 0 (QKV) and N_feat % 4 == 0.
// pre.a / pre.b[4i + j]: cos / sin of row w + 4i, column 4l + j.
__device__ __forceinline__ void epi_preload_qkv4(const EpiParams& e, int col0, int crow0,
                                                 int nrows, int ew, int lane, EpiPre& pre) {
  const int col = col0 + 4 * lane;
  const bool rot = e.kind == EPI_QKV && col < e.rope_cols;
  const int half = e.head_dim >> 1;
  const int ih = (col % e.head_dim) % half;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ew + 4 * i;
    float4 c01 = make_float4(1.f, 0.f, 1.f, 0.f), c23 = c01;
    if (rot && r < nrows) {
      const float4* src = reinterpret_cast<const float4*>(e.rope + (size_t)(crow0 + r) * half + ih);
      c01 = src[0];
      c23 = src[1];
    }
    pre.a[4 * i + 0] = c01.x; pre.b[4 * i + 0] = c01.y;
    pre.a[4 * i + 1] = c01.z; pre.b[4 * i + 1] = c01.w;
    pre.a[4 * i + 2] = c23.x; pre.b[4 * i + 2] = c23.y;
    pre.a[4 * i + 3] = c23.z; pre.b[4 * i + 3] = c23.w;
  }
}

template <typename T>
__device__ __forceinline__ void epi_apply_qkv4(const EpiParams& e, const float* buf, int col0,
                                               int crow0, int nrows, int ew, int lane,
                                               const float* s_scale, int srow0,
                                               const EpiPre& pre) {
  const int col = col0 + 4 * lane;
  if (col >= e.N_feat) return;
  const bool rot = e.kind == EPI_QKV && col < e.rope_cols;
  const int half = e.head_dim >> 1;
  const bool lo = half > 0 && (col % e.head_dim) < half;
  const int pc = 4 * lane + (lo ? half : -half);   // partner columns in the tile
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ew + 4 * i;
    if (r >= nrows) continue;
    const float sc = s_scale[crow0 + r - srow0];
    const float4 a = *reinterpret_cast<const float4*>(buf + r * kBufLd + 4 * lane);
    float v[4] = {a.x * sc, a.y * sc, a.z * sc, a.w * sc};
    if (rot) {
      const float4 q = *reinterpret_cast<const float4*>(buf + r * kBufLd + pc);
      const float pv[4] = {q.x * sc, q.y * sc, q.z * sc, q.w * sc};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float c = pre.a[4 * i + j], sn = pre.b[4 * i + j];
        v[j] = lo ? (v[j] * c - pv[j] * sn) : (v[j] * c + pv[j] * sn);
      }
    }
    T* dst = static_cast<T*>(e.out) + (size_t)(crow0 + r) * e.ldo + col;
    if constexpr (sizeof(T) == 2) {
      __nv_bfloat162 p0 = __floats2bfloat162_rn(v[0], v[1]);
      __nv_bfloat162 p1 = __floats2bfloat162_rn(v[2], v[3]);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&p0);
      pk.y = *reinterpret_cast<uint32_t*>(&p1);
      *reinterpret_cast<uint2*>(dst) = pk;
    } else {
      *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
    }
  }
}

// SWIGLU over one 16-row chunk, same mapping (warp w: rows w + 4i; lane l:
// columns 4l .. 4l + 3 = gate, up, gate, up): two outputs per lane and row,
// one 4-byte store.  Needs N_feat % 4 == 0 and ldo even.
template <typename T>
__device__ __forceinline__ void epi_apply_swiglu4(const EpiParams& e, const float* buf, int col0,
                                                  int crow0, int nrows, int ew, int lane,
                                                  const float* s_scale, int srow0) {
  const int col = col0 + 4 * lane;
  if (col >= e.N_feat) return;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ew + 4 * i;
    if (r >= nrows) continue;
    const float sc = s_scale[crow0 + r - srow0];
    const float4 a = *reinterpret_cast<const float4*>(buf + r * kBufLd + 4 * lane);
    const float h0 = silu_f(a.x * sc) * (a.y * sc);
    const float h1 = silu_f(a.z * sc) * (a.w * sc);
    T* dst = static_cast<T*>(e.out) + (size_t)(crow0 + r) * e.ldo + (col >> 1);
    if constexpr (sizeof(T) == 2) {
      *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(h0, h1);
    } else {
      *reinterpret_cast<float2*>(dst) = make_float2(h0, h1);
    }
  }
}

// KV over one 16-row chunk, same mapping (warp w: rows w + 4i; lane l: columns
// 4l .. 4l + 3 of one head, one of K or V, one layer): K rotated at the row's
// cache position (partners four consecutive columns half a head away), every
// row written to its cache slot as 8 bytes per lane.  Needs head_dim % 8 ==
// 0 and n_kv * head_dim % 4 == 0.  pre.a / pre.b[4i + j]: cos / sin of row
// w + 4i, column 4l + j (K columns); pre.s[i]: (request * n_kv) * cap +
// position of row w + 4i, or -1 (outside the slab, or past the chunk).
__device__ __forceinline__ void epi_preload_kv4(const EpiParams& e, int col0, int crow0,
                                                int nrows, int ew, int lane, EpiPre& pre) {
  const int col = col0 + 4 * lane;
  const int kvd = e.n_kv * e.head_dim;
  const bool cv = col < e.N_feat;
  const bool rotk = cv && ((col / kvd) & 1) == 0;
  const int half = e.head_dim >> 1;
  const int ih = ((col % kvd) % e.head_dim) % half;
  const int n_used = e.row_off[e.n_req];   // rows past it are computed, not stored
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ew + 4 * i;
    const int row = crow0 + (r < nrows ? r : 0);
    const int req = row_request(e.row_off, e.n_req, row);
    const int pos = e.pos0[req] + (row - e.row_off[req]);
    pre.s[i] = (r >= nrows || row >= n_used || pos < 0 || pos >= e.cap)
                   ? -1
                   : (req * e.n_kv) * e.cap + pos;
    float4 c01 = make_float4(1.f, 0.f, 1.f, 0.f), c23 = c01;
    if (rotk && r < nrows) {
      const float4* src = reinterpret_cast<const float4*>(e.rope + (size_t)row * half + ih);
      c01 = src[0];
      c23 = src[1];
    }
    pre.a[4 * i + 0] = c01.x; pre.b[4 * i + 0] = c01.y;
    pre.a[4 * i + 1] = c01.z; pre.b[4 * i + 1] = c01.w;
    pre.a[4 * i + 2] = c23.x; pre.b[4 * i + 2] = c23.y;
    pre.a[4 * i + 3] = c23.z; pre.b[4 * i + 3] = c23.w;
  }
}

template <typename T>
__device__ __forceinline__ void epi_apply_kv4(const EpiParams& e, const float* buf, int col0,
                                              int nrows, int ew, int lane, const EpiPre& pre) {
  const int col = col0 + 4 * lane;
  if (col >= e.N_feat) return;
  const int kvd = e.n_kv * e.head_dim;
  const int layer = col / (2 * kvd);
  const int kind = (col / kvd) & 1;
  const int c = col % kvd;
  const int head = c / e.head_dim;
  const int i0 = c % e.head_dim;
  const int half = e.head_dim >> 1;
  const bool lo = i0 < half;
  const int pc = 4 * lane + (lo ? half : -half);   // partner columns in the tile
  T* dst = static_cast<T*>(kind == 0 ? e.cache_k[layer] : e.cache_v[layer]);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ew + 4 * i;
    if (r >= nrows || pre.s[i] < 0) continue;
    const float4 a = *reinterpret_cast<const float4*>(buf + r * kBufLd + 4 * lane);
    float v[4] = {a.x, a.y, a.z, a.w};
    if (kind == 0) {
      const float4 q = *reinterpret_cast<const float4*>(buf + r * kBufLd + pc);
      const float pv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float cs = pre.a[4 * i + j], sn = pre.b[4 * i + j];
        v[j] = lo ? (v[j] * cs - pv[j] * sn) : (v[j] * cs + pv[j] * sn);
      }
    }
    // ((req * n_kv + head) * cap + pos) * head_dim + i0
    T* d = dst + ((size_t)pre.s[i] + (size_t)head * e.cap) * e.head_dim + i0;
    if constexpr (sizeof(T) == 2) {
      __nv_bfloat162 p0 = __floats2bfloat162_rn(v[0], v[1]);
      __nv_bfloat162 p1 = __floats2bfloat162_rn(v[2], v[3]);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&p0);
      pk.y = *reinterpret_cast<uint32_t*>(&p1);
      *reinterpret_cast<uint2*>(d) = pk;
    } else {
      *reinterpret_cast<float4*>(d) = make_float4(v[0], v[1], v[2], v[3]);
    }
  }
}

// After all chunks of a RESID tile: fold the per-warp sums of squares.
__device__ __forceinline__ void epi_resid_flush(const EpiParams& e, int ftile, int row0, int n,
                                                const float* s_red, int s_red_ld, int nwarps,
                                                int tid, int nthreads) {
  for (int r = tid; r < n; r += nthreads) {
    float acc = 0.f;
    for (int w = 0; w < nwarps; ++w) acc += s_red[w * s_red_ld + r];
    e.ssq_out[(size_t)ftile * e.M_rows + row0 + r] = acc;
  }
}

}  // namespace dfl
