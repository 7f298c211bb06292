// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Computes acc = X . W^T for every dense contraction of the drafter pass
// (fusion, injection, QKV, O, gate/up, down, LM head) and applies a fused
// epilogue (epilogue.cuh).  W is [N_feat][K] bf16 (a weight matrix), X is
// [M_rows][K] bf16 (activations).
//
// Mapping.  The MMA's M side (128 TMEM lanes) is a 128-row slice of W, its N
// side is a tile of n_tile activation rows (16 at batch 1, up to 256), so a
// tile of output is D[128 features][n_tile rows] in TMEM.  Work units are
// (tile, 64-wide K block) pairs; the grid is one CTA per SM and CTA c owns the
// contiguous unit range [c*U/G, (c+1)*U/G) (stream-K), so every SM streams the
// same number of weight bytes whatever the matrix shape.  A tile whose K range
// is split over several CTAs is finished by the CTA holding its first K blocks
// (they end that CTA's range, so it is among the last to get there): the
// others post fp32 partial sums and a release-add on the tile's counter, and
// it adds them, in a fixed order, to its own accumulator.  With row tiles of
// 32..256 rows (the kMulti instantiation) every contributor of a split tile
// posts its partial sums and then finishes a share of the tile's rows from all
// slots, in slot order; tiles run row-tile-major (tile t is row tile
// t / n_ftiles), so the grid's halves read each weight tile at the same time
// for different row tiles; and a phase takes a slightly smaller grid where
// that gives every CTA whole half tiles (tc_plan).
//
// Chains.  One launch runs up to kMaxPhases dependent GEMMs ("phases", e.g.
// W_o -> W_gate|up -> W_down -> next layer's W_qkv), each GEMM's activations
// being an earlier phase's output.  The activation tiles of phase k wait on a
// grid-wide counter that every CTA bumps (release) once its epilogue work for
// phase k-1 is done; the weight tiles of phase k (which depend on nothing) only
// wait for the CTA's own epilogue of phase k-1, so a CTA's weight stream starts
// as soon as it has finished its part of the previous phase, without the
// launch, TMEM allocation and pipeline fill of a new kernel.  (Streaming them
// even earlier was measured to lose: the extra traffic slows the epilogues
// that everyone waits for.)
//
// Roles (7 warps): warp 0 lane 0 loads weight tiles into a multi-stage shared
// memory ring (evict-first in L2); warp 6 lane 0 loads the matching activation
// tiles (evict-last); each producer completes its own full barrier of the stage
// (so that, when a CTA gives up, each can wait for exactly its own copies).  Warp 1 owns the
// TMEM allocation and its lane 0 issues tcgen05.mma (128 x n_tile x 16, four
// per 64-wide K block) and tcgen05.commit to release ring slots; warps 2-5
// drain TMEM (tcgen05.ld, 32 lanes each) and run the epilogue.  A CTA's tiles
// alternate between two TMEM accumulators, so the MMAs of the next tile never
// wait for the epilogue of the previous one.  Every wait (mbarrier or phase
// counter) is bounded in time (2 s, or the limit stored in the workspace
// header by dflash_workspace_set_wait_limit); on expiry the CTA records
// DFLASH_ERR_TIMEOUT in the status word, drains its outstanding copies and
// MMAs (bounded by 2 s), frees TMEM and exits.
#include <cstring>
#include <mutex>

#include <math_constants.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "gemm.h"
#include "ptx.cuh"
#include "sampling.cuh"
#include "topk8.cuh"

namespace dfl {

namespace {

constexpr int kThreads = 224;
constexpr int kEpiThreads = 128;
constexpr int kABytes = kTileN * 128;  // 128 weight rows x 64 bf16
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct TcPhase {
  int N_feat, K, n_rtiles, n_ftiles, kblocks;
  int grid;        // CTAs sharing the units: min(launch grid, total_units)
  long long total_units;
  int max_slots;
  int* counters;   // split-tile arrival counters of this phase [grid]
  EpiParams epi;
};

// Tile t of a phase: row-tile-major, so with several row tiles the CTAs of
// the grid's first and second halves stream the same weight tiles at about
// the same time for different row tiles, and the second read hits L2.
__device__ __forceinline__ void tile_coords(const TcPhase& P, long long t, int& ftile,
                                            int& rtile) {
  rtile = static_cast<int>(t / P.n_ftiles);
  ftile = static_cast<int>(t - (long long)rtile * P.n_ftiles);
}

struct TcParams {
  int M_rows, n_tile, stages, n_phases;
  int tk_kpad;     // list length of a fused top-K (0: none in this chain)
  float* part;     // split-tile partial sums [grid][max_slots][n_tile][128]
  int* sync;       // [kMaxPhases] phase-done counters, then the exit counter
  int* status;
  TcPhase ph[kMaxPhases];
};

struct TcMaps {
  CUtensorMap w[kMaxPhases];
  CUtensorMap x[kMaxPhases];
};

__host__ __device__ __forceinline__ int cta_of_unit(long long u, long long U, int G) {
  return static_cast<int>(((u + 1) * G - 1) / U);
}

struct SmemLayout {
  uint32_t a_off, b_off, bar_off, buf_off, scale_off, red_off, tk_off, total;
};

// Fused top-K state: per epilogue warp and tile row, max, sum of exp and a
// sorted list of kpad (value, id) pairs.
__host__ __device__ inline uint32_t tk_state_floats(int n_tile, int kpad) {
  return kpad ? static_cast<uint32_t>(4 * n_tile * (2 + 2 * kpad)) : 0u;
}

__host__ __device__ inline SmemLayout smem_layout(int stages, int n_tile, int tk_kpad = 0) {
  SmemLayout L;
  const uint32_t b_bytes = n_tile * 128;
  L.a_off = 0;
  L.b_off = stages * kABytes;
  L.bar_off = L.b_off + stages * b_bytes;
  const uint32_t bar_bytes = (3 * stages + 6) * 8 + 16 + 16;
  L.buf_off = (L.bar_off + bar_bytes + 15) / 16 * 16;
  L.scale_off = L.buf_off + kChunk * kBufLd * 4;
  L.red_off = L.scale_off + n_tile * 4;
  L.tk_off = L.red_off + 4 * n_tile * 4;
  L.total = L.tk_off + tk_state_floats(n_tile, tk_kpad) * 4 + 1024;  // + slack for the 1024-B base
  return L;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Release-add: everything this CTA wrote before the preceding barrier is
// visible to whoever acquires the new value.
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("fence.acq_rel.gpu;\n\tred.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v)
               : "memory");
}
// Wait until *p >= target (bounded by limit_ns; false on expiry or abort).
// The polling thread backs off between reads: a hot loop takes issue slots
// from the epilogue warp that shares its scheduler.
__device__ __forceinline__ bool wait_counter(const int* p, int target, const volatile int* abort,
                                             uint64_t limit_ns) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    __nanosleep(32);
    if (ld_acquire(p) >= target) return true;
    if (abort && *abort) return false;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// The wait limit of this launch: the workspace header's 64-bit field at byte 8
// (the status word is at byte 0); 0, or anything above a minute, means the
// default.  Only host copies write it, so it may be read before the grid
// dependency wait.
__device__ __forceinline__ uint64_t wait_limit_ns(const int* status) {
  const uint64_t v = *reinterpret_cast<const volatile uint64_t*>(status + 2);
  return (v == 0 || v > 60000000000ull) ? kTimeoutNs : v;
}


// Sort the warp's 32 (value, id) pairs into lanes 0..31 by (value desc, id asc)
// (bitonic network over shuffles).
__device__ __forceinline__ void warp_sort_desc(float& v, int& id, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, j);
      const int oi = __shfl_xor_sync(0xffffffffu, id, j);
      const bool keep_better = ((lane & j) == 0) == ((lane & k) == 0);
      if (keep_better == tk_better(ov, oi, v, id)) { v = ov; id = oi; }
    }
  }
}

// Fold one epilogue chunk of LM-head values into warp ew's per-row state
// (online max / sum of exp, and the sorted list of the K <= 8 best by value
// desc, id asc) with one lane per tile row: lane j walks the warp's 32 columns
// of chunk row j in column order with its state in registers (one exp per
// value, a register insert only when the value beats the K-th kept; a CTA
// meets its tiles in column order, so an equal value never displaces a kept
// one).
// With sampling the list ranks Gumbel scores while (max, sum) covers logits.
__device__ __forceinline__ void tk_update_rows(const EpiParams& E, float* tk, int kpad, int n_tile,
                                               const float* buf, const float* s_scale, int c0,
                                               int nr, int col0, int ew, int lane) {
  constexpr int KM = 8;
  const int K = E.tk_K;
  const int row = c0 + lane;
  if (lane >= nr || row % E.L == 0) return;
  float* st = tk + (ew * n_tile + row) * (2 + 2 * kpad);
  float m = st[0], sum = st[1];
  float tv[KM];
  int ti[KM];
#pragma unroll
  for (int q = 0; q < KM; ++q) {
    tv[q] = q < K ? st[2 + q] : -CUDART_INF_F;
    ti[q] = q < K ? __float_as_int(st[2 + kpad + q]) : 0x7fffffff;
  }
  float thr = tv[0];
#pragma unroll
  for (int q = 0; q < KM; ++q)
    if (q == K - 1) thr = tv[q];
  const float sc = s_scale[row];
  const float* src = buf + lane * kBufLd + ew * 32;
  const int ncol = min(32, E.N_feat - (col0 + ew * 32));
  const bool smp = E.tk_inv_t > 0.f;
  const long long grow = E.tk_row0 + (row / E.L * (E.L - 1) + row % E.L - 1);
  for (int q = 0; q < ncol; ++q) {
    const float l = src[q] * sc;
    if (l > m) {
      sum = (m == -CUDART_INF_F ? 0.f : sum * exp2f((m - l) * 1.4426950408889634f)) + 1.f;
      m = l;
    } else {
      sum += exp2f((l - m) * 1.4426950408889634f);
    }
    const int id = col0 + ew * 32 + q;
    const float v = smp ? gumbel_score(l, E.tk_inv_t, E.tk_seed, grow, id) : l;
    if (v > thr) {
      // sorted insert (value desc; an equal value stays ahead: it came first)
#pragma unroll
      for (int j = KM - 1; j >= 0; --j) {
        if (j < K) {
          const float pv = j > 0 ? tv[j > 0 ? j - 1 : 0] : CUDART_INF_F;
          const int pi = j > 0 ? ti[j > 0 ? j - 1 : 0] : 0;
          if (v > pv) { tv[j] = pv; ti[j] = pi; }
          else if (v > tv[j]) { tv[j] = v; ti[j] = id; }
        }
      }
#pragma unroll
      for (int q2 = 0; q2 < KM; ++q2)
        if (q2 == K - 1) thr = tv[q2];
    }
  }
  st[0] = m;
  st[1] = sum;
#pragma unroll
  for (int q = 0; q < KM; ++q)
    if (q < K) {
      st[2 + q] = tv[q];
      st[2 + kpad + q] = __int_as_float(ti[q]);
    }
}

// Final top-K of one logits row from the per-CTA records (K <= 8), by the 128
// epilogue threads of one CTA: each thread folds records etid, etid + 128, ...;
// a butterfly merges each warp; the four warps' lists (32 entries) are sorted
// across one warp.  scratch: 4 * 18 floats of shared memory.
__device__ __forceinline__ void tk_row_merge(const EpiParams& E, int n_rec, int n_out, int orow,
                                             int etid, int ew, int lane, float* scratch) {
  const int K = E.tk_K;
  float m = -CUDART_INF_F, sm = 0.f;
  float tv[8];
  int ti[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) { tv[q] = -CUDART_INF_F; ti[q] = 0x7fffffff; }
  for (int r = etid; r < n_rec; r += kEpiThreads) {
    const float* rec = E.tk_part + ((size_t)r * n_out + orow) * kTkStride;
    float v[8];
    int id[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      v[q] = q < K ? __ldcg(rec + 2 + q) : -CUDART_INF_F;
      id[q] = q < K ? __float_as_int(__ldcg(rec + 2 + kTkMax + q)) : 0x7fffffff;
    }
    lse_merge(m, sm, __ldcg(rec), __ldcg(rec + 1));
    tk_merge8(tv, ti, v, id);
  }
  tk_lane_merge(tv, ti, m, sm, 1, 16);
  if (lane == 0) {
    float* o = scratch + ew * 18;
    o[0] = m;
    o[1] = sm;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      o[2 + q] = tv[q];
      o[10 + q] = __int_as_float(ti[q]);
    }
  }
  ptx::named_bar_sync(1, kEpiThreads);
  if (ew == 0) {
    const float* o = scratch + (lane >> 3) * 18;
    float v = o[2 + (lane & 7)];
    int id = __float_as_int(o[10 + (lane & 7)]);
    warp_sort_desc(v, id, lane);
    float M = -CUDART_INF_F, S = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) lse_merge(M, S, scratch[w * 18], scratch[w * 18 + 1]);
    const float lse = M + logf(S);
    if (lane < K) {
      E.tk_ids[(size_t)orow * K + lane] = id;
      E.tk_logp[(size_t)orow * K + lane] =
          E.tk_inv_t > 0.f ? sampled_logq(v, E.tk_t, E.tk_seed, E.tk_row0 + orow, id, lse)
                           : v - lse;
    }
  }
  ptx::named_bar_sync(1, kEpiThreads);
}

// Lane r of the warp gets the sum over the 32 lanes of v[r] (a butterfly that
// halves the values each lane keeps at every step: 31 shuffles for 32 sums).
__device__ __forceinline__ float warp_transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? v[i] : v[i + w];
      const float keep = upper ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

// Eight floats of a staged row as eight bf16 (16 bytes).
__device__ __forceinline__ uint4 pack8_bf16(const float* src) {
  const float4 a = *reinterpret_cast<const float4*>(src);
  const float4 b = *reinterpret_cast<const float4*>(src + 4);
  __nv_bfloat162 h[4] = {__floats2bfloat162_rn(a.x, a.y), __floats2bfloat162_rn(a.z, a.w),
                         __floats2bfloat162_rn(b.x, b.y), __floats2bfloat162_rn(b.z, b.w)};
  return *reinterpret_cast<const uint4*>(h);
}

// Write back rows [crow0, crow0 + nr) of a 128-column tile staged in buf
// (buf[r * kBufLd + c]: the value of tile column c; SWIGLU: output column c of
// the tile's 64).  16-byte segments when the destination's rows and the tile
// allow it (bf16 outputs, 16-byte aligned rows, N_feat % 8 == 0), else one
// element per thread and step.  All epilogue threads call it.
template <typename T>
__device__ __forceinline__ void epi_copy_out(const EpiParams& E, const float* buf, int col0,
                                             int crow0, int nr, int etid) {
  static_assert(sizeof(T) == 2, "the tensor-core GEMM runs bf16");
  const bool v16 = (E.N_feat & 7) == 0;
  switch (E.kind) {
    case EPI_STORE:
    case EPI_QKV: {
      T* out = static_cast<T*>(E.out);
      if (v16 && (E.ldo & 7) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
        for (int i = etid; i < nr * 16; i += kEpiThreads) {
          const int r = i >> 4, c = (i & 15) * 8;
          if (col0 + c < E.N_feat)
            *reinterpret_cast<uint4*>(out + (size_t)(crow0 + r) * E.ldo + col0 + c) =
                pack8_bf16(buf + r * kBufLd + c);
        }
      } else {
        for (int i = etid; i < nr * kTileN; i += kEpiThreads) {
          const int r = i >> 7, c = i & 127;
          if (col0 + c < E.N_feat)
            out[(size_t)(crow0 + r) * E.ldo + col0 + c] = from_f32<T>(buf[r * kBufLd + c]);
        }
      }
      break;
    }
    case EPI_KV: {
      // row r of the batch goes to cache slot (request, head, pos) of its
      // columns' layer and kind: 8 columns (16 bytes) at a time
      const int kvd = E.n_kv * E.head_dim;
      const int n_used = E.row_off[E.n_req];   // rows past it are computed, not stored
      const bool v8 = (E.head_dim & 7) == 0;
      for (int i = etid; i < nr * 16; i += kEpiThreads) {
        const int r = i >> 4, c = (i & 15) * 8;
        const int row = crow0 + r;
        if (col0 + c >= E.N_feat || row >= n_used) continue;
        const int req = row_request(E.row_off, E.n_req, row);
        const int pos = E.pos0[req] + (row - E.row_off[req]);
        if (pos < 0 || pos >= E.cap) continue;
        for (int e = 0; e < 8; e += v8 ? 8 : 1) {
          const int col = col0 + c + e;
          if (col >= E.N_feat) break;
          const int layer = col / (2 * kvd), kind = (col / kvd) & 1, cc = col % kvd;
          T* dst = static_cast<T*>(kind == 0 ? E.cache_k[layer] : E.cache_v[layer]) +
                   (((size_t)req * E.n_kv + cc / E.head_dim) * E.cap + pos) * E.head_dim +
                   cc % E.head_dim;
          if (v8 && col + 8 <= E.N_feat && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
            *reinterpret_cast<uint4*>(dst) = pack8_bf16(buf + r * kBufLd + c);
          } else {
            const int ne = v8 ? 8 : 1;
            for (int q = 0; q < ne && col + q < E.N_feat; ++q)
              dst[q] = from_f32<T>(buf[r * kBufLd + c + e + q]);
          }
        }
      }
      break;
    }
    case EPI_SWIGLU: {
      T* out = static_cast<T*>(E.out);
      const int oc0 = col0 >> 1;
      const int n_out = E.N_feat >> 1;
      if (v16 && (E.ldo & 7) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
        for (int i = etid; i < nr * 8; i += kEpiThreads) {
          const int r = i >> 3, c = (i & 7) * 8;
          if (oc0 + c < n_out)
            *reinterpret_cast<uint4*>(out + (size_t)(crow0 + r) * E.ldo + oc0 + c) =
                pack8_bf16(buf + r * kBufLd + c);
        }
      } else {
        for (int i = etid; i < nr * (kTileN / 2); i += kEpiThreads) {
          const int r = i >> 6, c = i & 63;
          if (oc0 + c < n_out)
            out[(size_t)(crow0 + r) * E.ldo + oc0 + c] = from_f32<T>(buf[r * kBufLd + c]);
        }
      }
      break;
    }
    case EPI_RESID: {
      T* xn = static_cast<T*>(E.xn);
      const T* gain = static_cast<const T*>(E.gain);
      const bool vec = v16 && (reinterpret_cast<uintptr_t>(E.x) & 15) == 0 &&
                       (reinterpret_cast<uintptr_t>(xn) & 15) == 0 &&
                       (reinterpret_cast<uintptr_t>(gain) & 15) == 0;
      if (vec) {
        for (int i = etid; i < nr * 32; i += kEpiThreads) {
          const int r = i >> 5, c = (i & 31) * 4;
          if (col0 + c < E.N_feat)
            *reinterpret_cast<float4*>(E.x + (size_t)(crow0 + r) * E.N_feat + col0 + c) =
                *reinterpret_cast<const float4*>(buf + r * kBufLd + c);
        }
        for (int i = etid; i < nr * 16; i += kEpiThreads) {
          const int r = i >> 4, c = (i & 15) * 8;
          if (col0 + c >= E.N_feat) continue;
          const uint4 gw = __ldg(reinterpret_cast<const uint4*>(gain + col0 + c));
          const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gw);
          float v[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 gf = __bfloat1622float2(g2[q]);
            v[2 * q] = buf[r * kBufLd + c + 2 * q] * gf.x;
            v[2 * q + 1] = buf[r * kBufLd + c + 2 * q + 1] * gf.y;
          }
          *reinterpret_cast<uint4*>(xn + (size_t)(crow0 + r) * E.N_feat + col0 + c) = pack8_bf16(v);
        }
      } else {
        for (int i = etid; i < nr * kTileN; i += kEpiThreads) {
          const int r = i >> 7, c = i & 127;
          if (col0 + c >= E.N_feat) continue;
          const size_t idx = (size_t)(crow0 + r) * E.N_feat + col0 + c;
          const float xv = buf[r * kBufLd + c];
          E.x[idx] = xv;
          xn[idx] = from_f32<T>(xv * to_f32<T>(gain[col0 + c]));
        }
      }
      break;
    }
    case EPI_LOGITS: {
      if (E.logits == nullptr) break;
      const bool vec = (E.N_feat & 3) == 0 && (reinterpret_cast<uintptr_t>(E.logits) & 15) == 0;
      for (int i = etid; i < nr * (vec ? 32 : kTileN); i += kEpiThreads) {
        const int r = vec ? (i >> 5) : (i >> 7);
        const int c = vec ? (i & 31) * 4 : (i & 127);
        const int row = crow0 + r;
        const int rq = row / E.L;
        const int j = row - rq * E.L;
        if (j < 1 || col0 + c >= E.N_feat) continue;
        float* dst = E.logits + ((size_t)rq * (E.L - 1) + (j - 1)) * E.N_feat + col0 + c;
        if (vec) *reinterpret_cast<float4*>(dst) = *reinterpret_cast<const float4*>(buf + r * kBufLd + c);
        else *dst = buf[r * kBufLd + c];
      }
      break;
    }
    default: {   // EPI_STORE_F32
      const bool vec = (E.N_feat & 3) == 0 && (E.ldo & 3) == 0 &&
                       (reinterpret_cast<uintptr_t>(E.logits) & 15) == 0;
      for (int i = etid; i < nr * (vec ? 32 : kTileN); i += kEpiThreads) {
        const int r = vec ? (i >> 5) : (i >> 7);
        const int c = vec ? (i & 31) * 4 : (i & 127);
        if (col0 + c >= E.N_feat) continue;
        float* dst = E.logits + (size_t)(crow0 + r) * E.ldo + col0 + c;
        if (vec) *reinterpret_cast<float4*>(dst) = *reinterpret_cast<const float4*>(buf + r * kBufLd + c);
        else *dst = buf[r * kBufLd + c];
      }
      break;
    }
  }
}

// Epilogue of rows [rs0, rs1) of a tile with more than one 16-row chunk (row
// tiles of 32..256 activation rows), 16 rows at a time: each thread keeps its
// tile column f, and every global load a batch needs (up to three partial-sum
// slots, residual rows, RoPE factors) is issued before any is used, so a batch
// costs one memory round trip (the chunk path takes one per input, after a
// shared-memory transpose).  The sum is slot 0 + slot 1 + ... in that order
// (deterministic): slot 0 from TMEM when `tmem` (a tile this CTA owns alone),
// else every slot from the partial-sum buffer.  STORE, STORE_F32, QKV, RESID,
// SWIGLU, KV and LOGITS without a fused top-K.
template <typename T>
__device__ __forceinline__ void epi_tile_batched(const EpiParams& E, bool tmem, uint32_t tacc,
                                                 int col0, int row0, int rs0, int rs1,
                                                 int n_tile, const float* slots, int nslots,
                                                 const float* s_scale, int srow0, float* s_red,
                                                 float* buf, int f, int ew, int lane) {
  constexpr int RB = kChunk;
  const int col = col0 + f;
  const bool cvalid = col < E.N_feat;
  const int half = E.head_dim >> 1;
  const float gain =
      (E.kind == EPI_RESID && cvalid) ? to_f32<T>(static_cast<const T*>(E.gain)[col]) : 0.f;
  // RoPE columns: the rotated part of Q and K (QKV), the K part (KV)
  const bool rot = (E.kind == EPI_QKV && col < E.rope_cols) ||
                   (E.kind == EPI_KV && cvalid && ((col / (E.n_kv * E.head_dim)) & 1) == 0);
  const int ihalf = rot ? (col % E.head_dim) % half : 0;
  // the row scales and the zeroed sums of squares are written by all threads
  ptx::named_bar_sync(1, kEpiThreads);
  for (int rb = rs0; rb < rs1; rb += RB) {
    const int nr = min(RB, rs1 - rb);
    float acc[RB], v0[RB], v1[RB], in_a[RB], in_b[RB];
    // slot 0 (unless it is the TMEM accumulator), slot 1 and slot 2 at once
    const float* pb = slots + (size_t)rb * kTileN + f;
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      if (!tmem) acc[r] = r < nr ? __ldcg(pb + (size_t)r * kTileN) : 0.f;
      v0[r] = (nslots > 1 && r < nr) ? __ldcg(pb + (size_t)(n_tile + r) * kTileN) : 0.f;
      v1[r] = (nslots > 2 && r < nr) ? __ldcg(pb + (size_t)(2 * n_tile + r) * kTileN) : 0.f;
    }
    if (E.kind == EPI_RESID) {
#pragma unroll
      for (int r = 0; r < RB; ++r)
        in_a[r] = (r < nr && cvalid) ? __ldcg(E.x + (size_t)(row0 + rb + r) * E.N_feat + col) : 0.f;
    } else if (rot) {
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        const float2 cs = r < nr ? __ldg(E.rope + (size_t)(row0 + rb + r) * half + ihalf)
                                 : make_float2(1.f, 0.f);
        in_a[r] = cs.x;
        in_b[r] = cs.y;
      }
    }
    if (tmem) {
      __syncwarp();
      ptx::tmem_ld_32x16(tacc + static_cast<uint32_t>(rb), acc);
    }
#pragma unroll
    for (int r = 0; r < RB; ++r) acc[r] += v0[r];
#pragma unroll
    for (int r = 0; r < RB; ++r) acc[r] += v1[r];
    // (more than three contributors: the rest in order, one slot at a time)
    for (int s = 3; s < nslots; ++s) {
      const float* ps = slots + ((size_t)s * n_tile + rb) * kTileN + f;
#pragma unroll
      for (int r = 0; r < RB; ++r) v0[r] = r < nr ? __ldcg(ps + (size_t)r * kTileN) : 0.f;
#pragma unroll
      for (int r = 0; r < RB; ++r) acc[r] += v0[r];
    }
    // the batch's values of column f
    float val[RB];
    switch (E.kind) {
      case EPI_STORE:
      case EPI_LOGITS:
#pragma unroll
        for (int r = 0; r < RB; ++r) val[r] = acc[r] * (r < nr ? s_scale[row0 + rb + r - srow0] : 0.f);
        break;
      case EPI_SWIGLU:
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          const float v = acc[r] * (r < nr ? s_scale[row0 + rb + r - srow0] : 0.f);
          const float other = __shfl_xor_sync(0xffffffffu, v, 1);
          val[r] = silu_f(v) * other;   // (meaningful on even columns)
        }
        break;
      case EPI_RESID: {
        float sq[32];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          val[r] = in_a[r] + acc[r];
          sq[r] = (r < nr && cvalid) ? val[r] * val[r] : 0.f;
          sq[r + RB] = 0.f;
        }
        const float rs = warp_transpose_sum32(sq, lane);
        if (lane < nr) s_red[ew * n_tile + (row0 + rb + lane - srow0)] += rs;
        break;
      }
      case EPI_QKV: {
        // the RoPE partner column (f +- head_dim / 2) belongs to another warp:
        // exchange through the chunk buffer
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          acc[r] *= r < nr ? s_scale[row0 + rb + r - srow0] : 0.f;
          buf[r * kBufLd + f] = acc[r];
        }
        ptx::named_bar_sync(1, kEpiThreads);
        const int i = col % E.head_dim;
        const int pf = (i < half) ? f + half : f - half;
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          val[r] = acc[r];
          if (rot) {
            const float pv = buf[r * kBufLd + pf];
            val[r] = (i < half) ? (acc[r] * in_a[r] - pv * in_b[r]) : (acc[r] * in_a[r] + pv * in_b[r]);
          }
        }
        ptx::named_bar_sync(1, kEpiThreads);
        break;
      }
      case EPI_KV: {
        // K columns rotate with their partner column (another warp's)
#pragma unroll
        for (int r = 0; r < RB; ++r) buf[r * kBufLd + f] = acc[r];
        ptx::named_bar_sync(1, kEpiThreads);
        const int i = col % E.head_dim;
        const int pf = (i < half) ? f + half : f - half;
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          val[r] = acc[r];
          if (rot) {
            const float pv = buf[r * kBufLd + pf];
            val[r] = (i < half) ? (acc[r] * in_a[r] - pv * in_b[r]) : (acc[r] * in_a[r] + pv * in_b[r]);
          }
        }
        ptx::named_bar_sync(1, kEpiThreads);
        break;
      }
      default:   // EPI_STORE_F32
#pragma unroll
        for (int r = 0; r < RB; ++r) val[r] = acc[r];
        break;
    }
    // Stage the batch row-major in the chunk buffer and write it back as
    // 16-byte row segments: a thread's own column would take one store per
    // row of 2-4 bytes per lane, and those scattered stores, not the loads,
    // bounded this epilogue.
    if (E.kind == EPI_SWIGLU) {
      if ((f & 1) == 0) {
#pragma unroll
        for (int r = 0; r < RB; ++r) buf[r * kBufLd + (f >> 1)] = val[r];
      }
    } else {
#pragma unroll
      for (int r = 0; r < RB; ++r) buf[r * kBufLd + f] = val[r];
    }
    ptx::named_bar_sync(1, kEpiThreads);
    const int etid = (ew << 5) | lane;
    epi_copy_out<T>(E, buf, col0, row0 + rb, nr, etid);
    ptx::named_bar_sync(1, kEpiThreads);
  }
  // every warp's sums of squares are in s_red (read by the flush that follows)
  ptx::named_bar_sync(1, kEpiThreads);
}

// Share [rs0, rs1) of a split tile finished from shared memory (second pass
// of the shared split-tile epilogue).  When a CTA gets here its MMAs are done
// and neither producer writes the ring before this CTA publishes the phase, so
// the ring holds the inputs: one bulk copy per partial-sum slot (a share's
// rows are contiguous in a slot) plus the residual rows (RESID) or RoPE rows
// (QKV), all landing on sbar.  Then warp w takes rows w, w + 4, ... and lane l
// columns 4l .. 4l + 3: slots summed in slot order, the epilogue applied, and
// each row written as one contiguous segment per warp.  Returns false (status
// set) if the copies did not land in time.  Needs N_feat % 128 == 0 and the
// inputs within ring_bytes (the caller checks).
template <typename T>
__device__ __forceinline__ bool epi_share_smem(const EpiParams& E, uint8_t* ring, uint64_t* sbar,
                                               uint32_t& sphase, const float* slots, int nslots,
                                               int n_tile, int col0, int row0, int rs0, int rs1,
                                               int ftile, const float* s_scale, int ew, int lane,
                                               uint64_t lim, volatile int* flags, int* status) {
  const int R = rs1 - rs0;
  const int half = E.head_dim >> 1;
  const bool has_x = E.kind == EPI_RESID;
  // rotated tiles: Q and K of QKV; K of KV (a tile lies in one kind: the
  // caller checks that n_kv * head_dim is a multiple of the tile width)
  const bool trot = (E.kind == EPI_QKV && col0 < E.rope_cols) ||
                    (E.kind == EPI_KV && ((col0 / (E.n_kv * E.head_dim)) & 1) == 0);
  const uint32_t seg = static_cast<uint32_t>(R) * kTileN * 4;
  const uint32_t in_bytes = has_x ? seg : trot ? static_cast<uint32_t>(R * half * 8) : 0u;
  float* sl = reinterpret_cast<float*>(ring);
  float* sin_ = sl + (size_t)nslots * R * kTileN;
  if (ew == 0) {
    // the slots and residual rows were written with ordinary stores by other
    // CTAs (acquired before this call); the copies read them through the async proxy
    asm volatile("fence.proxy.async.global;" ::: "memory");
    if (lane == 0) ptx::mbar_arrive_expect_tx(sbar, nslots * seg + in_bytes);
    __syncwarp();
    const uint64_t pol = ptx::policy_evict_first();
    if (lane < nslots)
      ptx::bulk_load(sl + (size_t)lane * R * kTileN, slots + ((size_t)lane * n_tile + rs0) * kTileN,
                     seg, sbar, pol);
    if (has_x)
      for (int r = lane; r < R; r += 32)
        ptx::bulk_load(sin_ + (size_t)r * kTileN, E.x + (size_t)(row0 + rs0 + r) * E.N_feat + col0,
                       kTileN * 4, sbar, pol);
    if (trot && lane == 0)
      ptx::bulk_load(sin_, E.rope + (size_t)(row0 + rs0) * half, in_bytes, sbar, pol);
  }
  const bool ok = ptx::mbar_wait_bounded(sbar, sphase, lim, flags);
  if (ptx::named_bar_or(1, kEpiThreads, !ok)) {
    if (threadIdx.x == 64) {
      record_status(status, DFLASH_ERR_TIMEOUT);
      flags[0] = 1;
      // the copies must land before the CTA exits
      ptx::mbar_wait_bounded(sbar, sphase, kTimeoutNs, nullptr);
    }
    return false;
  }
  sphase ^= 1u;
  const int c4 = 4 * lane;
  const int col = col0 + c4;
  float4 g4 = make_float4(0.f, 0.f, 0.f, 0.f);
  if (has_x) {
    const uint2 gw = __ldg(reinterpret_cast<const uint2*>(static_cast<const T*>(E.gain) + col));
    const float2 ga = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw.x));
    const float2 gb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw.y));
    g4 = make_float4(ga.x, ga.y, gb.x, gb.y);
  }
  const int ih = (col % E.head_dim) % (half > 0 ? half : 1);
  const bool lo = half > 0 && (col % E.head_dim) < half;
  auto st4 = [&](T* dst, float a, float b, float c, float d) {
    const __nv_bfloat162 p0 = __floats2bfloat162_rn(a, b), p1 = __floats2bfloat162_rn(c, d);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&p0);
    w.y = *reinterpret_cast<const uint32_t*>(&p1);
    *reinterpret_cast<uint2*>(dst) = w;
  };
  // Four rows per warp and step (r, r + 4, r + 8, r + 12): independent chains,
  // so a warp has several rows' loads, math and stores in flight.
  constexpr int RQ = 4;
  for (int r0 = ew; r0 < R; r0 += 4 * RQ) {
    float4 a[RQ];
    float sc[RQ];
#pragma unroll
    for (int q = 0; q < RQ; ++q) {
      const int r = min(r0 + 4 * q, R - 1);
      a[q] = *reinterpret_cast<const float4*>(sl + (size_t)r * kTileN + c4);
      sc[q] = s_scale[rs0 + r];
    }
    for (int sidx = 1; sidx < nslots; ++sidx) {
#pragma unroll
      for (int q = 0; q < RQ; ++q) {
        const int r = min(r0 + 4 * q, R - 1);
        const float4 b =
            *reinterpret_cast<const float4*>(sl + ((size_t)sidx * R + r) * kTileN + c4);
        a[q].x += b.x; a[q].y += b.y; a[q].z += b.z; a[q].w += b.w;
      }
    }
    switch (E.kind) {
      case EPI_STORE:
#pragma unroll
        for (int q = 0; q < RQ; ++q)
          if (r0 + 4 * q < R)
            st4(static_cast<T*>(E.out) + (size_t)(row0 + rs0 + r0 + 4 * q) * E.ldo + col,
                a[q].x * sc[q], a[q].y * sc[q], a[q].z * sc[q], a[q].w * sc[q]);
        break;
      case EPI_STORE_F32:
#pragma unroll
        for (int q = 0; q < RQ; ++q)
          if (r0 + 4 * q < R)
            *reinterpret_cast<float4*>(E.logits + (size_t)(row0 + rs0 + r0 + 4 * q) * E.ldo + col) =
                a[q];
        break;
      case EPI_LOGITS: {
        if (E.logits == nullptr) break;
#pragma unroll
        for (int q = 0; q < RQ; ++q) {
          const int row = row0 + rs0 + r0 + 4 * q;
          const int rq = row / E.L;
          const int j = row - rq * E.L;
          if (r0 + 4 * q < R && j >= 1)
            *reinterpret_cast<float4*>(E.logits + ((size_t)rq * (E.L - 1) + (j - 1)) * E.N_feat +
                                       col) =
                make_float4(a[q].x * sc[q], a[q].y * sc[q], a[q].z * sc[q], a[q].w * sc[q]);
        }
        break;
      }
      case EPI_SWIGLU: {
        // columns (gate, up, gate, up): two outputs per row
#pragma unroll
        for (int q = 0; q < RQ; ++q) {
          const float g0 = a[q].x * sc[q], u0 = a[q].y * sc[q];
          const float g1 = a[q].z * sc[q], u1 = a[q].w * sc[q];
          const __nv_bfloat162 h = __floats2bfloat162_rn(silu_f(g0) * u0, silu_f(g1) * u1);
          if (r0 + 4 * q < R)
            *reinterpret_cast<__nv_bfloat162*>(static_cast<T*>(E.out) +
                                               (size_t)(row0 + rs0 + r0 + 4 * q) * E.ldo +
                                               (col >> 1)) = h;
        }
        break;
      }
      case EPI_RESID: {
        float ss[RQ];
#pragma unroll
        for (int q = 0; q < RQ; ++q) {
          const int r = min(r0 + 4 * q, R - 1);
          const float4 xi = *reinterpret_cast<const float4*>(sin_ + (size_t)r * kTileN + c4);
          const float4 x = make_float4(xi.x + a[q].x, xi.y + a[q].y, xi.z + a[q].z, xi.w + a[q].w);
          if (r0 + 4 * q < R) {
            const size_t idx = (size_t)(row0 + rs0 + r) * E.N_feat + col;
            *reinterpret_cast<float4*>(E.x + idx) = x;
            st4(static_cast<T*>(E.xn) + idx, x.x * g4.x, x.y * g4.y, x.z * g4.z, x.w * g4.w);
          }
          ss[q] = (x.x * x.x + x.y * x.y) + (x.z * x.z + x.w * x.w);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
          for (int q = 0; q < RQ; ++q) ss[q] += __shfl_xor_sync(0xffffffffu, ss[q], off);
        }
        if (lane < RQ) {
          float v = ss[0];
#pragma unroll
          for (int q = 1; q < RQ; ++q)
            if (lane == q) v = ss[q];
          if (r0 + 4 * lane < R)
            E.ssq_out[(size_t)ftile * E.M_rows + row0 + rs0 + r0 + 4 * lane] = v;
        }
        break;
      }
      case EPI_QKV: {
        // the partner columns (col +- head_dim / 2) sit half / 4 lanes away
        const int pl = half >> 2;
#pragma unroll
        for (int q = 0; q < RQ; ++q) {
          const int r = min(r0 + 4 * q, R - 1);
          float v[4] = {a[q].x * sc[q], a[q].y * sc[q], a[q].z * sc[q], a[q].w * sc[q]};
          if (trot) {
            const float* cs = sin_ + ((size_t)r * half + ih) * 2;
            float pv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) pv[e] = __shfl_xor_sync(0xffffffffu, v[e], pl);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float c = cs[2 * e], sn = cs[2 * e + 1];
              v[e] = lo ? (v[e] * c - pv[e] * sn) : (v[e] * c + pv[e] * sn);
            }
          }
          if (r0 + 4 * q < R)
            st4(static_cast<T*>(E.out) + (size_t)(row0 + rs0 + r) * E.ldo + col, v[0], v[1],
                v[2], v[3]);
        }
        break;
      }
      case EPI_KV: {
        // as QKV without the row scale, each row to its request's cache slot
        const int kvd = E.n_kv * E.head_dim;
        const int layer = col / (2 * kvd), cc = col % kvd;
        const int head = cc / E.head_dim, ii = cc % E.head_dim;
        T* cache = static_cast<T*>(trot ? E.cache_k[layer] : E.cache_v[layer]);
        const int n_used = E.row_off[E.n_req];   // rows past it are computed, not stored
        const int pl = half >> 2;
#pragma unroll
        for (int q = 0; q < RQ; ++q) {
          const int r = min(r0 + 4 * q, R - 1);
          float v[4] = {a[q].x, a[q].y, a[q].z, a[q].w};
          if (trot) {
            const float* cs = sin_ + ((size_t)r * half + ih) * 2;
            float pv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) pv[e] = __shfl_xor_sync(0xffffffffu, v[e], pl);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float c = cs[2 * e], sn = cs[2 * e + 1];
              v[e] = lo ? (v[e] * c - pv[e] * sn) : (v[e] * c + pv[e] * sn);
            }
          }
          const int row = row0 + rs0 + r;
          if (r0 + 4 * q < R && row < n_used) {
            const int req = row_request(E.row_off, E.n_req, row);
            const int pos = E.pos0[req] + (row - E.row_off[req]);
            if (pos >= 0 && pos < E.cap) {
              T* dst = cache + (((size_t)req * E.n_kv + head) * E.cap + pos) * E.head_dim + ii;
              if ((reinterpret_cast<uintptr_t>(dst) & 7) == 0) {
                st4(dst, v[0], v[1], v[2], v[3]);
              } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) dst[e] = from_f32<T>(v[e]);
              }
            }
          }
        }
        break;
      }
      default:
        break;
    }
  }
  // the ring's next writer is the async proxy (the next phase's copies)
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  ptx::named_bar_sync(1, kEpiThreads);
  return true;
}

// kMulti: row tiles of 32..256 rows (several 16-row chunks per tile); else
// one 16-row chunk per tile.  Two instantiations keep each path's registers
// and code apart.
template <typename T, bool kMulti>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ TcMaps maps, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const SmemLayout SL = smem_layout(p.stages, p.n_tile, p.tk_kpad);
  const uint32_t b_bytes = p.n_tile * 128;
  uint8_t* sA = smem + SL.a_off;
  uint8_t* sB = smem + SL.b_off;
  uint64_t* full_w = reinterpret_cast<uint64_t*>(smem + SL.bar_off);   // weight copy landed
  uint64_t* full_x = full_w + p.stages;                                  // activation copy landed
  uint64_t* empty = full_x + p.stages;
  uint64_t* accf = empty + p.stages;   // [2] accumulator a holds a finished tile
  uint64_t* acce = accf + 2;           // [2] accumulator a has been drained
  uint64_t* drain = acce + 2;
  uint64_t* sbar = drain + 1;          // bulk copies of a shared split tile's inputs landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbar + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 4);  // [0] abort, [2] progress
  float* buf = reinterpret_cast<float*>(smem + SL.buf_off);
  float* s_scale = reinterpret_cast<float*>(smem + SL.scale_off);
  float* s_red = reinterpret_cast<float*>(smem + SL.red_off);
  float* tk = reinterpret_cast<float*>(smem + SL.tk_off);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int c = blockIdx.x;
  // two accumulators of n_tile columns: the MMAs of a CTA's next tile run while
  // the epilogue drains the previous one
  const uint32_t tmem_cols = 2 * p.n_tile < 32 ? 32u : static_cast<uint32_t>(2 * p.n_tile);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      ptx::mbar_init(&full_w[s], 1);
      ptx::mbar_init(&full_x[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&accf[a], 1);
      ptx::mbar_init(&acce[a], kEpiThreads);
    }
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(sbar, 1);
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;   // phases whose epilogue this CTA has finished
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int k = 0; k < p.n_phases; ++k) {
      ptx::prefetch_tmap(&maps.w[k]);
      ptx::prefetch_tmap(&maps.x[k]);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint64_t lim = wait_limit_ns(p.status);
  // Weights are never written by a kernel: the weight stream starts before the
  // previous kernel completes; everything else waits for it.
  // L2 prefetch of the residual rows the first phase's epilogue will read (a
  // hint only, so it may precede the wait below; in a layer's chain those rows
  // were written two kernels back and are long out of L2).
  if (!kMulti && warp >= 2 && warp <= 5 && p.ph[0].epi.kind == EPI_RESID) {
    const TcPhase& P0 = p.ph[0];
    const int G0 = P0.grid;
    if (c < G0) {
      const long long ub = (long long)c * P0.total_units / G0;
      const long long ue = (long long)(c + 1) * P0.total_units / G0;
      for (long long t = ub / P0.kblocks; t * P0.kblocks < ue; ++t) {
        int ftile, rtile;
        tile_coords(P0, t, ftile, rtile);
        const int row0 = rtile * p.n_tile;
        // only the CTA that applies the epilogue of tile t (its first units)
        if (cta_of_unit(t * P0.kblocks, P0.total_units, G0) == c)
          epi_prefetch_inputs<T>(P0.epi, ftile * kTileN, row0,
                                 min(p.n_tile, P0.epi.M_rows - row0), (warp & 3) * 32 + lane);
      }
    }
  }
  // (griddepcontrol.wait holds the whole warp, so the weight producer's
  // warp skips it altogether; its other lanes have no work)
  if (warp != 0) pdl_wait();
  pdl_trigger();

  if (warp == 0 || warp == 6) {
    // ---------------- TMA producers (weights: warp 0, activations: warp 6) ----------------
    if (lane == 0) {
      const bool wprod = warp == 0;
      const uint64_t pol = wprod ? ptx::policy_evict_first() : ptx::policy_evict_last();
      const uint32_t bytes = wprod ? static_cast<uint32_t>(kABytes) : b_bytes;
      uint64_t* full = wprod ? full_w : full_x;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0;   // bit s: stage s has an issued copy
      uint32_t last_phase = 0;    // bit s: parity of that copy's phase
      for (int k = 0; k < p.n_phases && !flags[0]; ++k) {
        const TcPhase& P = p.ph[k];
        const long long U = P.total_units;
        const int Gk = P.grid;
        const long long u_begin = c < Gk ? (long long)c * U / Gk : 0;
        const long long u_end = c < Gk ? (long long)(c + 1) * U / Gk : 0;
        const int KB = P.kblocks;
        if (!wprod && k > 0) {
          if (!wait_counter(&p.sync[k - 1], G, flags, lim)) {
            record_status(p.status, DFLASH_ERR_TIMEOUT);
            flags[0] = 1;
            break;
          }
          // the tiles about to be read by TMA (async proxy) were written with
          // ordinary stores by other CTAs
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        if (wprod && k > 0) {
          // Phase k's weights wait for this CTA's own epilogue of phase k-1:
          // streaming them earlier competes with that epilogue's loads and
          // stores, delays the phase hand-over and costs more than it saves.
          const uint64_t t0 = global_ns();
          while (flags[2] < k) {
            if (flags[0] || global_ns() - t0 > lim) break;
            __nanosleep(32);   // (the epilogue warp on this scheduler is busy)
          }
          if (flags[2] < k) {
            if (!flags[0]) record_status(p.status, DFLASH_ERR_TIMEOUT);
            flags[0] = 1;
            break;
          }
        }
        const CUtensorMap* map = wprod ? &maps.w[k] : &maps.x[k];
        uint8_t* dst0 = wprod ? sA : sB;
        const uint32_t stride = wprod ? static_cast<uint32_t>(kABytes) : b_bytes;
        for (long long u = u_begin; u < u_end; ++u) {
          const int t = static_cast<int>(u / KB);
          const int kb = static_cast<int>(u - (long long)t * KB);
          int ftile, rtile;
          tile_coords(P, t, ftile, rtile);
          if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, lim, flags)) {
            record_status(p.status, DFLASH_ERR_TIMEOUT);
            flags[0] = 1;
            break;
          }
          ptx::mbar_arrive_expect_tx(&full[stage], bytes);
          ptx::tma_load_2d(dst0 + stage * stride, map, &full[stage], kb * 64,
                           wprod ? ftile * kTileN : rtile * p.n_tile, pol);
          issued_mask |= 1u << stage;
          last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == p.stages) { stage = 0; phase ^= 1u; }
        }
      }
      if (flags[0]) {
        // drain: every copy this producer issued must land before the CTA may
        // exit (its own barrier of the stage completes exactly then)
        for (int s = 0; s < p.stages; ++s)
          if (issued_mask & (1u << s))
            ptx::mbar_wait_bounded(&full[s], (last_phase >> s) & 1u, kTimeoutNs, nullptr);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(128, p.n_tile);
      int stage = 0;
      uint32_t phase = 0;
      int tile_i = 0;   // tiles of this CTA so far: accumulator tile_i & 1
      bool issued_any = false;
      for (int k = 0; k < p.n_phases && !flags[0]; ++k) {
        const TcPhase& P = p.ph[k];
        const long long U = P.total_units;
        const int Gk = P.grid;
        const long long u_end = c < Gk ? (long long)(c + 1) * U / Gk : 0;
        const int KB = P.kblocks;
        long long u = c < Gk ? (long long)c * U / Gk : 0;
        while (u < u_end && !flags[0]) {
          const int t = static_cast<int>(u / KB);
          const int kb0 = static_cast<int>(u - (long long)t * KB);
          const int n = static_cast<int>((KB - kb0) < (u_end - u) ? (KB - kb0) : (u_end - u));
          const int acc = tile_i & 1;
          const uint32_t acc_phase = static_cast<uint32_t>(tile_i >> 1) & 1u;
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * p.n_tile);
          if (!ptx::mbar_wait_bounded(&acce[acc], acc_phase ^ 1u, lim, flags)) {
            record_status(p.status, DFLASH_ERR_TIMEOUT);
            flags[0] = 1;
            break;
          }
          ptx::tc_fence_after();
          bool ok = true;
          for (int i = 0; i < n; ++i) {
            if (!ptx::mbar_wait_bounded(&full_w[stage], phase, lim, flags) ||
                !ptx::mbar_wait_bounded(&full_x[stage], phase, lim, flags)) {
              record_status(p.status, DFLASH_ERR_TIMEOUT);
              flags[0] = 1;
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint64_t a_desc = ptx::sw128_kmajor_desc(ptx::smem_addr(sA + stage * kABytes));
            const uint64_t b_desc = ptx::sw128_kmajor_desc(ptx::smem_addr(sB + stage * b_bytes));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::mma_bf16(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc,
                            (i > 0 || kk > 0) ? 1u : 0u);
            ptx::mma_commit(&empty[stage]);
            issued_any = true;
            if (++stage == p.stages) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          ptx::mma_commit(&accf[acc]);
          ++tile_i;
          u += n;
        }
      }
      if (flags[0] && issued_any) {
        // drain: wait for the MMAs already issued before TMEM is released
        ptx::mma_commit(drain);
        ptx::mbar_wait_bounded(drain, 0u, kTimeoutNs, nullptr);
      }
    }
  } else {
    // ---------------- epilogue warps (2-5) ----------------
    const int ew = warp & 3;            // TMEM lane quarter this warp may access
    const int f = ew * 32 + lane;       // tile column (weight row) of this thread
    const int etid = threadIdx.x - 64;  // 0..127
    int tile_i = 0;
    uint32_t sphase = 0;                // parity of sbar's next completion
    bool stop = false;
    for (int k = 0; k < p.n_phases && !stop; ++k) {
      const TcPhase& P = p.ph[k];
      const EpiParams& E = P.epi;
      const long long U = P.total_units;
      const int Gk = P.grid;
      const long long u_end = c < Gk ? (long long)(c + 1) * U / Gk : 0;
      const int KB = P.kblocks;
      long long u = c < Gk ? (long long)c * U / Gk : 0;
      if (k > 0) {
        // the epilogue reads what earlier phases wrote (row norms, residual)
        bool ok = true;
        if (etid == 0) ok = wait_counter(&p.sync[k - 1], G, flags, lim);
        if (ptx::named_bar_or(1, kEpiThreads, !ok)) {
          record_status(p.status, DFLASH_ERR_TIMEOUT);
          flags[0] = 1;
          break;
        }
      }
      // With one row tile, the RMS row scales of the phase are computed once,
      // ahead of its first accumulator.
      const bool scales_once = P.n_rtiles == 1;
      if (scales_once) {
        epi_row_scales(E, 0, min(p.n_tile, E.M_rows), s_scale, etid, kEpiThreads);
        ptx::named_bar_sync(1, kEpiThreads);
      }
      // fused top-K (one row tile only): empty per-warp state
      const bool fused_tk = E.kind == EPI_LOGITS && E.tk_part != nullptr && p.tk_kpad > 0;
      const int tk_stride = 2 + 2 * p.tk_kpad;
      if (fused_tk) {
        for (int i = etid; i < 4 * p.n_tile * tk_stride; i += kEpiThreads) {
          const int q = i % tk_stride;
          tk[i] = q == 0 ? -CUDART_INF_F
                : q == 1 ? 0.f
                : q < 2 + p.tk_kpad ? -CUDART_INF_F : __int_as_float(0x7fffffff);
        }
        ptx::named_bar_sync(1, kEpiThreads);
      }
      // Several 16-row chunks per tile: a split tile's epilogue is shared by
      // all its contributors.  Each posts its partial sums (c_first too) in
      // a first pass over its tiles, then finishes its share of the tile's rows
      // from all the slots in a second pass (below).
      const bool bphase = kMulti && !fused_tk;
      while (u < u_end) {
        const int acc = tile_i & 1;
        const uint32_t acc_phase = static_cast<uint32_t>(tile_i >> 1) & 1u;
        const uint32_t tacc = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) +
                              static_cast<uint32_t>(acc * p.n_tile);
        const int t = static_cast<int>(u / KB);
        const int kb0 = static_cast<int>(u - (long long)t * KB);
        const int n = static_cast<int>((KB - kb0) < (u_end - u) ? (KB - kb0) : (u_end - u));
        int ftile, rtile;
        tile_coords(P, t, ftile, rtile);
        const int row0 = rtile * p.n_tile;
        const int nrows = min(p.n_tile, E.M_rows - row0);
        const int c_first = cta_of_unit((long long)t * KB, U, Gk);
        const int c_last = cta_of_unit((long long)t * KB + KB - 1, U, Gk);
        const int nslots = c_last - c_first + 1;
        // A tile split over several CTAs is finished by c_first: the tile's
        // first K blocks close c_first's unit range, so it is among the last to
        // finish its share.  The others post partial sums (slot c - c_first)
        // and a release-add; c_first adds them, in slot order, to its own
        // accumulator read straight from TMEM.
        const bool single = nslots == 1;
        const bool reducer = !single && c == c_first;
        // One 16-row chunk per tile: what the epilogue reads besides the
        // accumulator is loaded while the MMAs run -- the chunk's EpiPre and,
        // for a split tile, the sum of the other CTAs' partials (their K
        // blocks open their unit ranges, so they are posted early).  A partial
        // slot is then stored column-major, [128 columns][16 rows]: thread f
        // writes and reads its column's 16 values as four float4.
        const bool early = !kMulti;
        const bool resid4 = early && E.kind == EPI_RESID && (E.N_feat & 3) == 0;
        const bool qkv4 = early && (E.N_feat & 3) == 0 && (E.ldo & 3) == 0 &&
                          ((E.kind == EPI_QKV && (E.head_dim & 7) == 0) || E.kind == EPI_STORE);
        const bool kv4 = early && E.kind == EPI_KV && (E.head_dim & 7) == 0 &&
                         ((E.n_kv * E.head_dim) & 3) == 0 && (E.N_feat & 3) == 0;
        const bool swiglu4 = early && E.kind == EPI_SWIGLU && (E.N_feat & 3) == 0 &&
                             (E.ldo & 1) == 0;
        EpiPre pre;
        float4 psum[4];
        if (early && (single || reducer)) {
          if (resid4) epi_preload_resid4<T>(E, ftile * kTileN, row0, nrows, ew, lane, pre);
          else if (qkv4) epi_preload_qkv4(E, ftile * kTileN, row0, nrows, ew, lane, pre);
          else if (kv4) epi_preload_kv4(E, ftile * kTileN, row0, nrows, ew, lane, pre);
          else epi_preload<T>(E, ftile * kTileN, row0, nrows, f, pre);
          epi_touch_out<T>(E, ftile * kTileN, row0, f);
        }
        if (early && reducer) {
          bool got = true;
          if (etid == 0) got = wait_counter(&P.counters[c_first], nslots - 1, flags, lim);
          if (ptx::named_bar_or(1, kEpiThreads, !got)) {
            record_status(p.status, DFLASH_ERR_TIMEOUT);
            flags[0] = 1;
            stop = true;
            break;
          }
          const float4* slots4 = reinterpret_cast<const float4*>(
              p.part + (size_t)c_first * P.max_slots * kChunk * kTileN);
#pragma unroll
          for (int q = 0; q < 4; ++q) psum[q] = make_float4(0.f, 0.f, 0.f, 0.f);
          // slots 1.. in order, five slots' loads in flight together
          for (int s0 = 1; s0 < nslots; s0 += 5) {
            float4 v[5][4];
#pragma unroll
            for (int sq = 0; sq < 5; ++sq)
#pragma unroll
              for (int q = 0; q < 4; ++q)
                v[sq][q] = s0 + sq < nslots
                               ? __ldcg(slots4 + (size_t)(s0 + sq) * (kChunk * kTileN / 4) +
                                        f * 4 + q)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int sq = 0; sq < 5; ++sq)
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                psum[q].x += v[sq][q].x;
                psum[q].y += v[sq][q].y;
                psum[q].z += v[sq][q].z;
                psum[q].w += v[sq][q].w;
              }
          }
        }

        const bool ok = ptx::mbar_wait_bounded(&accf[acc], acc_phase, lim, flags);
        if (!ok) {
          record_status(p.status, DFLASH_ERR_TIMEOUT);
          flags[0] = 1;
        }
        if (ptx::named_bar_or(1, kEpiThreads, !ok)) {
          stop = true;
          break;
        }
        ptx::tc_fence_after();

        if (!single && (!reducer || bphase)) {
          float* my_part = p.part + ((size_t)c_first * P.max_slots + (c - c_first)) *
                                        (size_t)p.n_tile * kTileN;
          for (int c0 = 0; c0 < nrows; c0 += kChunk) {
            float v[16];
            __syncwarp();
            ptx::tmem_ld_32x16(tacc + static_cast<uint32_t>(c0), v);
            if (early) {
              float4* d4 = reinterpret_cast<float4*>(my_part) + f * 4;
#pragma unroll
              for (int q = 0; q < 4; ++q)
                d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            } else {
              // row-major: each warp store is one 128-byte row segment
#pragma unroll
              for (int j = 0; j < 16; ++j) my_part[(size_t)(c0 + j) * kTileN + f] = v[j];
            }
          }
          ptx::tc_fence_before();
          ptx::mbar_arrive(&acce[acc]);
          ptx::named_bar_sync(1, kEpiThreads);
          if (etid == 0) red_release_add(&P.counters[c_first], 1);
        } else {
          if (!scales_once) epi_row_scales(E, row0, nrows, s_scale, etid, kEpiThreads);
          for (int i = etid; i < 4 * p.n_tile; i += kEpiThreads) s_red[i] = 0.f;
          if (reducer && !early) {
            bool got = true;
            if (etid == 0) got = wait_counter(&P.counters[c_first], nslots - 1, flags, lim);
            if (ptx::named_bar_or(1, kEpiThreads, !got)) {
              record_status(p.status, DFLASH_ERR_TIMEOUT);
              flags[0] = 1;
              stop = true;
              break;
            }
          }
          const float* slots = p.part + (size_t)c_first * P.max_slots * p.n_tile * kTileN;
          // several chunks per tile: 32 rows at a time, every load of a batch in flight
          const bool batched = bphase;   // (single tiles here: reducers post instead)
          if (batched)
            epi_tile_batched<T>(E, true, tacc, ftile * kTileN, row0, 0, nrows, p.n_tile, slots, 1,
                                s_scale, row0, s_red, buf, f, ew, lane);
          for (int c0 = 0; !batched && c0 < nrows; c0 += kChunk) {
            const int nr = min(kChunk, nrows - c0);
            float sum[kChunk];
            __syncwarp();
            ptx::tmem_ld_32x16(tacc + static_cast<uint32_t>(c0), sum);
            // slots 1.. in order; four slots' loads (16 rows each) in flight together
            for (int s0 = 1; !early && s0 < nslots; s0 += 4) {
              float v[4][kChunk];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float* src = slots + ((size_t)(s0 + q) * p.n_tile + c0) * kTileN + f;
#pragma unroll
                for (int j = 0; j < kChunk; ++j)
                  v[q][j] = (s0 + q < nslots && j < nr) ? __ldcg(src + (size_t)j * kTileN) : 0.f;
              }
#pragma unroll
              for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int j = 0; j < kChunk; ++j) sum[j] += v[q][j];
            }
            if (early && reducer) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                sum[4 * q] += psum[q].x;
                sum[4 * q + 1] += psum[q].y;
                sum[4 * q + 2] += psum[q].z;
                sum[4 * q + 3] += psum[q].w;
              }
            }
#pragma unroll
            for (int j = 0; j < kChunk; ++j) buf[j * kBufLd + f] = sum[j];
            ptx::named_bar_sync(1, kEpiThreads);
            if (!early) epi_preload<T>(E, ftile * kTileN, row0 + c0, nr, f, pre);
            if (resid4)
              epi_apply_resid4<T>(E, buf, ftile * kTileN, row0, nr, ew, lane, row0, s_red,
                                  p.n_tile, pre);
            else if (qkv4)
              epi_apply_qkv4<T>(E, buf, ftile * kTileN, row0, nr, ew, lane, s_scale, row0, pre);
            else if (kv4)
              epi_apply_kv4<T>(E, buf, ftile * kTileN, nr, ew, lane, pre);
            else if (swiglu4)
              epi_apply_swiglu4<T>(E, buf, ftile * kTileN, row0 + c0, nr, ew, lane, s_scale, row0);
            else
              epi_apply_chunk<T>(E, buf, ftile * kTileN, row0 + c0, nr, f, s_scale, row0, s_red,
                                 p.n_tile, ew, pre);
            if (fused_tk) {
              tk_update_rows(E, tk, p.tk_kpad, p.n_tile, buf, s_scale, c0, nr, ftile * kTileN,
                             ew, lane);
              __syncwarp();
            }
            ptx::named_bar_sync(1, kEpiThreads);
          }
          ptx::tc_fence_before();
          ptx::mbar_arrive(&acce[acc]);
          if (E.kind == EPI_RESID)
            epi_resid_flush(E, ftile, row0, nrows, s_red, p.n_tile, 4, etid, kEpiThreads);
          if (reducer && etid == 0) P.counters[c_first] = 0;   // for the next launch
          ptx::named_bar_sync(1, kEpiThreads);
        }
        ++tile_i;
        u += n;
      }
      if (bphase && !stop) {
        // second pass: contributor j = c - c_first of a split tile finishes its
        // rows [j nrows / nslots, (j + 1) nrows / nslots) once all have posted
        long long u2 = c < Gk ? (long long)c * U / Gk : 0;
        while (u2 < u_end) {
          const int t = static_cast<int>(u2 / KB);
          const int kb0 = static_cast<int>(u2 - (long long)t * KB);
          const int n = static_cast<int>((KB - kb0) < (u_end - u2) ? (KB - kb0) : (u_end - u2));
          u2 += n;
          const int c_first = cta_of_unit((long long)t * KB, U, Gk);
          const int nslots = cta_of_unit((long long)t * KB + KB - 1, U, Gk) - c_first + 1;
          if (nslots == 1) continue;
          int ftile, rtile;
          tile_coords(P, t, ftile, rtile);
          const int row0 = rtile * p.n_tile;
          const int nrows = min(p.n_tile, E.M_rows - row0);
          const int j = c - c_first;
          const int rs0 = j * nrows / nslots, rs1 = (j + 1) * nrows / nslots;
          bool got = true;
          if (etid == 0) got = wait_counter(&P.counters[c_first], nslots, flags, lim);
          if (ptx::named_bar_or(1, kEpiThreads, !got)) {
            record_status(p.status, DFLASH_ERR_TIMEOUT);
            flags[0] = 1;
            stop = true;
            break;
          }
          if (!scales_once)
            epi_row_scales(E, row0 + rs0, rs1 - rs0, s_scale + rs0, etid, kEpiThreads);
          const float* slots = p.part + (size_t)c_first * P.max_slots * p.n_tile * kTileN;
          // from shared memory when the share's inputs fit in the ring
          const size_t share_in = (size_t)(nslots + 1) * (rs1 - rs0) * kTileN * 4;
          const uintptr_t ptr_or = reinterpret_cast<uintptr_t>(E.out) |
                                   reinterpret_cast<uintptr_t>(E.logits) |
                                   reinterpret_cast<uintptr_t>(E.x) |
                                   reinterpret_cast<uintptr_t>(E.xn) |
                                   reinterpret_cast<uintptr_t>(E.gain);
          const bool vec_ok = (E.N_feat % kTileN) == 0 && (E.ldo & 3) == 0 &&
                              (ptr_or & 15) == 0 &&
                              (E.kind != EPI_QKV || (E.head_dim & 7) == 0) &&
                              (E.kind != EPI_KV || ((E.head_dim & 7) == 0 &&
                                                    (E.n_kv * E.head_dim) % kTileN == 0));
          if (vec_ok && share_in <= SL.bar_off) {
            if (!scales_once) ptx::named_bar_sync(1, kEpiThreads);   // s_scale written
            if (!epi_share_smem<T>(E, smem, sbar, sphase, slots, nslots, p.n_tile,
                                   ftile * kTileN, row0, rs0, rs1, ftile, s_scale, ew, lane, lim,
                                   flags, p.status)) {
              stop = true;
              break;
            }
          } else {
            for (int i = etid; i < 4 * p.n_tile; i += kEpiThreads) s_red[i] = 0.f;
            epi_tile_batched<T>(E, false, 0u, ftile * kTileN, row0, rs0, rs1, p.n_tile, slots,
                                nslots, s_scale, row0, s_red, buf, f, ew, lane);
            if (E.kind == EPI_RESID)
              epi_resid_flush(E, ftile, row0 + rs0, rs1 - rs0, s_red + rs0, p.n_tile, 4, etid,
                              kEpiThreads);
            ptx::named_bar_sync(1, kEpiThreads);
          }
          // the last contributor through resets the counter for the next launch
          if (etid == 0 && atomicAdd(&P.counters[c_first], 1) == 2 * nslots - 1)
            P.counters[c_first] = 0;
        }
      }
      if (stop) break;
      if (fused_tk) {
        // this CTA's record of every mask row: merge the four warps' states
        ptx::named_bar_sync(1, kEpiThreads);
        const int K = E.tk_K;
        const int n_out = E.M_rows / E.L * (E.L - 1);
        const int n_rows = min(p.n_tile, E.M_rows);
        // eight rows per warp pass, lane = 4 * row slot + warp state
        for (int base = ew; base < n_rows; base += 32) {
          const int row = base + 4 * (lane >> 2);
          const bool live = row < n_rows && row % E.L != 0;
          const float* st = tk + ((lane & 3) * p.n_tile + (live ? row : 0)) * tk_stride;
          float m = live ? st[0] : -CUDART_INF_F;
          float sm = live ? st[1] : 0.f;
          float tv[8];
          int ti[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            tv[q] = live && q < K ? st[2 + q] : -CUDART_INF_F;
            ti[q] = live && q < K ? __float_as_int(st[2 + p.tk_kpad + q]) : 0x7fffffff;
          }
          tk_lane_merge(tv, ti, m, sm, 1, 2);
          if (live && (lane & 3) == 0) {
            const int orow = row / E.L * (E.L - 1) + row % E.L - 1;
            float* rec = E.tk_part + ((size_t)c * n_out + orow) * kTkStride;
            rec[0] = m;
            rec[1] = sm;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (q < K) {
                rec[2 + q] = tv[q];
                rec[2 + kTkMax + q] = __int_as_float(ti[q]);
              }
          }
        }
        if (E.tk_ids != nullptr) {
          // Final merge: the last n_merge CTAs to publish their records wait
          // for the rest, then each merges rows slot, slot + n_merge, ...
          int* arrive = p.sync + kMaxPhases + 1;
          int* merged = p.sync + kMaxPhases + 2;
          const int n_merge = min(n_out, G);
          ptx::named_bar_sync(1, kEpiThreads);
          if (etid == 0) {
            __threadfence();
            flags[1] = atomicAdd(arrive, 1);
          }
          ptx::named_bar_sync(1, kEpiThreads);
          const int slot = flags[1] - (G - n_merge);
          if (slot >= 0) {
            bool ok = true;
            if (etid == 0) {
              ok = wait_counter(arrive, G, flags, lim);
              __threadfence();
            }
            if (ptx::named_bar_or(1, kEpiThreads, !ok)) {
              record_status(p.status, DFLASH_ERR_TIMEOUT);
              flags[0] = 1;
            } else {
              for (int orow = slot; orow < n_out; orow += n_merge)
                tk_row_merge(E, G, n_out, orow, etid, ew, lane, tk);
              // the last merger resets both counters for the next launch
              if (etid == 0 && atomicAdd(merged, 1) == n_merge - 1) {
                *arrive = 0;
                *merged = 0;
              }
            }
          }
        }
      }
      // this CTA's share of phase k is written: publish it
      ptx::named_bar_sync(1, kEpiThreads);
      if (etid == 0) {
        red_release_add(&p.sync[k], 1);
        flags[2] = k + 1;   // the weight stream of phase k+1 may start
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    ptx::tmem_dealloc(tmem_base, tmem_cols);
  }
  // The last CTA out resets the phase counters for the next launch (every CTA
  // has passed all of its waits by now).
  if (threadIdx.x == 0) {
    __threadfence();
    const int prev = atomicAdd(&p.sync[kMaxPhases], 1);
    if (prev == G - 1) {
      for (int k = 0; k < kMaxPhases; ++k) p.sync[k] = 0;
      p.sync[kMaxPhases] = 0;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

template <typename T, bool kMulti>
void set_smem_attr_once(int bytes) {
  static int done = 0;
  if (done < bytes) {
    cudaFuncSetAttribute(gemm_tc_kernel<T, kMulti>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         bytes);
    done = bytes;
  }
}

}  // namespace

bool encode_kmajor_map(CUtensorMap* map, const void* base, int rows, int K,
                       long long row_stride_elems, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_stride_elems) * 2};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int tc_row_tile(int M_rows) {
  int n = 16;
  while (n < M_rows && n < 256) n <<= 1;
  return n;
}

TcPlan tc_plan(int M_rows, int N_feat, int K, int grid, int tk_kpad) {
  TcPlan pl{};
  pl.n_tile = tc_row_tile(M_rows);
  pl.n_rtiles = ceil_div(M_rows, pl.n_tile);
  pl.n_ftiles = ceil_div(N_feat, kTileN);
  pl.kblocks = K / 64;
  pl.total_units = (long long)pl.n_ftiles * pl.n_rtiles * pl.kblocks;
  pl.grid = static_cast<int>(pl.total_units < grid ? pl.total_units : grid);
  if (pl.grid < 1) pl.grid = 1;
  // Several row tiles (compute-bound tiles of up to 256 rows): where a grid
  // of at least five sixths of the SMs gives every CTA whole half tiles, use
  // it -- split tiles then have two contributors at most, each ending on the
  // half-tile boundary, or none, which shortens the finish after the MMAs
  // more than the idle SMs lengthen them.
  if (pl.n_rtiles > 1 && pl.kblocks >= 2 && pl.kblocks % 2 == 0) {
    const long long half = pl.kblocks / 2;
    for (int g = pl.grid; g >= (5 * pl.grid + 5) / 6; --g) {
      if (pl.total_units % g == 0 && (pl.total_units / g) % half == 0) {
        pl.grid = g;
        break;
      }
    }
  }
  const int n_tiles = pl.n_ftiles * pl.n_rtiles;
  int ms = 1;
  for (int t = 0; t < n_tiles; ++t) {
    const int a = cta_of_unit((long long)t * pl.kblocks, pl.total_units, pl.grid);
    const int b = cta_of_unit((long long)t * pl.kblocks + pl.kblocks - 1, pl.total_units, pl.grid);
    if (b - a + 1 > ms) ms = b - a + 1;
  }
  pl.max_slots = ms;
  pl.part_bytes = (size_t)pl.grid * ms * pl.n_tile * kTileN * sizeof(float);
  // the deepest ring that fits: it also carries the weight stream across the
  // hand-over between the phases of a chain
  int stages = 1;
  while (stages < 24 && smem_layout(stages + 1, pl.n_tile, tk_kpad).total <= 227u * 1024u) ++stages;
  pl.stages = stages;
  pl.smem_bytes = smem_layout(stages, pl.n_tile, tk_kpad).total;
  return pl;
}

dflash_status launch_gemm_chain(const GemmPhase* ph, int n_phases, int M_rows, float* part,
                                int* counters, int* status, cudaStream_t st) {
  if (n_phases < 1 || n_phases > kMaxPhases)
    return set_error(DFLASH_ERR_INVALID_ARG, "GEMM chain: 1..%d phases", kMaxPhases);
  const int G = num_sms();
  TcMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  TcParams p{};
  p.M_rows = M_rows;
  p.n_phases = n_phases;
  p.part = part;
  p.sync = counters + kMaxPhases * G;
  p.status = status;
  int smem = 0;
  for (int k = 0; k < n_phases; ++k)
    if (ph[k].epi.kind == EPI_LOGITS && ph[k].epi.tk_part != nullptr) {
      p.tk_kpad = (ph[k].epi.tk_K + 7) / 8 * 8;
      if (ph[k].epi.tk_ids == nullptr || k != n_phases - 1 || ph[k].epi.tk_K > kTkMax)
        return set_error(DFLASH_ERR_INVALID_ARG,
                         "fused top-K: outputs set, LM head the last phase, K <= %d", kTkMax);
    }
  for (int k = 0; k < n_phases; ++k) {
    const TcPlan pl = tc_plan(M_rows, ph[k].N, ph[k].K, G, p.tk_kpad);
    p.n_tile = pl.n_tile;
    p.stages = pl.stages;
    smem = pl.smem_bytes;
    if (p.tk_kpad && pl.n_rtiles != 1)
      return set_error(DFLASH_ERR_UNSUPPORTED, "fused top-K needs one row tile");
    TcPhase& P = p.ph[k];
    P.N_feat = ph[k].N;
    P.K = ph[k].K;
    P.n_rtiles = pl.n_rtiles;
    P.n_ftiles = pl.n_ftiles;
    P.kblocks = pl.kblocks;
    P.grid = pl.grid;
    P.total_units = pl.total_units;
    P.max_slots = pl.max_slots;
    P.counters = counters + k * G;
    P.epi = ph[k].epi;
    maps.w[k] = *ph[k].tmW;
    if (!encode_kmajor_map(&maps.x[k], ph[k].X, M_rows, ph[k].K, ph[k].ldx, pl.n_tile))
      return set_error(DFLASH_ERR_CUDA, "cannot encode the activation TMA descriptor");
  }
  TraceScope ts("gemm_tc", st);
  static_assert(sizeof(TcParams) + sizeof(TcMaps) <= 32000, "kernel parameter space");
  if (p.n_tile > kChunk) {
    set_smem_attr_once<__nv_bfloat16, true>(smem);
    launch_k(gemm_tc_kernel<__nv_bfloat16, true>, dim3(G), dim3(kThreads), smem, st, maps, p);
  } else {
    set_smem_attr_once<__nv_bfloat16, false>(smem);
    launch_k(gemm_tc_kernel<__nv_bfloat16, false>, dim3(G), dim3(kThreads), smem, st, maps, p);
  }
  return check_launch("gemm_tc");
}

int gemm_counter_ints() { return kMaxPhases * num_sms() + kMaxPhases + 3; }

}  // namespace dfl
