// Vocabulary-wide log-softmax and top-K for K <= 8, streamed through shared
// memory (step a6 when the logits are already in memory: the stress workload,
// the batched drafter's rows, any standalone call).
//
// "Accelerating Speculative Decoding with Block Diffusion Draft Trees",
// section 3.4.2 (q_i = softmax(l_i)) and section 3.4.4 (Lemma 1: per depth
// only the top-K tokens, by descending probability, enter the tree).
//
// The pass reads every logit once; it is HBM-bound only if the loads never
// wait for the arithmetic and the arithmetic per logit stays small.  Work is
// cut into pieces (a row, or a contiguous part of one when there are fewer
// rows than warps) and every warp streams its own pieces, one after another,
// through a private ring of 4 KB bulk copies (cp.async.bulk, completion on an
// mbarrier); its lane 0 keeps the ring full, running ahead across piece
// boundaries.  Per 4 KB stage a lane holds eight 16-byte vectors in registers:
//   * sum of exp: every lane keeps its own running max m (rescaled at most
//     once per stage) and four pairs of partial sums of exp(x - m);
//   * top-K: the warp keeps a sorted list (lane j: its j-th best, value desc,
//     id asc).  A value strictly below the list's K-th cannot be in the
//     piece's top-K, so a stage costs one compare of each lane's maximum; for
//     the rare lane at or above it the warp re-reads that lane's logits from
//     the slot (one word per lane) and inserts the qualifying ones one at a
//     time.  Because one warp sees the whole piece, its threshold is the
//     piece's running K-th best and insertions stay near K ln(n / n0) per
//     piece.  The first stage seeds the threshold with the K-th largest lane
//     maximum (K values at or above it).
// At the end of a piece the warp reduces its (max, sum) pairs; a split row's
// warps publish records and the last to arrive merges them.
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "topk8.cuh"

#include <math_constants.h>

namespace dfl {

namespace {

constexpr int kWarps = 8;                       // warps per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kStageBytes = 4096;               // one bulk copy
constexpr int kStages = 3;                      // per warp
constexpr int kVec = kStageBytes / 16 / 32;     // 16-byte vectors per lane per stage (8)
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kRecStride = 2 + 2 * 32;          // the partial-record layout of the workspace

template <typename T> struct VecN;
template <> struct VecN<float> { static constexpr int N = 4; };
template <> struct VecN<__nv_bfloat16> { static constexpr int N = 8; };

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16 bytes of -inf logits (the slots past a piece's end).
template <typename T> __device__ __forceinline__ uint4 neg_inf16();
template <> __device__ __forceinline__ uint4 neg_inf16<float>() {
  return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
}
template <> __device__ __forceinline__ uint4 neg_inf16<__nv_bfloat16>() {
  return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
}

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) {
  return *reinterpret_cast<const __nv_bfloat162*>(&w);
}
__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 h) {
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Maximum of a vector, kept packed for bf16 (two candidates per word).
template <typename T>
__device__ __forceinline__ uint32_t vec_max_packed(const uint4& r) {
  if constexpr (sizeof(T) == 4) {
    return __float_as_uint(fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)),
                                 fmaxf(__uint_as_float(r.z), __uint_as_float(r.w))));
  } else {
    return as_u32(__hmax2(__hmax2(as_bf2(r.x), as_bf2(r.y)), __hmax2(as_bf2(r.z), as_bf2(r.w))));
  }
}
template <typename T>
__device__ __forceinline__ uint32_t max_packed(uint32_t a, uint32_t b) {
  if constexpr (sizeof(T) == 4) return __float_as_uint(fmaxf(__uint_as_float(a), __uint_as_float(b)));
  else return as_u32(__hmax2(as_bf2(a), as_bf2(b)));
}
template <typename T>
__device__ __forceinline__ float unpack_max(uint32_t p) {
  if constexpr (sizeof(T) == 4) return __uint_as_float(p);
  else return fmaxf(__uint_as_float(p << 16), __uint_as_float(p & 0xffff0000u));
}

// acc += exp2((x - m) log2 e) over a lane's stage, in fp32 pairs; the 32-bit
// words of a vector go to the four accumulators in turn.
template <typename T>
__device__ __forceinline__ void exp_sum(const uint4 (&r)[kVec], float m, float2 (&acc)[4]) {
  const float mo = m == -CUDART_INF_F ? 0.f : -m * kLog2e;
  const float2 c2 = make_float2(kLog2e, kLog2e), o2 = make_float2(mo, mo);
#pragma unroll
  for (int q = 0; q < kVec; ++q) {
    const uint32_t w[4] = {r[q].x, r[q].y, r[q].z, r[q].w};
    if constexpr (sizeof(T) == 4) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float2 t = __ffma2_rn(
            make_float2(__uint_as_float(w[2 * k]), __uint_as_float(w[2 * k + 1])), c2, o2);
        acc[2 * (q & 1) + k] = __fadd2_rn(acc[2 * (q & 1) + k], make_float2(ex2(t.x), ex2(t.y)));
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 t = __ffma2_rn(
            make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u)), c2, o2);
        acc[k] = __fadd2_rn(acc[k], make_float2(ex2(t.x), ex2(t.y)));
      }
    }
  }
}

// The warp's sorted list: lane j < K holds its j-th best (value desc, id asc).
// Insert (cv, cid) if it ranks among the K best; returns the new K-th value
// (-inf while the list has fewer than K entries).
__device__ __forceinline__ float list_insert(float& lv, int& li, int K, int lane, float cv,
                                             int cid) {
  const bool ahead = lane < K && tk_better(lv, li, cv, cid);
  const int pos = __popc(__ballot_sync(0xffffffffu, ahead));
  const float pv = __shfl_up_sync(0xffffffffu, lv, 1);
  const int pi = __shfl_up_sync(0xffffffffu, li, 1);
  if (pos < K) {
    if (lane == pos) { lv = cv; li = cid; }
    else if (lane > pos && lane < K) { lv = pv; li = pi; }
  }
  return __shfl_sync(0xffffffffu, lv, K - 1);
}

struct StreamArgs {
  int rows, vocab, K, splits, chunk, n_pieces;
  long long ld;
  float* part;         // [rows][splits][2 + 2*32] when splits > 1
  int* counters;       // [rows]
  int32_t* ids;
  float* logp;
  int* status;         // workspace status word or null
};

// Piece pc: its row, first logit, number of logits, and the bytes covered by
// 16-byte bulk copies (the rest, fewer than 16 bytes, is read directly).
struct Piece {
  int row, v0, n_el;
  long long nb;
};
template <int ES>
__device__ __forceinline__ Piece piece_of(const StreamArgs& a, int pc) {
  Piece p;
  p.row = pc / a.splits;
  const int split = pc - p.row * a.splits;
  p.v0 = split * a.chunk;
  const int v1 = min(a.vocab, p.v0 + a.chunk);
  p.n_el = v1 > p.v0 ? v1 - p.v0 : 0;
  p.nb = (long long)p.n_el * ES / 16 * 16;
  return p;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
topk_stream_kernel(const T* __restrict__ logits, const StreamArgs a) {
  constexpr int VN = VecN<T>::N;
  constexpr int es = sizeof(T);
  extern __shared__ __align__(128) uint8_t ring_all[];
  __shared__ uint64_t full_all[kWarps][kStages];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = ring_all + warp * kStages * kStageBytes;
  uint64_t* full = full_all[warp];
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) ptx::mbar_init(&full[s], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  pdl_wait();
  pdl_trigger();

  const int K = a.K;
  const int GW = gridDim.x * kWarps;
  const int gw = blockIdx.x * kWarps + warp;
  const uint64_t pol = ptx::policy_evict_first();

  // Issue cursor (the same in every lane; lane 0 issues): the next stage of
  // the warp's sequence of (piece, 4 KB slice), running ahead of consumption.
  int ipc = gw;
  long long ioff = 0, inb = 0;
  const uint8_t* isrc = nullptr;
  auto cursor_at = [&](int pc) {
    inb = 0;
    if (pc < a.n_pieces) {
      const Piece p = piece_of<es>(a, pc);
      inb = p.nb;
      isrc = reinterpret_cast<const uint8_t*>(logits + (long long)p.row * a.ld + p.v0);
    }
  };
  cursor_at(ipc);
  uint32_t n_issued = 0;
  auto issue_next = [&](int slot) {
    while (ipc < a.n_pieces && ioff >= inb) {
      ipc += GW;
      ioff = 0;
      cursor_at(ipc);
    }
    if (ipc >= a.n_pieces) return;
    const uint32_t bytes = static_cast<uint32_t>(inb - ioff < kStageBytes ? inb - ioff : kStageBytes);
    if (lane == 0) {
      ptx::mbar_arrive_expect_tx(&full[slot], bytes);
      ptx::bulk_load(ring + slot * kStageBytes, isrc + ioff, bytes, &full[slot], pol);
    }
    ioff += bytes;
    ++n_issued;
  };
#pragma unroll
  for (int s = 0; s < kStages; ++s) issue_next(s);

  uint32_t seq = 0;   // stages consumed so far
  bool ab = false;
  for (int pc = gw; pc < a.n_pieces && !ab; pc += GW) {
    const Piece p = piece_of<es>(a, pc);
    float m = -CUDART_INF_F;
    float2 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
    float lv = -CUDART_INF_F;     // this lane's entry of the warp list
    int li = 0x7fffffff;
    float thr = -CUDART_INF_F;    // warp-uniform: the list's K-th, or the seed
    bool first = true;
    for (long long off = 0; off < p.nb; off += kStageBytes, ++seq) {
      const int slot = static_cast<int>(seq % kStages);
      const uint32_t par = (seq / kStages) & 1u;
      if (!ptx::mbar_wait_bounded(&full[slot], par, kTimeoutNs, nullptr)) {
        record_status(a.status, DFLASH_ERR_TIMEOUT);
        ab = true;
        break;
      }
      const int nvec = static_cast<int>((p.nb - off < kStageBytes ? p.nb - off : kStageBytes) / 16);
      const uint4* sv = reinterpret_cast<const uint4*>(ring + slot * kStageBytes);
      uint4 r[kVec];
      if (nvec == kStageBytes / 16) {
#pragma unroll
        for (int q = 0; q < kVec; ++q) r[q] = sv[lane + 32 * q];
      } else {
#pragma unroll
        for (int q = 0; q < kVec; ++q)
          r[q] = lane + 32 * q < nvec ? sv[lane + 32 * q] : neg_inf16<T>();
      }
      uint32_t t2 = vec_max_packed<T>(r[0]);
#pragma unroll
      for (int q = 1; q < kVec; ++q) t2 = max_packed<T>(t2, vec_max_packed<T>(r[q]));
      const float tmax = unpack_max<T>(t2);

      if (first) {
        // seed: the K-th largest lane maximum (K distinct values at or above it)
        uint32_t bits = ordered_bits(tmax);
        float seed = -CUDART_INF_F;
        for (int q = 0; q < K; ++q) {
          const uint32_t mb = __reduce_max_sync(0xffffffffu, bits);
          seed = from_ordered_bits(mb);
          const unsigned h = __ballot_sync(0xffffffffu, bits == mb);
          if (lane == __ffs(h) - 1) bits = 0u;
        }
        thr = fmaxf(thr, seed);
        first = false;
      }
      unsigned hot = __ballot_sync(0xffffffffu, tmax >= thr);
      if (hot) {
        // rare: a lane holds values at or above the threshold.  The warp
        // re-reads that lane's 32 words of the slot, one word per lane (lane
        // t: word t & 3 of the lane's vector t >> 2), and inserts the values
        // at or above the threshold one at a time.
        const uint32_t* sw = reinterpret_cast<const uint32_t*>(ring + slot * kStageBytes);
        const int qv = lane >> 2, kw = lane & 3;
        const int id0 = p.v0 + static_cast<int>(off / es);
        while (hot) {
          const int src = __ffs(hot) - 1;
          hot &= hot - 1;
          const int j = src + 32 * qv;                  // the vector's index in the stage
          const bool ok = j < nvec;
          const uint32_t w = ok ? sw[4 * j + kw] : 0u;
#pragma unroll
          for (int h = 0; h < (es == 2 ? 2 : 1); ++h) {
            const float xv = es == 2 ? __uint_as_float(h ? (w & 0xffff0000u) : (w << 16))
                                     : __uint_as_float(w);
            unsigned bal = __ballot_sync(0xffffffffu, ok && xv >= thr);
            while (bal) {
              const int sl = __ffs(bal) - 1;
              bal &= bal - 1;
              const float cv = __shfl_sync(0xffffffffu, xv, sl);
              const int cid = id0 + (src + 32 * (sl >> 2)) * VN + (es == 2 ? 2 * (sl & 3) + h : (sl & 3));
              thr = fmaxf(thr, list_insert(lv, li, K, lane, cv, cid));
            }
          }
        }
      }
      // every lane is done with the slot: refill it
      __syncwarp();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue_next(slot);
      // sum of exp(x - m): rescale once per stage when the lane's max grows
      if (tmax > m) {
        const float f = m == -CUDART_INF_F ? 0.f : ex2((m - tmax) * kLog2e);
        const float2 f2 = make_float2(f, f);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = __fmul2_rn(acc[i], f2);
        m = tmax;
      }
      exp_sum<T>(r, m, acc);
    }
    if (ab) break;
    // the piece's last logits past the 16-byte bulk copies (fewer than one vector)
    const int nb_el = static_cast<int>(p.nb / es);
    if (nb_el < p.n_el) {
      const bool has = lane < p.n_el - nb_el;
      const float xt = has ? to_f32<T>(logits[(long long)p.row * a.ld + p.v0 + nb_el + lane])
                           : -CUDART_INF_F;
      unsigned bal = __ballot_sync(0xffffffffu, has && xt >= thr);
      while (bal) {
        const int sl = __ffs(bal) - 1;
        bal &= bal - 1;
        const float cv = __shfl_sync(0xffffffffu, xt, sl);
        thr = fmaxf(thr, list_insert(lv, li, K, lane, cv, p.v0 + nb_el + sl));
      }
      if (xt > m) {
        const float f = m == -CUDART_INF_F ? 0.f : ex2((m - xt) * kLog2e);
        const float2 f2 = make_float2(f, f);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = __fmul2_rn(acc[i], f2);
        m = xt;
      }
      if (has) acc[0].x += ex2((xt - m) * kLog2e);
    }

    // ---- end of the piece: the warp's (max, sum), then its list ----
    float s = (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y) + (acc[2].x + acc[2].y) +
              (acc[3].x + acc[3].y);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      lse_merge(m, s, __shfl_xor_sync(0xffffffffu, m, off), __shfl_xor_sync(0xffffffffu, s, off));
    if (a.splits == 1) {
      const float lse = m + logf(s);
      if (lane < K) {
        a.ids[(long long)p.row * K + lane] = li;
        a.logp[(long long)p.row * K + lane] = lv - lse;
      }
      continue;
    }
    const int split = pc - p.row * a.splits;
    float* rec = a.part + ((long long)p.row * a.splits + split) * kRecStride;
    if (lane == 0) {
      rec[0] = m;
      rec[1] = s;
    }
    if (lane < 8) {
      rec[2 + lane] = lv;
      rec[2 + 32 + lane] = __int_as_float(li);
    }
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atomicAdd(&a.counters[p.row], 1) == a.splits - 1;
    if (!__shfl_sync(0xffffffffu, last, 0)) continue;
    __threadfence();
    // the last warp of the row: lane sp takes split sp's record (splits <= 32)
    const bool has = lane < a.splits;
    const float* my = a.part + ((long long)p.row * a.splits + (has ? lane : 0)) * kRecStride;
    float tv[8];
    int ti[8];
    m = has ? __ldcg(my) : -CUDART_INF_F;
    s = has ? __ldcg(my + 1) : 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      tv[q] = has ? __ldcg(my + 2 + q) : -CUDART_INF_F;
      ti[q] = has ? __float_as_int(__ldcg(my + 2 + 32 + q)) : 0x7fffffff;
    }
    tk_lane_merge(tv, ti, m, s, 1, 16);
    const float lse = m + logf(s);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < K && lane == q) {
        a.ids[(long long)p.row * K + q] = ti[q];
        a.logp[(long long)p.row * K + q] = tv[q] - lse;
      }
    if (lane == 0) a.counters[p.row] = 0;
  }
  if (ab) {
    // every copy this warp issued must land before it may exit: the ones past
    // the consumed stages, waited for in issue order (bounded)
    for (uint32_t sq = seq; sq < n_issued; ++sq)
      ptx::mbar_wait_bounded(&full[sq % kStages], (sq / kStages) & 1u, kTimeoutNs, nullptr);
  }
}

template <typename T>
void launch_stream_t(const TopkLaunch& a, cudaStream_t st) {
  StreamArgs s{};
  s.rows = a.rows;
  s.vocab = a.vocab;
  s.K = a.K;
  s.splits = a.splits;
  s.chunk = ceil_div(ceil_div(a.vocab, a.splits), 8) * 8;
  s.n_pieces = a.rows * a.splits;
  s.ld = a.ld;
  s.part = a.part;
  s.counters = a.counters;
  s.ids = a.ids;
  s.logp = a.logp;
  s.status = a.status;
  const int smem = kWarps * kStages * kStageBytes;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(topk_stream_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    attr = true;
  }
  const int grid = min(ceil_div(s.n_pieces, kWarps), 2 * num_sms());
  TraceScope ts("lse_topk", st);
  launch_k(topk_stream_kernel<T>, dim3(grid), dim3(kThreads), smem, st,
           static_cast<const T*>(a.logits), s);
}

}  // namespace

int topk_stream_workers() { return 2 * num_sms() * kWarps; }

bool topk_stream_supported(const TopkLaunch& a) {
  const int es = a.dtype == DFLASH_BF16 ? 2 : 4;
  return a.K >= 1 && a.K <= 8 && !(a.inv_t > 0.f) && a.splits >= 1 && a.splits <= 32 &&
         (reinterpret_cast<uintptr_t>(a.logits) % 16) == 0 && (a.ld * es) % 16 == 0;
}

void launch_topk_stream(const TopkLaunch& a, cudaStream_t st) {
  if (a.rows <= 0) return;
  if (a.dtype == DFLASH_BF16) launch_stream_t<__nv_bfloat16>(a, st);
  else launch_stream_t<float>(a, st);
}

}  // namespace dfl
