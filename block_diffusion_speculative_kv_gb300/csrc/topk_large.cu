// Log-softmax and top-K for K up to 1024 per row (step a6 in the exact mode of
// Lemma 1, K = min(B, |V|)).
//
// "Accelerating Speculative Decoding with Block Diffusion Draft Trees",
// section 3.4.4, Lemma 1: the best tree of budget B only uses, at each depth,
// tokens of rank at most B, so the top-min(B, |V|) lists make the construction
// exact.  The order is (logit desc, token id asc), as for small K.
//
// Design: the order (logit desc, id asc) is the order of one 64-bit key per
// element, the order-preserving bits of the logit above the complement of the
// id, and all keys of a row are distinct.  So "the K best" is "the keys at or
// above the K-th largest key", found by a radix select with no tie rule left
// to apply: eight-bit digits from the top, each pass over only the candidates
// that share the digits chosen so far (a pass emits the candidates of higher
// bins and keeps those of the chosen bin), stopping once the kept candidates
// are exactly the ones still needed.
//   kernel 1: one CTA per (row, chunk of 16384 logits): the chunk's keys in
//             shared memory, its (max, sum of exp), its best min(K, chunk)
//             keys to a partial record (unsorted);
//   kernel 2: one CTA per row: the partial records' keys in shared memory, the
//             best K of them, a bitonic sort of those, and log-probabilities
//             from the merged (max, sum of exp).
#include <math_constants.h>

#include "common.cuh"
#include "kernels.h"

namespace dfl {

namespace {

constexpr int kLgThreads = 1024;
constexpr int kLgChunk = 16384;
constexpr float kLgLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint64_t rank_key(uint32_t ordered, int id) {
  return (static_cast<uint64_t>(ordered) << 32) | static_cast<uint64_t>(~static_cast<uint32_t>(id));
}

__device__ __forceinline__ void lg_merge(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -CUDART_INF_F) { m = M; s = 0.f; return; }
  const float a = (m == -CUDART_INF_F) ? 0.f : s * exp2f((m - M) * kLgLog2e);
  const float b = (m2 == -CUDART_INF_F) ? 0.f : s2 * exp2f((m2 - M) * kLgLog2e);
  m = M;
  s = a + b;
}

// Block-wide selection of the k largest among nc distinct 64-bit keys
// (1 <= k <= nc).  Candidates are indices into the caller's arrays; pass 0
// takes 0..nc-1 directly.  Each pass histograms the next eight key bits of the
// candidates (all of which share the bits above), finds the bin holding the
// k-th largest, hands every candidate of a higher bin to emit(idx) and keeps
// the candidates of that bin for the next pass; once the kept candidates are
// exactly the ones still needed they are all emitted.  emit is called exactly
// k times, in no particular order.  Every thread of the block calls this.
template <typename KeyF, typename EmitF>
__device__ void block_topk(int nc, int k, uint16_t* cand_a, uint16_t* cand_b, KeyF key,
                           EmitF emit, int* hist, int* misc) {
  const int tid = threadIdx.x, T = blockDim.x, lane = tid & 31, warp = tid >> 5;
  bool identity = true;
  for (int pass = 0; pass < 8; ++pass) {
    if (nc == k) {
      for (int c = tid; c < nc; c += T) emit(identity ? c : static_cast<int>(cand_a[c]));
      return;
    }
    const int shift = 56 - 8 * pass;
    for (int i = tid; i < 256; i += T) hist[i] = 0;
    if (tid == 0) misc[3] = 0;
    __syncthreads();
    for (int base = tid - lane; base < nc; base += T) {
      const int c = base + lane;
      int bin = 256 + lane;   // no bin: a lane past the end
      if (c < nc) bin = static_cast<int>((key(identity ? c : cand_a[c]) >> shift) & 255u);
      // lanes with the same bin add once
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (bin < 256 && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      int cnt[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) { cnt[j] = hist[255 - 8 * lane - j]; sum += cnt[j]; }
      int incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      int run = incl - sum;   // candidates in bins above this lane's
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (run < k && run + cnt[j] >= k) {
          misc[0] = 255 - 8 * lane - j;
          misc[1] = run;
          misc[2] = cnt[j];
        }
        run += cnt[j];
      }
    }
    __syncthreads();
    const int b = misc[0], above = misc[1], in_bin = misc[2];
    for (int c = tid; c < nc; c += T) {
      const int idx = identity ? c : static_cast<int>(cand_a[c]);
      const int d = static_cast<int>((key(idx) >> shift) & 255u);
      if (d > b) emit(idx);
      else if (d == b) cand_b[atomicAdd(&misc[3], 1)] = static_cast<uint16_t>(idx);
    }
    __syncthreads();
    k -= above;
    nc = in_bin;
    uint16_t* t = cand_a;
    cand_a = cand_b;
    cand_b = t;
    identity = false;
  }
  // all 64 bits resolved: the keys are distinct, so one candidate is left
  for (int c = tid; c < nc && c < k; c += T) emit(static_cast<int>(cand_a[c]));
}

__device__ __forceinline__ void block_ms(float& m, float& s, float* s_m, float* s_s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
    lg_merge(m, s, m2, s2);
  }
  if (lane == 0) { s_m[warp] = m; s_s[warp] = s; }
  __syncthreads();
  if (warp == 0) {
    m = lane < (int)(blockDim.x >> 5) ? s_m[lane] : -CUDART_INF_F;
    s = lane < (int)(blockDim.x >> 5) ? s_s[lane] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
      lg_merge(m, s, m2, s2);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kLgThreads)
topk_large_part_kernel(const T* __restrict__ logits, long long ld, int vocab, int K, int splits,
                       int chunk, float* __restrict__ pv, int* __restrict__ pi,
                       float2* __restrict__ pms) {
  extern __shared__ __align__(16) uint32_t skey[];   // [kLgChunk] keys, then 2 x [kLgChunk] u16
  uint16_t* cand_a = reinterpret_cast<uint16_t*>(skey + kLgChunk);
  uint16_t* cand_b = cand_a + kLgChunk;
  __shared__ int hist[256];
  __shared__ int misc[4];
  __shared__ float s_m[32], s_s[32];
  __shared__ int s_cnt;
  constexpr int kPer = kLgChunk / kLgThreads;
  const int row = blockIdx.x / splits, split = blockIdx.x % splits;
  const int tid = threadIdx.x;
  const int v0 = split * chunk;
  const int n = min(chunk, vocab - v0);
  const T* rp = logits + (long long)row * ld + v0;
  pdl_wait();
  pdl_trigger();
  // all of a thread's loads in flight together, then the (max, sum of exp)
  float x[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = tid + j * kLgThreads;
    x[j] = i < n ? to_f32<T>(rp[i]) : -CUDART_INF_F;
  }
  float m = -CUDART_INF_F;
#pragma unroll
  for (int j = 0; j < kPer; ++j) m = fmaxf(m, x[j]);
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = tid + j * kLgThreads;
    if (i < n) skey[i] = ordered_bits(x[j]);
    if (x[j] != -CUDART_INF_F) s += exp2f((x[j] - m) * kLgLog2e);
  }
  block_ms(m, s, s_m, s_s);
  const size_t rec = (size_t)row * splits + split;
  if (tid == 0) {
    pms[rec] = make_float2(m, s);
    s_cnt = 0;
  }
  __syncthreads();
  float* ov = pv + rec * K;
  int* oi = pi + rec * K;
  block_topk(n, min(K, n), cand_a, cand_b,
             [&](int i) { return rank_key(skey[i], v0 + i); },
             [&](int i) {
               const int slot = atomicAdd(&s_cnt, 1);
               ov[slot] = from_ordered_bits(skey[i]);
               oi[slot] = v0 + i;
             },
             hist, misc);
}

__global__ void __launch_bounds__(kLgThreads)
topk_large_merge_kernel(int vocab, int K, int splits, int chunk, const float* __restrict__ pv,
                        const int* __restrict__ pi, const float2* __restrict__ pms,
                        int32_t* __restrict__ ids_out, float* __restrict__ logp_out) {
  extern __shared__ __align__(16) uint32_t smem2[];
  __shared__ int hist[256];
  __shared__ int misc[4];
  __shared__ float s_m[32], s_s[32];
  __shared__ int s_cnt;
  __shared__ float s_lse;
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int ck = min(K, chunk);                                   // records of a full chunk
  const int n_last = vocab - (splits - 1) * chunk;
  const int N = (splits - 1) * ck + min(K, n_last);
  int P = 1;
  while (P < K) P <<= 1;
  uint64_t* win = reinterpret_cast<uint64_t*>(smem2);             // [P] winners, sorted here
  uint32_t* ckey = smem2 + 2 * P;                                 // [N]
  int* cid = reinterpret_cast<int*>(ckey + N);                    // [N]
  uint16_t* cand_a = reinterpret_cast<uint16_t*>(cid + N);        // [N]
  uint16_t* cand_b = cand_a + N;                                  // [N]
  pdl_wait();
  pdl_trigger();
  for (int e = tid; e < N; e += kLgThreads) {
    const int sp = e / ck, j = e - sp * ck;
    const size_t at = ((size_t)row * splits + sp) * K + j;
    ckey[e] = ordered_bits(__ldcg(pv + at));
    cid[e] = __ldcg(pi + at);
  }
  for (int i = K + tid; i < P; i += kLgThreads) win[i] = 0ull;   // below every real key
  float m = -CUDART_INF_F, s = 0.f;
  for (int sp = tid; sp < splits; sp += kLgThreads) {
    const float2 ms = __ldcg(pms + (size_t)row * splits + sp);
    lg_merge(m, s, ms.x, ms.y);
  }
  block_ms(m, s, s_m, s_s);
  if (tid == 0) {
    s_lse = m + logf(s);
    s_cnt = 0;
  }
  __syncthreads();
  block_topk(N, K, cand_a, cand_b, [&](int i) { return rank_key(ckey[i], cid[i]); },
             [&](int i) { win[atomicAdd(&s_cnt, 1)] = rank_key(ckey[i], cid[i]); }, hist, misc);
  __syncthreads();
  // bitonic sort of the P winner keys, descending
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P; i += kLgThreads) {
        const int j = i ^ stride;
        if (j > i) {
          const uint64_t a = win[i], b = win[j];
          const bool desc = (i & size) == 0;
          if (desc ? a < b : a > b) { win[i] = b; win[j] = a; }
        }
      }
      __syncthreads();
    }
  }
  const float lse = s_lse;
  for (int r = tid; r < K; r += kLgThreads) {
    const uint64_t w = win[r];
    ids_out[(size_t)row * K + r] = static_cast<int32_t>(~static_cast<uint32_t>(w));
    logp_out[(size_t)row * K + r] = from_ordered_bits(static_cast<uint32_t>(w >> 32)) - lse;
  }
}

}  // namespace

int topk_large_splits(int vocab) { return ceil_div(vocab, kLgChunk); }

size_t topk_large_part_bytes(int rows, int vocab, int K) {
  const size_t recs = (size_t)rows * topk_large_splits(vocab);
  return align_up(recs * K * sizeof(float), 256) + align_up(recs * K * sizeof(int), 256) +
         align_up(recs * sizeof(float2), 256);
}

size_t topk_large_merge_smem(int vocab, int K) {
  const int splits = topk_large_splits(vocab);
  const int chunk = kLgChunk;
  const int ck = K < chunk ? K : chunk;
  const int n_last = vocab - (splits - 1) * chunk;
  const size_t N = (size_t)(splits - 1) * ck + (K < n_last ? K : n_last);
  size_t P = 1;
  while (P < (size_t)K) P <<= 1;
  if (N > 65535) return (size_t)1 << 40;   // candidate indices are 16-bit
  return sizeof(uint64_t) * P + (sizeof(uint32_t) + sizeof(int) + 2 * sizeof(uint16_t)) * N;
}

dflash_status launch_topk_large(const TopkLaunch& a, void* part, cudaStream_t st) {
  if (a.rows <= 0) return DFLASH_OK;
  const int splits = topk_large_splits(a.vocab);
  const size_t smem2 = topk_large_merge_smem(a.vocab, a.K);
  if (smem2 > 200 * 1024)
    return set_error(DFLASH_ERR_UNSUPPORTED, "top-%d over a vocabulary of %d needs %zu bytes of "
                     "shared memory in the merge", a.K, a.vocab, smem2);
  const size_t recs = (size_t)a.rows * splits;
  char* p = static_cast<char*>(part);
  float* pv = reinterpret_cast<float*>(p);
  int* pi = reinterpret_cast<int*>(p + align_up(recs * a.K * sizeof(float), 256));
  float2* pms = reinterpret_cast<float2*>(p + align_up(recs * a.K * sizeof(float), 256) +
                                          align_up(recs * a.K * sizeof(int), 256));
  const size_t smem1 = (sizeof(uint32_t) + 2 * sizeof(uint16_t)) * kLgChunk;
  static bool attr = false;   // per process
  if (!attr) {
    cudaFuncSetAttribute(topk_large_part_kernel<float>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
    cudaFuncSetAttribute(topk_large_part_kernel<__nv_bfloat16>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
    cudaFuncSetAttribute(topk_large_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         200 * 1024);
    attr = true;
  }
  {
    TraceScope ts("lse_topk_large", st);
    if (a.dtype == DFLASH_BF16)
      launch_k(topk_large_part_kernel<__nv_bfloat16>, dim3(a.rows * splits), dim3(kLgThreads),
               smem1, st, static_cast<const __nv_bfloat16*>(a.logits), a.ld, a.vocab, a.K, splits,
               kLgChunk, pv, pi, pms);
    else
      launch_k(topk_large_part_kernel<float>, dim3(a.rows * splits), dim3(kLgThreads), smem1, st,
               static_cast<const float*>(a.logits), a.ld, a.vocab, a.K, splits, kLgChunk, pv, pi,
               pms);
  }
  TraceScope ts("lse_topk_large_merge", st);
  launch_k(topk_large_merge_kernel, dim3(a.rows), dim3(kLgThreads), smem2, st, a.vocab, a.K,
           splits, kLgChunk, pv, pi, pms, a.ids, a.logp);
  return DFLASH_OK;
}

}  // namespace dfl
