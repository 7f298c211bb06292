// Block attention of the drafter (step a4, attention part).
//
// "DFlash: Block Diffusion for Flash Speculative Decoding", section 3.4.4: the
// block's queries attend bidirectionally within the block and to the target
// context injected into the layer's KV cache (section 3.4.3).  With grouped
// query attention, the G = n_q / n_kv query heads of a KV head share its keys,
// so a KV head's work is G * L query rows (64 for 32/8 heads and L = 16).
//
// bf16 path (split-KV): grid (chunk, kv head, request), sized to one wave.
// Chunk c covers context positions [c*chunk, (c+1)*chunk) of the request
// (empty chunks past ctx_len exit at once); the last chunk also takes the
// block's own L keys as one extra tile.  A CTA keeps its query rows in shared memory, streams 64-key
// tiles of K and V through a double-buffered cp.async ring (XOR-swizzled 16 B
// chunks, conflict-free for ldmatrix), computes S = Q K^T and O += P V with
// bf16 mma.sync (fp32 accumulators) and an online softmax in base 2, and
// writes an unnormalised partial (O, running max, running sum).  A second
// kernel merges the partials of each (request, KV head) with the usual
// log-sum-exp rescaling and writes bf16 outputs.
//
// fp32 path: one warp per query row, lanes over the head dimension, every key
// in turn with an online softmax (used for fp32 models).
#include "attention.h"
#include "common.cuh"
#include "mma_sync.cuh"

#include <math_constants.h>

namespace dfl {

namespace {

using namespace mmas;

constexpr int kKeyTile = 64;
constexpr int kStages = 6;   // K/V tiles in flight per CTA (~192 KB at head_dim 128)

template <int HD>
__global__ void __launch_bounds__(256, 1)
attn_split_kernel(const AttnParams p) {
  constexpr int NCH = HD / 8;  // 16-byte chunks per row
  extern __shared__ __align__(128) uint8_t smem[];
  const int QR = p.G * p.L;
  const int QRp = (QR + 15) / 16 * 16;
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + QRp * HD * 2;
  uint8_t* sV = sK + kStages * kKeyTile * HD * 2;

  const int chunk_id = blockIdx.x;
  const int g = blockIdx.y;
  const int req = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const bool has_block = chunk_id == p.n_chunks - 1;
  const int ctx = min(max(p.ctx_len[req], 0), p.cap);  // never read past the cache slab
  const int k_begin = chunk_id * p.chunk;
  const int k_end = min(ctx, k_begin + p.chunk);
  const int nct = k_end > k_begin ? (k_end - k_begin + kKeyTile - 1) / kKeyTile : 0;

  const size_t part_row0 = (((size_t)req * p.n_kv + g) * p.n_chunks + chunk_id) * QR;
  if (nct == 0 && !has_block) {
    pdl_wait();
    pdl_trigger();
    for (int r = tid; r < QR; r += blockDim.x) {
      p.part_ml[(part_row0 + r) * 2 + 0] = -CUDART_INF_F;
      p.part_ml[(part_row0 + r) * 2 + 1] = 0.f;
    }
    return;
  }

  const __nv_bfloat16* cbase_k = p.cache_k + ((size_t)req * p.n_kv + g) * p.cap * HD;
  const __nv_bfloat16* cbase_v = p.cache_v + ((size_t)req * p.n_kv + g) * p.cap * HD;
  const __nv_bfloat16* bbase_k = p.qkv + (size_t)req * p.L * p.qkv_ld + (size_t)(p.n_q + g) * HD;
  const __nv_bfloat16* bbase_v =
      p.qkv + (size_t)req * p.L * p.qkv_ld + (size_t)(p.n_q + p.n_kv + g) * HD;

  // tile t < nct: context keys k_begin + 64t ...; tile nct (last chunk only):
  // the block's L keys, read from the QKV output
  auto load_tile = [&](int buf, int t) {
    uint8_t* dK = sK + buf * kKeyTile * HD * 2;
    uint8_t* dV = sV + buf * kKeyTile * HD * 2;
    const bool blk = t >= nct;
    const int key0 = blk ? 0 : k_begin + t * kKeyTile;
    const int kend = blk ? p.L : k_end;
    const __nv_bfloat16* kb = blk ? bbase_k : cbase_k;
    const __nv_bfloat16* vb = blk ? bbase_v : cbase_v;
    const long long ld = blk ? p.qkv_ld : HD;
    for (int i = tid; i < kKeyTile * NCH; i += blockDim.x) {
      const int r = i / NCH, ch = i % NCH;
      const int key = key0 + r;
      const bool valid = key < kend;
      const size_t off = (size_t)(valid ? key : key0) * ld + ch * 8;
      cp_async16(smem_u32(dK) + swz<HD>(r, ch), kb + off, valid);
      cp_async16(smem_u32(dV) + swz<HD>(r, ch), vb + off, valid);
    }
  };
  const int ntiles = nct + (has_block ? 1 : 0);
  // Two groups of four warps take alternate tiles (group 0 even, group 1 odd)
  // from one ring; each warp owns 16 query rows.  kStages-2 tiles run ahead.
  constexpr int kAhead = kStages - 2;
  const int npre = ntiles < kAhead ? ntiles : kAhead;
  // The context part of the cache is written only by the injection, several
  // kernels back: the first context tiles are requested before waiting for
  // the QKV GEMM, the block tile after.  Each tile is its own cp.async group.
  int issued = 0;
  while (issued < npre && issued < nct) {
    load_tile(issued, issued);
    cp_async_commit();
    ++issued;
  }
  pdl_wait();
  pdl_trigger();

  // ---- stage Q (rows: head g*G + r/L, token r%L) ----
  for (int i = tid; i < QRp * NCH; i += blockDim.x) {
    const int r = i / NCH, ch = i % NCH;
    const bool valid = r < QR;
    const int h = g * p.G + (valid ? r / p.L : 0);
    const int j = valid ? r % p.L : 0;
    const __nv_bfloat16* src = p.qkv + ((size_t)req * p.L + j) * p.qkv_ld + (size_t)h * HD + ch * 8;
    cp_async16(smem_u32(sQ) + swz<HD>(r, ch), src, valid);
  }
  cp_async_commit();   // Q in its own group
  while (issued < npre) {   // a block tile among the first ring slots
    load_tile(issued, issued);
    cp_async_commit();
    ++issued;
  }

  const int grp = warp >> 2;
  const int qrow0 = (warp & 3) * 16;
  const bool warp_active = qrow0 < QR;
  const int gq = lane >> 2, tq = lane & 3;
  float o[HD / 8][4];
#pragma unroll
  for (int n = 0; n < HD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  uint32_t qa[HD / 16][4];

  for (int it = 0; 2 * it < ntiles; ++it) {
    // issue the two tiles kAhead ahead (their buffers were last read in
    // iteration it-1, released by that iteration's closing barrier)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int tn = 2 * it + npre + e;
      if (tn < ntiles) load_tile(tn % kStages, tn);
      cp_async_commit();
    }
    // groups complete in commit order.  In the first iteration Q sits among
    // the first groups: wait for all but the two groups just committed.
    // Later, tiles 2it and 2it+1 have at most kAhead newer groups.
    if (it == 0) cp_async_wait<2>();
    else cp_async_wait<kAhead>();
    __syncthreads();
    const int t = 2 * it + grp;
    if (it == 0 && warp_active) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const int r = qrow0 + (lane & 15);
        const int ch = kk * 2 + (lane >> 4);
        ldsm_x4(smem_u32(sQ) + swz<HD>(r, ch), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
      }
    }
    if (warp_active && t < ntiles) {
      const bool blk = t >= nct;
      const int key0 = blk ? 0 : k_begin + t * kKeyTile;
      const int kend = blk ? p.L : k_end;
      const uint32_t kb = smem_u32(sK + (t % kStages) * kKeyTile * HD * 2);
      const uint32_t vb = smem_u32(sV + (t % kStages) * kKeyTile * HD * 2);
      float s[kKeyTile / 8][4];
#pragma unroll
      for (int n = 0; n < kKeyTile / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
      // S = Q K^T
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
        for (int np = 0; np < kKeyTile / 16; ++np) {
          const int r = np * 16 + ((lane >> 4) << 3) + (lane & 7);
          const int ch = kk * 2 + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + swz<HD>(r, ch), b0, b1, b2, b3);
          mma16816(s[2 * np], qa[kk], b0, b1);
          mma16816(s[2 * np + 1], qa[kk], b2, b3);
        }
      }
      // scale, mask, online softmax (base 2)
      const int rq0 = qrow0 + gq, rq1 = rq0 + 8;
      const bool iso0 = blk && !p.anchor_sees_block && (rq0 % p.L) == 0;
      const bool iso1 = blk && !p.anchor_sees_block && (rq1 % p.L) == 0;
      float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
      for (int n = 0; n < kKeyTile / 8; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = key0 + n * 8 + 2 * tq + e;
          const bool ok = key < kend;
          float v0 = s[n][e] * p.scale_log2;
          float v1 = s[n][2 + e] * p.scale_log2;
          if (!ok || (iso0 && key > 0)) v0 = -CUDART_INF_F;
          if (!ok || (iso1 && key > 0)) v1 = -CUDART_INF_F;
          s[n][e] = v0;
          s[n][2 + e] = v1;
          mx0 = fmaxf(mx0, v0);
          mx1 = fmaxf(mx1, v1);
        }
      }
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float base0 = (mn0 == -CUDART_INF_F) ? 0.f : mn0;
      const float base1 = (mn1 == -CUDART_INF_F) ? 0.f : mn1;
      const float c0 = exp2f(m0 - base0), c1 = exp2f(m1 - base1);
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int n = 0; n < kKeyTile / 8; ++n) {
        s[n][0] = exp2f(s[n][0] - base0);
        s[n][1] = exp2f(s[n][1] - base0);
        s[n][2] = exp2f(s[n][2] - base1);
        s[n][3] = exp2f(s[n][3] - base1);
        rs0 += s[n][0] + s[n][1];
        rs1 += s[n][2] + s[n][3];
      }
      l0 = l0 * c0 + rs0;
      l1 = l1 * c1 + rs1;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int n = 0; n < HD / 8; ++n) {
        o[n][0] *= c0; o[n][1] *= c0;
        o[n][2] *= c1; o[n][3] *= c1;
      }
      // O += P V
#pragma unroll
      for (int kk = 0; kk < kKeyTile / 16; ++kk) {
        uint32_t pa[4];
        pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
        pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
        pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < HD / 16; ++dp) {
          const int r = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int ch = dp * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + swz<HD>(r, ch), b0, b1, b2, b3);
          mma16816(o[2 * dp], pa, b0, b1);
          mma16816(o[2 * dp + 1], pa, b2, b3);
        }
      }
    }
    __syncthreads();
  }

  // row sums: reduce over the quad (each group its own)
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  // ---- merge the two groups' states (group 1 -> shared memory -> group 0) ----
  float* mo = reinterpret_cast<float*>(sK);   // [QRp][HD]; the ring is free now
  float* mml = mo + QRp * HD;                   // [QRp][2] running max and sum
  if (grp == 1 && warp_active) {
    const int rq0 = qrow0 + gq, rq1 = rq0 + 8;
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) {
      const int dc = n * 8 + 2 * tq;
      mo[rq0 * HD + dc] = o[n][0];
      mo[rq0 * HD + dc + 1] = o[n][1];
      mo[rq1 * HD + dc] = o[n][2];
      mo[rq1 * HD + dc + 1] = o[n][3];
    }
    if (tq == 0) {
      mml[rq0 * 2] = m0; mml[rq0 * 2 + 1] = l0;
      mml[rq1 * 2] = m1; mml[rq1 * 2 + 1] = l1;
    }
  }
  __syncthreads();
  if (grp == 1) return;
  if (warp_active) {
    const int rq0 = qrow0 + gq, rq1 = rq0 + 8;
    const float om0 = mml[rq0 * 2], ol0 = mml[rq0 * 2 + 1];
    const float om1 = mml[rq1 * 2], ol1 = mml[rq1 * 2 + 1];
    const float nm0 = fmaxf(m0, om0), nm1 = fmaxf(m1, om1);
    const float b0 = (nm0 == -CUDART_INF_F) ? 0.f : nm0;
    const float b1 = (nm1 == -CUDART_INF_F) ? 0.f : nm1;
    const float a0 = exp2f(m0 - b0), c0 = exp2f(om0 - b0);
    const float a1 = exp2f(m1 - b1), c1 = exp2f(om1 - b1);
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) {
      const int dc = n * 8 + 2 * tq;
      o[n][0] = o[n][0] * a0 + mo[rq0 * HD + dc] * c0;
      o[n][1] = o[n][1] * a0 + mo[rq0 * HD + dc + 1] * c0;
      o[n][2] = o[n][2] * a1 + mo[rq1 * HD + dc] * c1;
      o[n][3] = o[n][3] * a1 + mo[rq1 * HD + dc + 1] * c1;
    }
    l0 = l0 * a0 + ol0 * c0;
    l1 = l1 * a1 + ol1 * c1;
    m0 = nm0;
    m1 = nm1;
  }
  if (warp_active) {
    const int rq0 = qrow0 + gq, rq1 = rq0 + 8;
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) {
      const int d = n * 8 + 2 * tq;
      if (rq0 < QR) {
        float2* dst = reinterpret_cast<float2*>(p.part_o + (part_row0 + rq0) * HD + d);
        *dst = make_float2(o[n][0], o[n][1]);
      }
      if (rq1 < QR) {
        float2* dst = reinterpret_cast<float2*>(p.part_o + (part_row0 + rq1) * HD + d);
        *dst = make_float2(o[n][2], o[n][3]);
      }
    }
    if (tq == 0) {
      if (rq0 < QR) {
        p.part_ml[(part_row0 + rq0) * 2 + 0] = m0;
        p.part_ml[(part_row0 + rq0) * 2 + 1] = l0;
      }
      if (rq1 < QR) {
        p.part_ml[(part_row0 + rq1) * 2 + 0] = m1;
        p.part_ml[(part_row0 + rq1) * 2 + 1] = l1;
      }
    }
  }
  (void)nwarps;
}

// Merge the partials of one (request, KV head) with log-sum-exp rescaling: a
// warp per query row (4 rows per CTA), lanes over the head dimension.  Up to
// kAllParts chunks: every partial (max, sum and output slice) is loaded at
// once and the maximum taken from the loaded values, one round trip in all.
// More chunks: the maxima are gathered first, then the rescaled partials are
// accumulated with U chunks' loads in flight.
constexpr int kAllParts = 24;

template <int HD>
__global__ void __launch_bounds__(128)
attn_combine_kernel(const AttnParams p) {
  const int QR = p.G * p.L;
  const int req = blockIdx.z, g = blockIdx.y;
  const int r = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  if (r >= QR) return;
  const int nparts = p.n_chunks;
  const size_t base = ((size_t)req * p.n_kv + g) * nparts * QR;
  constexpr int DPL = HD / 32;
  static_assert(DPL == 4 || DPL == 2, "head_dim 128 or 64");
  float acc[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
  float Lsum = 0.f;
  auto load_o = [&](size_t row, bool live, float (&v)[DPL]) {
    const float* src = p.part_o + row * HD + lane * DPL;
    if constexpr (DPL == 4) {
      const float4 t = live ? *reinterpret_cast<const float4*>(src) : make_float4(0.f, 0.f, 0.f, 0.f);
      v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
      const float2 t = live ? *reinterpret_cast<const float2*>(src) : make_float2(0.f, 0.f);
      v[0] = t.x; v[1] = t.y;
    }
  };
  if (nparts <= kAllParts) {
    float m[kAllParts], l[kAllParts], v[kAllParts][DPL];
#pragma unroll
    for (int u = 0; u < kAllParts; ++u) {
      const bool in = u < nparts;
      const size_t row = base + (size_t)(in ? u : 0) * QR + r;
      const float2 ml = in ? *reinterpret_cast<const float2*>(p.part_ml + row * 2)
                           : make_float2(-CUDART_INF_F, 0.f);
      m[u] = ml.x;
      l[u] = ml.y;
      // (an empty chunk writes no output slice: loaded here, never used)
      load_o(row, in, v[u]);
    }
    float M = -CUDART_INF_F;
#pragma unroll
    for (int u = 0; u < kAllParts; ++u)
      if (l[u] > 0.f) M = fmaxf(M, m[u]);
#pragma unroll
    for (int u = 0; u < kAllParts; ++u) {
      if (l[u] > 0.f) {
        const float w = exp2f(m[u] - M);
        Lsum += w * l[u];
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] += w * v[u][i];
      }
    }
  } else {
    float M = -CUDART_INF_F;
    for (int c0 = 0; c0 < nparts; c0 += 32) {
      const int c = c0 + lane;
      if (c < nparts) {
        const size_t row = base + (size_t)c * QR + r;
        if (p.part_ml[row * 2 + 1] > 0.f) M = fmaxf(M, p.part_ml[row * 2]);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    constexpr int U = 8;   // chunk partials in flight per lane (16 B each)
    for (int c0 = 0; c0 < nparts; c0 += U) {
      float w[U], l[U], v[U][DPL];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u;
        const size_t row = base + (size_t)(c < nparts ? c : 0) * QR + r;
        const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + row * 2);
        l[u] = (c < nparts) ? ml.y : 0.f;
        w[u] = (l[u] > 0.f) ? exp2f(ml.x - M) : 0.f;
        load_o(row, l[u] > 0.f, v[u]);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        Lsum += w[u] * l[u];
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] += w[u] * v[u][i];
      }
    }
  }
  // (a row that saw no key at all, a tree node past the last one, gets zeros)
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  const int h = g * p.G + r / p.L, j = r % p.L;
  // blockIdx.z: a request, or with query tiles (tree attention) a (request,
  // tile) pair whose rows are nodes tile * L + j of out_rows per request
  size_t orow = (size_t)req * p.L + j;
  if (p.n_qt > 0) {
    const int node = (req % p.n_qt) * p.L + j;
    if (node >= p.out_rows) return;
    orow = (size_t)(req / p.n_qt) * p.out_rows + node;
  }
  __nv_bfloat16* dst = p.out + orow * p.out_ld + (size_t)h * HD + lane * DPL;
#pragma unroll
  for (int i = 0; i < DPL; ++i) dst[i] = __float2bfloat16_rn(acc[i] * inv);
}

// The same merge for at most kFewParts chunks (many requests: few chunks per
// request): a warp merges kRowsPerWarp rows of the flattened (request, KV head,
// query row) space, every row's partials loaded before any is combined, so
// that one round trip serves several rows.
constexpr int kFewParts = 4;
constexpr int kRowsPerWarp = 4;

template <int HD>
__global__ void __launch_bounds__(128)
attn_combine_few_kernel(const AttnParams p) {
  constexpr int DPL = HD / 32;
  const int QR = p.G * p.L;
  const int lane = threadIdx.x & 31;
  const long long total = (long long)p.n_req * p.n_kv * QR;
  const long long row0 = ((long long)blockIdx.x * 4 + (threadIdx.x >> 5)) * kRowsPerWarp;
  pdl_wait();
  pdl_trigger();
  const int np = p.n_chunks;
  float m[kRowsPerWarp][kFewParts], l[kRowsPerWarp][kFewParts];
  float v[kRowsPerWarp][kFewParts][DPL];
#pragma unroll
  for (int j = 0; j < kRowsPerWarp; ++j) {
    const long long w = row0 + j;
    const bool live = w < total;
    const long long ww = live ? w : 0;
    const long long unit_g = ww / QR;          // request * n_kv + KV head
    const int r = static_cast<int>(ww - unit_g * QR);
    const size_t base = (size_t)unit_g * np * QR + r;
#pragma unroll
    for (int u = 0; u < kFewParts; ++u) {
      const bool in = live && u < np;
      const size_t row = base + (size_t)(in ? u : 0) * QR;
      const float2 ml = in ? *reinterpret_cast<const float2*>(p.part_ml + row * 2)
                           : make_float2(-CUDART_INF_F, 0.f);
      m[j][u] = ml.x;
      l[j][u] = ml.y;
      const float* src = p.part_o + row * HD + lane * DPL;
      if constexpr (DPL == 4) {
        const float4 t = in ? *reinterpret_cast<const float4*>(src) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[j][u][0] = t.x; v[j][u][1] = t.y; v[j][u][2] = t.z; v[j][u][3] = t.w;
      } else {
        const float2 t = in ? *reinterpret_cast<const float2*>(src) : make_float2(0.f, 0.f);
        v[j][u][0] = t.x; v[j][u][1] = t.y;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kRowsPerWarp; ++j) {
    const long long w = row0 + j;
    if (w >= total) break;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int u = 0; u < kFewParts; ++u)
      if (l[j][u] > 0.f) M = fmaxf(M, m[j][u]);
    float acc[DPL], Lsum = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
#pragma unroll
    for (int u = 0; u < kFewParts; ++u) {
      if (l[j][u] > 0.f) {
        const float wt = exp2f(m[j][u] - M);
        Lsum += wt * l[j][u];
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] += wt * v[j][u][i];
      }
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    const long long unit_g = w / QR;
    const int r = static_cast<int>(w - unit_g * QR);
    const int req = static_cast<int>(unit_g / p.n_kv), g = static_cast<int>(unit_g % p.n_kv);
    const int h = g * p.G + r / p.L, jj = r % p.L;
    __nv_bfloat16* dst = p.out + ((size_t)req * p.L + jj) * p.out_ld + (size_t)h * HD + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; ++i) dst[i] = __float2bfloat16_rn(acc[i] * inv);
  }
}

// fp32 reference-precision path: one warp per (request, query head, token).
template <int HD>
__global__ void __launch_bounds__(128)
attn_f32_kernel(const AttnParamsF32 p) {
  constexpr int DPL = HD / 32;
  const int wid = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int total = p.n_req * p.n_q * p.L;
  pdl_wait();
  pdl_trigger();
  if (wid >= total) return;
  const int j = wid % p.L;
  const int h = (wid / p.L) % p.n_q;
  const int req = wid / (p.L * p.n_q);
  const int g = h / (p.n_q / p.n_kv);
  const int ctx = min(max(p.ctx_len[req], 0), p.cap);
  const float* q = p.qkv + ((size_t)req * p.L + j) * p.qkv_ld + (size_t)h * HD;
  float qv[DPL], o[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) { qv[i] = q[lane + 32 * i]; o[i] = 0.f; }
  float m = -CUDART_INF_F, l = 0.f;
  const float scale = rsqrtf(static_cast<float>(HD));
  const bool iso = !p.anchor_sees_block && j == 0;
  const int nkeys = ctx + (iso ? 1 : p.L);
  for (int s = 0; s < nkeys; ++s) {
    const float* kr;
    const float* vr;
    if (s < ctx) {
      const size_t off = (((size_t)req * p.n_kv + g) * p.cap + s) * HD;
      kr = p.cache_k + off;
      vr = p.cache_v + off;
    } else {
      const int jj = s - ctx;
      kr = p.qkv + ((size_t)req * p.L + jj) * p.qkv_ld + (size_t)(p.n_q + g) * HD;
      vr = p.qkv + ((size_t)req * p.L + jj) * p.qkv_ld + (size_t)(p.n_q + p.n_kv + g) * HD;
    }
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) part = fmaf(qv[i], kr[lane + 32 * i], part);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    const float sc = part * scale;
    const float mn = fmaxf(m, sc);
    const float corr = expf(m - mn);
    const float pw = expf(sc - mn);
    l = l * corr + pw;
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[i] = o[i] * corr + pw * vr[lane + 32 * i];
    m = mn;
  }
  float* dst = p.out + ((size_t)req * p.L + j) * p.out_ld + (size_t)h * HD;
#pragma unroll
  for (int i = 0; i < DPL; ++i) dst[lane + 32 * i] = o[i] / l;
}

}  // namespace

void launch_attn_combine(const AttnParams& p, int head_dim, dim3 cgrid, cudaStream_t st) {
  TraceScope ts("attn_combine", st);
  if (head_dim == 128) launch_k(attn_combine_kernel<128>, cgrid, dim3(128), 0, st, p);
  else launch_k(attn_combine_kernel<64>, cgrid, dim3(128), 0, st, p);
}

int attn_chunk(int max_ctx, int n_kv, int n_req) {
  // One CTA per SM holds a deep ring: when a wave covers every (request, KV
  // head) pair, size the chunks so the whole grid is one wave; otherwise aim
  // for several waves of short chunks so ragged contexts balance.
  const long long sms = num_sms();
  const long long pairs = (long long)n_kv * n_req;
  long long n_chunks = pairs <= sms ? sms / pairs : (4 * sms + pairs - 1) / pairs;
  if (n_chunks < 1) n_chunks = 1;
  long long c = (max_ctx + n_chunks - 1) / n_chunks;
  c = (c + kKeyTile - 1) / kKeyTile * kKeyTile;
  if (c < kKeyTile) c = kKeyTile;
  return static_cast<int>(c);
}

size_t attn_smem_bytes(int G, int L, int HD) {
  const int QRp = (G * L + 15) / 16 * 16;
  return (size_t)QRp * HD * 2 + 2 * kStages * kKeyTile * HD * 2;
}

dflash_status launch_attention_bf16(const AttnParams& p, int head_dim, cudaStream_t st) {
  const int QR = p.G * p.L;
  const int warps = (QR + 15) / 16;
  if (warps > 4) return set_error(DFLASH_ERR_UNSUPPORTED, "attention: G*L > 64 query rows");
  const size_t smem = attn_smem_bytes(p.G, p.L, head_dim);
  dim3 grid(p.n_chunks, p.n_kv, p.n_req);
  dim3 cgrid((QR + 3) / 4, p.n_kv, p.n_req);
  // few chunks per (request, KV head): several rows per warp
  const bool few = p.n_chunks <= kFewParts && p.n_qt == 0;
  const long long few_rows = (long long)p.n_req * p.n_kv * QR;
  const dim3 fgrid(static_cast<unsigned>((few_rows + 4 * kRowsPerWarp - 1) / (4 * kRowsPerWarp)));
  if (head_dim == 128) {
    static bool set = false;
    if (!set) {
      cudaFuncSetAttribute(attn_split_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           227 * 1024);
      set = true;
    }
    {
      TraceScope ts("attn_split", st);
      launch_k(attn_split_kernel<128>, grid, dim3(256), smem, st, p);
    }
    TraceScope ts("attn_combine", st);
    if (few) launch_k(attn_combine_few_kernel<128>, fgrid, dim3(128), 0, st, p);
    else launch_k(attn_combine_kernel<128>, cgrid, dim3(128), 0, st, p);
  } else if (head_dim == 64) {
    static bool set = false;
    if (!set) {
      cudaFuncSetAttribute(attn_split_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           227 * 1024);
      set = true;
    }
    {
      TraceScope ts("attn_split", st);
      launch_k(attn_split_kernel<64>, grid, dim3(256), smem, st, p);
    }
    TraceScope ts("attn_combine", st);
    if (few) launch_k(attn_combine_few_kernel<64>, fgrid, dim3(128), 0, st, p);
    else launch_k(attn_combine_kernel<64>, cgrid, dim3(128), 0, st, p);
  } else {
    return set_error(DFLASH_ERR_UNSUPPORTED, "attention: head_dim must be 64 or 128");
  }
  return check_launch("attention_bf16");
}

dflash_status launch_attention_f32(const AttnParamsF32& p, int head_dim, cudaStream_t st) {
  const int total = p.n_req * p.n_q * p.L;
  const int blocks = (total + 3) / 4;
  TraceScope ts("attn_f32", st);
  if (head_dim == 128) launch_k(attn_f32_kernel<128>, dim3(blocks), dim3(128), 0, st, p);
  else if (head_dim == 64) launch_k(attn_f32_kernel<64>, dim3(blocks), dim3(128), 0, st, p);
  else return set_error(DFLASH_ERR_UNSUPPORTED, "attention: head_dim must be 64 or 128");
  return check_launch("attention_f32");
}

}  // namespace dfl
