// Tree attention of the verification pass and the depth position ids.
//
// "Accelerating Speculative Decoding with Block Diffusion Draft Trees",
// section 3.4.5: the draft tree is flattened (node 0 is the root, the bonus
// token), every node gets the position id of its depth, and one forward pass
// of the target model scores all nodes under the ancestor-only mask: node i
// attends to the whole past context (the KV cache), to the root, to its
// ancestors and to itself, and to no other tree node.  This file is one
// target-layer attention of that pass, with grouped-query heads:
//
//   out[i, h] = softmax_j( q[i, h] . key_j / sqrt(hd) ) value_j
//   over key_j in { cache slot t < ctx_len } U { tree node j : mask[i] has bit j }
//
// and the rotation of the tree's queries and keys at position ctx_len + depth.
//
// Decomposition (same scheme as the drafter's block attention): query tiles of
// 16 nodes x the G query heads of a KV head (64 rows), the context split into
// chunks of keys, and the tree's own keys as one more chunk; each CTA writes an
// unnormalised partial (O, max, sum) of its rows and the drafter's combine
// kernel merges the partials.  Nodes are numbered in pop order, so an ancestor
// has a smaller number than its descendant: the tree chunk of query tile qt
// reads tree keys 0 .. 16 qt + 15 only.
#include <cmath>

#include "attention.h"
#include "common.cuh"
#include "kernels.h"
#include "mma_sync.cuh"

#include <math_constants.h>

namespace dfl {

namespace {

using namespace mmas;

constexpr int kKeyTile = 64;
constexpr int kStages = 6;
constexpr int kNodesPerTile = 16;
constexpr int kThreads = 256;

struct TreeAttnParams {
  AttnParams a;                 // cache, head counts, chunking, partials, output (with n_qt)
  const __nv_bfloat16* q;       // [n_req][B+1][q_ld], head h at column h*hd
  long long q_ld;
  const __nv_bfloat16* kt;      // the nodes' keys [n_req][B+1][kv_ld], KV head g at g*hd
  const __nv_bfloat16* vt;
  long long kv_ld;
  const uint32_t* mask;         // [n_req][B+1][mask_w]
  int mask_w;
  const int32_t* n_nodes;       // [n_req]: nodes 0 .. n_nodes[r] are live
  int B1;                       // B + 1
  int n_ctx_chunks;             // context chunks; chunk n_ctx_chunks is the tree's
};

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
tree_attn_split_kernel(const TreeAttnParams tp) {
  constexpr int NCH = HD / 8;
  const AttnParams& p = tp.a;
  extern __shared__ __align__(128) uint8_t smem[];
  const int QR = p.G * kNodesPerTile;   // <= 64
  const int QRp = (QR + 15) / 16 * 16;
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + QRp * HD * 2;
  uint8_t* sV = sK + kStages * kKeyTile * HD * 2;

  const int chunk_id = blockIdx.x;
  const int g = blockIdx.y;
  const int rq = blockIdx.z;            // (request, query tile)
  const int req = rq / p.n_qt, qt = rq % p.n_qt;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool tree_part = chunk_id == tp.n_ctx_chunks;
  const int last = min(max(tp.n_nodes[req], 0), tp.B1 - 1);   // last live node
  const int node0 = qt * kNodesPerTile;
  const int ctx = min(max(p.ctx_len[req], 0), p.cap);
  int key_begin = 0, key_end = 0;       // context keys, or tree keys
  if (tree_part) {
    key_end = node0 <= last ? min(node0 + kNodesPerTile - 1, last) + 1 : 0;
  } else {
    key_begin = chunk_id * p.chunk;
    key_end = min(ctx, key_begin + p.chunk);
  }
  const int ntiles = key_end > key_begin ? (key_end - key_begin + kKeyTile - 1) / kKeyTile : 0;
  const size_t part_row0 = (((size_t)rq * p.n_kv + g) * p.n_chunks + chunk_id) * QR;
  if (ntiles == 0 || node0 > last) {
    pdl_wait();
    pdl_trigger();
    for (int r = tid; r < QR; r += blockDim.x) {
      p.part_ml[(part_row0 + r) * 2 + 0] = -CUDART_INF_F;
      p.part_ml[(part_row0 + r) * 2 + 1] = 0.f;
    }
    return;
  }
  const __nv_bfloat16* kb_base =
      tree_part ? tp.kt + (size_t)req * tp.B1 * tp.kv_ld + (size_t)g * HD
                : p.cache_k + ((size_t)req * p.n_kv + g) * p.cap * HD;
  const __nv_bfloat16* vb_base =
      tree_part ? tp.vt + (size_t)req * tp.B1 * tp.kv_ld + (size_t)g * HD
                : p.cache_v + ((size_t)req * p.n_kv + g) * p.cap * HD;
  const long long kld = tree_part ? tp.kv_ld : HD;

  auto load_tile = [&](int buf, int t) {
    uint8_t* dK = sK + buf * kKeyTile * HD * 2;
    uint8_t* dV = sV + buf * kKeyTile * HD * 2;
    const int key0 = key_begin + t * kKeyTile;
    for (int i = tid; i < kKeyTile * NCH; i += blockDim.x) {
      const int r = i / NCH, ch = i % NCH;
      const int key = key0 + r;
      const bool valid = key < key_end;
      const size_t off = (size_t)(valid ? key : key0) * kld + ch * 8;
      cp_async16(smem_u32(dK) + swz<HD>(r, ch), kb_base + off, valid);
      cp_async16(smem_u32(dV) + swz<HD>(r, ch), vb_base + off, valid);
    }
  };
  constexpr int kAhead = kStages - 2;
  const int npre = ntiles < kAhead ? ntiles : kAhead;
  // context tiles (the cache, written kernels back) go out before the wait;
  // the tree's keys come from the projection just before this kernel
  int issued = 0;
  if (!tree_part) {
    while (issued < npre) {
      load_tile(issued, issued);
      cp_async_commit();
      ++issued;
    }
  }
  pdl_wait();
  pdl_trigger();

  // ---- Q: row r = head (r / 16) of the KV head's group, node node0 + r % 16 ----
  for (int i = tid; i < QRp * NCH; i += blockDim.x) {
    const int r = i / NCH, ch = i % NCH;
    const int node = node0 + r % kNodesPerTile;
    const bool valid = r < QR && node <= last;
    const int h = g * p.G + (valid ? r / kNodesPerTile : 0);
    const __nv_bfloat16* src =
        tp.q + ((size_t)req * tp.B1 + (valid ? node : 0)) * tp.q_ld + (size_t)h * HD + ch * 8;
    cp_async16(smem_u32(sQ) + swz<HD>(r, ch), src, valid);
  }
  cp_async_commit();
  while (issued < npre) {
    load_tile(issued, issued);
    cp_async_commit();
    ++issued;
  }

  const int grp = warp >> 2;
  const int qrow0 = (warp & 3) * 16;
  const bool warp_active = qrow0 < QR;
  const int gq = lane >> 2, tq = lane & 3;
  // this thread's two rows: nodes node0 + gq and node0 + gq + 8
  const int nodeA = node0 + gq, nodeB = nodeA + 8;
  const bool liveA = nodeA <= last, liveB = nodeB <= last;
  float o[HD / 8][4];
#pragma unroll
  for (int n = 0; n < HD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  uint32_t qa[HD / 16][4];

  for (int it = 0; 2 * it < ntiles; ++it) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int tn = 2 * it + npre + e;
      if (tn < ntiles) load_tile(tn % kStages, tn);
      cp_async_commit();
    }
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
      const int key0 = key_begin + t * kKeyTile;
      const uint32_t kb = smem_u32(sK + (t % kStages) * kKeyTile * HD * 2);
      const uint32_t vb = smem_u32(sV + (t % kStages) * kKeyTile * HD * 2);
      // ancestor bits of the two rows over this tile's 64 tree keys
      uint32_t mA0 = 0, mA1 = 0, mB0 = 0, mB1 = 0;
      if (tree_part) {
        const int w0 = key0 >> 5;
        const uint32_t* ra = tp.mask + ((size_t)req * tp.B1 + min(nodeA, last)) * tp.mask_w;
        const uint32_t* rb = tp.mask + ((size_t)req * tp.B1 + min(nodeB, last)) * tp.mask_w;
        mA0 = liveA && w0 < tp.mask_w ? ra[w0] : 0u;
        mA1 = liveA && w0 + 1 < tp.mask_w ? ra[w0 + 1] : 0u;
        mB0 = liveB && w0 < tp.mask_w ? rb[w0] : 0u;
        mB1 = liveB && w0 + 1 < tp.mask_w ? rb[w0 + 1] : 0u;
      }
      float s[kKeyTile / 8][4];
#pragma unroll
      for (int n = 0; n < kKeyTile / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
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
      float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
      for (int n = 0; n < kKeyTile / 8; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kt = n * 8 + 2 * tq + e;   // key within the tile
          const bool in = key0 + kt < key_end;
          bool okA = in && liveA, okB = in && liveB;
          if (tree_part) {
            okA = okA && (((kt < 32 ? mA0 >> kt : mA1 >> (kt - 32)) & 1u) != 0u);
            okB = okB && (((kt < 32 ? mB0 >> kt : mB1 >> (kt - 32)) & 1u) != 0u);
          }
          const float v0 = okA ? s[n][e] * p.scale_log2 : -CUDART_INF_F;
          const float v1 = okB ? s[n][2 + e] * p.scale_log2 : -CUDART_INF_F;
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

#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  // merge the two groups' states (group 1 -> shared memory -> group 0)
  float* mo = reinterpret_cast<float*>(sK);
  float* mml = mo + QRp * HD;
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
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) {
      const int d = n * 8 + 2 * tq;
      if (rq0 < QR)
        *reinterpret_cast<float2*>(p.part_o + (part_row0 + rq0) * HD + d) =
            make_float2(o[n][0], o[n][1]);
      if (rq1 < QR)
        *reinterpret_cast<float2*>(p.part_o + (part_row0 + rq1) * HD + d) =
            make_float2(o[n][2], o[n][3]);
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
}

// Rotation of one (node, head) row at position ctx_len + depth; a warp per row,
// lanes over the first half of the head dimension.
template <typename T>
__global__ void tree_rope_kernel(int n_req, int B1, int n_heads, int head_dim, const RopeFreqs fr,
                                 const int32_t* __restrict__ ctx_len,
                                 const int32_t* __restrict__ depth, T* __restrict__ x,
                                 long long ld) {
  const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  if (w >= (long long)n_req * B1 * n_heads) return;
  const int h = static_cast<int>(w % n_heads);
  const long long node = w / n_heads;            // req * B1 + i
  const int req = static_cast<int>(node / B1);
  const int dep = depth[node];
  if (dep < 0) return;                            // past the last node
  const int pos = ctx_len[req] + dep;
  const int half = head_dim / 2;
  T* row = x + node * ld + (long long)h * head_dim;
  for (int i = lane; i < half; i += 32) {
    const float2 cs = rope_cs(pos, i, fr);
    const float a = to_f32<T>(row[i]), b = to_f32<T>(row[i + half]);
    row[i] = from_f32<T>(a * cs.x - b * cs.y);
    row[i + half] = from_f32<T>(b * cs.x + a * cs.y);
  }
}

int tree_ctx_chunk(int max_ctx) {
  // chunks of 1024 context keys: with 17+ query tiles per KV head the grid
  // is many waves already; longer chunks mean fewer partials to merge
  const int c = 1024;
  return max_ctx < c ? ((max_ctx + kKeyTile - 1) / kKeyTile) * kKeyTile : c;
}

}  // namespace

}  // namespace dfl

using namespace dfl;

extern "C" {

size_t dflash_tree_attention_workspace_bytes(int n_req, int n_q, int n_kv, int head_dim, int B,
                                             int max_ctx) {
  if (n_req < 1 || n_kv < 1 || n_q < n_kv || n_q % n_kv || B < 0 || max_ctx < 0 || head_dim != 128)
    return 0;
  const int G = n_q / n_kv;
  const int n_qt = (B + 1 + kNodesPerTile - 1) / kNodesPerTile;
  const int chunk = tree_ctx_chunk(max_ctx > 0 ? max_ctx : 1);
  const int n_chunks = (max_ctx > 0 ? (max_ctx + chunk - 1) / chunk : 0) + 1;
  const size_t rows = (size_t)n_req * n_qt * n_kv * n_chunks * G * kNodesPerTile;
  return 256 + align_up(rows * head_dim * sizeof(float), 256) + align_up(rows * 2 * sizeof(float), 256);
}

dflash_status dflash_tree_attention(int n_req, int n_q, int n_kv, int head_dim, int B,
                                    const int32_t* ctx_len, int max_ctx, int cap,
                                    const void* cache_k, const void* cache_v, const void* q,
                                    long long q_ld, const void* k, const void* v, long long kv_ld,
                                    const uint32_t* mask, const int32_t* n_nodes, void* out,
                                    long long out_ld, void* ws, size_t ws_bytes, void* stream) {
  DFL_REQUIRE(n_req >= 0, "n_req must be >= 0");
  if (n_req == 0) return DFLASH_OK;
  DFL_REQUIRE(head_dim == 128, "tree attention: head_dim must be 128");
  DFL_REQUIRE(n_kv >= 1 && n_q >= n_kv && n_q % n_kv == 0 && n_q / n_kv <= 4,
              "tree attention: need n_q a multiple of n_kv, at most 4 query heads per KV head");
  DFL_REQUIRE(B >= 0 && B <= 1024, "need 0 <= B <= 1024");
  DFL_REQUIRE(max_ctx >= 0 && max_ctx <= cap, "need 0 <= max_ctx <= cap");
  DFL_REQUIRE(ctx_len && cache_k && cache_v && q && k && v && mask && n_nodes && out,
              "null pointer argument");
  DFL_REQUIRE(q_ld >= (long long)n_q * head_dim && kv_ld >= (long long)n_kv * head_dim &&
                  out_ld >= (long long)n_q * head_dim && q_ld % 8 == 0 && kv_ld % 8 == 0,
              "row strides too small or not multiples of 8");
  const size_t need = dflash_tree_attention_workspace_bytes(n_req, n_q, n_kv, head_dim, B, max_ctx);
  if (!ws || ws_bytes < need)
    return set_error(DFLASH_ERR_WORKSPACE, "tree attention workspace needs %zu bytes, got %zu",
                     need, ws_bytes);
  const int G = n_q / n_kv;
  const int B1 = B + 1;
  const int n_qt = (B1 + kNodesPerTile - 1) / kNodesPerTile;
  const int chunk = tree_ctx_chunk(max_ctx > 0 ? max_ctx : 1);
  const int n_ctx_chunks = max_ctx > 0 ? (max_ctx + chunk - 1) / chunk : 0;
  const size_t rows = (size_t)n_req * n_qt * n_kv * (n_ctx_chunks + 1) * G * kNodesPerTile;
  char* w = static_cast<char*>(ws);
  TreeAttnParams tp{};
  AttnParams& a = tp.a;
  a.cache_k = static_cast<const __nv_bfloat16*>(cache_k);
  a.cache_v = static_cast<const __nv_bfloat16*>(cache_v);
  a.ctx_len = ctx_len;
  a.cap = cap;
  a.n_req = n_req * n_qt;   // combine: blockIdx.z over (request, query tile)
  a.n_q = n_q;
  a.n_kv = n_kv;
  a.G = G;
  a.L = kNodesPerTile;
  a.chunk = chunk;
  a.n_chunks = n_ctx_chunks + 1;
  a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(head_dim));
  a.part_o = reinterpret_cast<float*>(w + 256);
  a.part_ml = reinterpret_cast<float*>(w + 256 + align_up(rows * head_dim * sizeof(float), 256));
  a.out = static_cast<__nv_bfloat16*>(out);
  a.out_ld = out_ld;
  a.n_qt = n_qt;
  a.out_rows = B1;
  tp.q = static_cast<const __nv_bfloat16*>(q);
  tp.q_ld = q_ld;
  tp.kt = static_cast<const __nv_bfloat16*>(k);
  tp.vt = static_cast<const __nv_bfloat16*>(v);
  tp.kv_ld = kv_ld;
  tp.mask = mask;
  tp.mask_w = (B1 + 31) / 32;
  tp.n_nodes = n_nodes;
  tp.B1 = B1;
  tp.n_ctx_chunks = n_ctx_chunks;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t smem = (size_t)((G * kNodesPerTile + 15) / 16 * 16) * head_dim * 2 +
                      2 * kStages * kKeyTile * head_dim * 2;
  static bool set = false;
  if (!set) {
    cudaFuncSetAttribute(tree_attn_split_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         227 * 1024);
    set = true;
  }
  {
    TraceScope ts("tree_attn_split", st);
    launch_k(tree_attn_split_kernel<128>, dim3(n_ctx_chunks + 1, n_kv, n_req * n_qt),
             dim3(kThreads), smem, st, tp);
  }
  launch_attn_combine(a, head_dim, dim3((G * kNodesPerTile + 3) / 4, n_kv, n_req * n_qt), st);
  return check_launch("tree attention");
}

dflash_status dflash_tree_rope(int n_req, int B, int n_heads, int head_dim, float theta,
                               const int32_t* ctx_len, const int32_t* depth, void* x,
                               long long ld, int dtype, void* stream) {
  DFL_REQUIRE(n_req >= 0 && B >= 0 && n_heads >= 1, "bad sizes");
  if (n_req == 0) return DFLASH_OK;
  DFL_REQUIRE(head_dim >= 2 && head_dim % 2 == 0 && head_dim <= 128, "head_dim: even, <= 128");
  DFL_REQUIRE(theta > 0.f, "rope theta must be > 0");
  DFL_REQUIRE(ld >= (long long)n_heads * head_dim, "row stride too small");
  DFL_REQUIRE(ctx_len && depth && x, "null pointer argument");
  DFL_REQUIRE(dtype == DFLASH_BF16 || dtype == DFLASH_F32, "dtype must be bf16 or f32");
  const RopeFreqs fr = rope_freqs(theta, head_dim);
  const long long warps = (long long)n_req * (B + 1) * n_heads;
  const dim3 grid(static_cast<unsigned>((warps * 32 + 255) / 256));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  TraceScope ts("tree_rope", st);
  if (dtype == DFLASH_BF16)
    launch_k(tree_rope_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, n_req, B + 1, n_heads,
             head_dim, fr, ctx_len, depth, static_cast<__nv_bfloat16*>(x), ld);
  else
    launch_k(tree_rope_kernel<float>, grid, dim3(256), 0, st, n_req, B + 1, n_heads, head_dim, fr,
             ctx_len, depth, static_cast<float*>(x), ld);
  return check_launch("tree rope");
}

}  // extern "C"
