// DDTree tree construction (step a7) and verifier walk (step a8).
//
// "Accelerating Speculative Decoding with Block Diffusion Draft Trees":
// section 3.4.4, Algorithm 1 (best-first search over rank tuples with a
// max-heap; each pop becomes a node and offers its next sibling and its first
// child), and section 3.4.5 (flattened tree with depth position ids, the
// ancestor-only attention mask, and the greedy verifier walk).
//
// GPU formulation of the heap.  The candidates alive at any time are exactly
// one per "open" parent: the parent's next unpopped child rank (children of a
// node are popped in rank order, since a sibling is offered only after its
// predecessor pops).  So the heap is kept as a set of slots in shared memory,
// one per open parent; slot s belongs to lane s % 32, which keeps the best key
// among its slots in a register.  Keys are 64-bit:
// order-preserving score bits, then the complemented creation counter, so
// equal scores pop in creation order.  A pop is a warp-wide maximum of the
// lanes' bests (redux.sync on the high word, and on the low word only when the
// high word ties); the popped slot advances to its next rank in place (or
// closes) and a new slot opens for the popped node's first child.  Candidate scores are the parent score plus
// one log-probability, a single fp32 add, so the result is bit-identical to a
// plain binary-heap implementation of the same rule.
#include "common.cuh"
#include "kernels.h"

namespace dfl {

namespace {

constexpr int kBuildWarps = 4;

__device__ __forceinline__ uint64_t make_key(float score, uint32_t seq) {
  return (static_cast<uint64_t>(ordered_bits(score)) << 32) |
         static_cast<uint64_t>(0xFFFFFFFFu - seq);
}
__device__ __forceinline__ uint32_t pack_info(int parent, int depth, int rank) {
  return static_cast<uint32_t>(parent) | (static_cast<uint32_t>(depth) << 11) |
         (static_cast<uint32_t>(rank) << 16);
}

struct WarpSmem {
  float* lp;        // [D*K]
  int* ids;         // [D*K]
  uint32_t* node;   // [B+1][4]: tok, parent, depth, rank
  uint32_t* slot;   // [B+1][4]: key low, key high (0 = closed), info, parent score bits
  uint32_t* stage;  // [32][W]
};

__host__ __device__ inline size_t build_warp_bytes(int D, int K, int B) {
  const int W = (B + 1 + 31) / 32;
  size_t b = 0;
  b += align_up(sizeof(uint32_t) * 4 * (B + 1), 16);
  b += align_up(sizeof(uint32_t) * 4 * (B + 1), 16);
  b += align_up(sizeof(float) * D * K, 16);
  b += align_up(sizeof(int) * D * K, 16);
  b += align_up(sizeof(uint32_t) * 32 * W, 16);
  return b;
}

// Warp-wide maximum of 64-bit keys; returns the lane holding it (keys unique
// unless all are 0) and the key.
__device__ __forceinline__ int warp_argmax_key(uint64_t k, uint64_t& kmax) {
  const unsigned FULL = 0xffffffffu;
  const uint32_t hi = static_cast<uint32_t>(k >> 32);
  const uint32_t lo = static_cast<uint32_t>(k);
  const uint32_t mhi = __reduce_max_sync(FULL, hi);
  unsigned b = __ballot_sync(FULL, hi == mhi);
  uint32_t mlo;
  if (__popc(b) == 1) {
    mlo = __shfl_sync(FULL, lo, __ffs(b) - 1);
  } else {
    mlo = __reduce_max_sync(FULL, hi == mhi ? lo : 0u);
    b = __ballot_sync(FULL, hi == mhi && lo == mlo);
  }
  kmax = (static_cast<uint64_t>(mhi) << 32) | mlo;
  return __ffs(b) - 1;
}

__global__ void __launch_bounds__(kBuildWarps * 32)
ddtree_build_kernel(int n_req, int D, int K, int B, const float* __restrict__ lp_g,
                    const int32_t* __restrict__ ids_g, const int32_t* __restrict__ root_tok,
                    int32_t* __restrict__ n_nodes_out, int32_t* __restrict__ tok_out,
                    int32_t* __restrict__ parent_out, int32_t* __restrict__ depth_out,
                    int32_t* __restrict__ rank_out, uint32_t* __restrict__ mask_out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int req = blockIdx.x * kBuildWarps + wib;
  pdl_wait();
  pdl_trigger();
  if (req >= n_req) return;
  const int W = (B + 1 + 31) / 32;

  unsigned char* base = smem_raw + build_warp_bytes(D, K, B) * wib;
  WarpSmem sm;
  {
    size_t off = 0;
    sm.node = reinterpret_cast<uint32_t*>(base + off); off += align_up(sizeof(uint32_t) * 4 * (B + 1), 16);
    sm.slot = reinterpret_cast<uint32_t*>(base + off); off += align_up(sizeof(uint32_t) * 4 * (B + 1), 16);
    sm.lp = reinterpret_cast<float*>(base + off); off += align_up(sizeof(float) * D * K, 16);
    sm.ids = reinterpret_cast<int*>(base + off); off += align_up(sizeof(int) * D * K, 16);
    sm.stage = reinterpret_cast<uint32_t*>(base + off);
  }
  const float* lp_r = lp_g + (size_t)req * D * K;
  const int32_t* ids_r = ids_g + (size_t)req * D * K;
  for (int i = lane; i < D * K; i += 32) { sm.lp[i] = lp_r[i]; sm.ids[i] = ids_r[i]; }
  if (lane == 0) {
    sm.node[0] = static_cast<uint32_t>(root_tok[req]);
    sm.node[1] = 0xFFFFFFFFu;  // parent -1
    sm.node[2] = 0;
    sm.node[3] = 0;
  }
  __syncwarp();

  // ---- Algorithm 1 ----
  // Each lane keeps the best key among its own slots.  A pop: warp argmax of
  // the lanes' bests; every lane reads the winner's slot record and the
  // log-probabilities it needs (broadcast loads) and computes the same new
  // keys; the node record and both slot updates go out as one predicated
  // scattered store; every lane then rescans the winner's slots (broadcast
  // loads, identical results), and the winner and the child's owner update
  // their bests with selects.  No divergent branch and no extra warp
  // reduction sits on the per-pop critical path.
  uint64_t lbest = 0;  // best key among this lane's slots
  int lbs = 0;         // its slot
  int n = 0, n_slots = 0;
  uint32_t seq = 0;
  if (B > 0) {
    const uint64_t k0 = make_key(__fadd_rn(0.f, sm.lp[0]), 0u);
    if (lane == 0) {
      sm.slot[0] = static_cast<uint32_t>(k0);
      sm.slot[1] = static_cast<uint32_t>(k0 >> 32);
      sm.slot[2] = pack_info(0, 1, 1);
      sm.slot[3] = __float_as_uint(0.f);
    }
    lbest = (lane == 0) ? k0 : 0ull;
    n_slots = 1;
    seq = 1;
  }
  __syncwarp();
  while (n < B) {
    uint64_t kmax;
    const int w = warp_argmax_key(lbest, kmax);
    if (kmax == 0) break;  // no candidate left
    const int slot = __shfl_sync(0xffffffffu, lbs, w);
    const uint4 rec = *reinterpret_cast<const uint4*>(sm.slot + 4 * slot);
    const uint32_t winfo = rec.z;
    const float wpsc = __uint_as_float(rec.w);
    const float wscore = from_ordered_bits(static_cast<uint32_t>(kmax >> 32));
    const int p = winfo & 0x7FF;
    const int d = (winfo >> 11) & 0x1F;
    const int r = (winfo >> 16) & 0x3F;
    const float lp_sib = sm.lp[(d - 1) * K + (r < K ? r : K - 1)];
    const float lp_child = sm.lp[(d < D ? d : D - 1) * K];
    const uint32_t tokv = static_cast<uint32_t>(sm.ids[(d - 1) * K + (r - 1)]);
    ++n;
    const bool has_sib = r < K;
    const bool has_child = d < D;
    const uint64_t sib_key = has_sib ? make_key(__fadd_rn(wpsc, lp_sib), seq) : 0ull;
    seq += has_sib ? 1u : 0u;
    const uint64_t child_key = make_key(__fadd_rn(wscore, lp_child), seq);
    seq += has_child ? 1u : 0u;
    const int cslot = n_slots;
    n_slots += has_child ? 1 : 0;
    // lanes 0-3: node record; 4-6: popped slot (key low, key high, info);
    // 8-11: child slot (key low, key high, info, parent score)
    const int q = lane & 3;
    const uint32_t node_v = q == 0 ? tokv : q == 1 ? static_cast<uint32_t>(p)
                          : q == 2 ? static_cast<uint32_t>(d) : static_cast<uint32_t>(r);
    const uint32_t sib_v = q == 0 ? static_cast<uint32_t>(sib_key)
                         : q == 1 ? static_cast<uint32_t>(sib_key >> 32) : pack_info(p, d, r + 1);
    const uint32_t ch_v = q == 0 ? static_cast<uint32_t>(child_key)
                        : q == 1 ? static_cast<uint32_t>(child_key >> 32)
                        : q == 2 ? pack_info(n, d + 1, 1) : __float_as_uint(wscore);
    const uint32_t val = lane < 4 ? node_v : (lane < 8 ? sib_v : ch_v);
    const int idx = lane < 4 ? 4 * n + q : (lane < 8 ? 4 * slot + q : 4 * cslot + q);
    uint32_t* dst = lane < 4 ? sm.node : sm.slot;
    const bool wr = lane < 4 || lane == 4 || lane == 5 || (lane == 6 && has_sib) ||
                    (lane >= 8 && lane < 12 && has_child);
    if (wr) dst[idx] = val;
    __syncwarp();
    // the winner's new best, computed by every lane (broadcast loads)
    uint64_t nb = 0;
    int nbs = w;
    for (int s0 = w; s0 < n_slots; s0 += 128) {
      uint64_t k[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int sl = s0 + 32 * u;
        k[u] = sl < n_slots ? *reinterpret_cast<const unsigned long long*>(sm.slot + 4 * sl) : 0ull;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (k[u] > nb) { nb = k[u]; nbs = s0 + 32 * u; }
    }
    const bool is_w = lane == w;
    const bool take_child = has_child && lane == (cslot & 31) && !is_w && child_key > lbest;
    lbest = is_w ? nb : (take_child ? child_key : lbest);
    lbs = is_w ? nbs : (take_child ? cslot : lbs);
  }
  __syncwarp();

  // ---- flattened tree (coalesced, -1 past the last node) ----
  const size_t nb_out = (size_t)req * (B + 1);
  for (int i = lane; i <= B; i += 32) {
    const bool live = i <= n;
    const uint4 rec = live ? *reinterpret_cast<const uint4*>(sm.node + 4 * i) : make_uint4(0, 0, 0, 0);
    tok_out[nb_out + i] = live ? static_cast<int32_t>(rec.x) : -1;
    parent_out[nb_out + i] = live ? static_cast<int32_t>(rec.y) : -1;
    depth_out[nb_out + i] = live ? static_cast<int32_t>(rec.z) : -1;
    rank_out[nb_out + i] = live ? static_cast<int32_t>(rec.w) : -1;
  }
  if (lane == 0) n_nodes_out[req] = n;

  // ---- ancestor mask, 32 rows at a time staged in shared memory ----
  uint32_t* mrow = mask_out + nb_out * W;
  for (int i0 = 0; i0 <= B; i0 += 32) {
    for (int t = lane; t < 32 * W; t += 32) sm.stage[t] = 0u;
    __syncwarp();
    const int i = i0 + lane;
    if (i <= n) {
      uint32_t* st = sm.stage + lane * W;
      int j = i;
      while (true) {
        st[j >> 5] |= 1u << (j & 31);
        if (j == 0) break;
        j = static_cast<int>(sm.node[4 * j + 1]);
      }
    }
    __syncwarp();
    const int rows = min(32, B + 1 - i0);
    for (int t = lane; t < rows * W; t += 32) mrow[(size_t)i0 * W + t] = sm.stage[t];
    __syncwarp();
  }
}

void launch_build(const TreeBuildLaunch& a, cudaStream_t st) {
  const size_t per_warp = build_warp_bytes(a.D, a.K, a.B);
  const size_t smem = per_warp * kBuildWarps;
  static bool attr_set = false;  // per instantiation, per process
  if (!attr_set) {
    cudaFuncSetAttribute(ddtree_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         200 * 1024);
    attr_set = true;
  }
  dim3 grid(ceil_div(a.n_req, kBuildWarps));
  TraceScope ts("ddtree_build", st);
  launch_k(ddtree_build_kernel, grid, dim3(kBuildWarps * 32), smem, st, a.n_req, a.D, a.K, a.B,
           a.topk_logp, a.topk_ids, a.root_tok, a.n_nodes, a.tok, a.parent, a.depth, a.rank,
           a.mask);
}

// ---------------------------------------------------------------------------
// Verifier walk: one warp per request.  Children of a node have larger indices
// than the node (they pop later), so the search for the matching child scans
// forward from the current node, 32 candidates per step.
// ---------------------------------------------------------------------------
__global__ void ddtree_accept_kernel(int n_req, int D, int B, const int32_t* __restrict__ n_nodes,
                                     const int32_t* __restrict__ tok,
                                     const int32_t* __restrict__ parent,
                                     const int32_t* __restrict__ target,
                                     int32_t* __restrict__ accept_len,
                                     int32_t* __restrict__ accepted, int32_t* __restrict__ bonus) {
  const int lane = threadIdx.x & 31;
  const int req = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  pdl_wait();
  pdl_trigger();
  if (req >= n_req) return;
  const unsigned FULL = 0xffffffffu;
  const size_t nb = (size_t)req * (B + 1);
  const int n = min(max(n_nodes[req], 0), B);
  int node = 0, len = 0;
  while (true) {
    const int y = target[nb + node];
    int found = -1;
    for (int c0 = node + 1; c0 <= n; c0 += 32) {
      const int c = c0 + lane;
      const bool hit = (c <= n) && parent[nb + c] == node && tok[nb + c] == y;
      const unsigned b = __ballot_sync(FULL, hit);
      if (b) { found = c0 + __ffs(b) - 1; break; }
    }
    if (found < 0 || len >= D) break;
    if (lane == 0) accepted[(size_t)req * D + len] = found;
    ++len;
    node = found;
  }
  for (int t = len + lane; t < D; t += 32) accepted[(size_t)req * D + t] = -1;
  if (lane == 0) {
    accept_len[req] = len;
    bonus[req] = target[nb + node];
  }
}

}  // namespace

size_t tree_build_smem_bytes(int D, int K, int B) {
  return build_warp_bytes(D, K, B) * kBuildWarps;
}

void launch_tree_build(const TreeBuildLaunch& a, cudaStream_t st) {
  if (a.n_req <= 0) return;
  launch_build(a, st);
}

void launch_tree_accept(const TreeAcceptLaunch& a, cudaStream_t st) {
  if (a.n_req <= 0) return;
  const int warps = 4;
  TraceScope ts("ddtree_accept", st);
  launch_k(ddtree_accept_kernel, dim3(ceil_div(a.n_req, warps)), dim3(warps * 32), 0, st,
           a.n_req, a.D, a.B, a.n_nodes, a.tok, a.parent, a.target, a.accept_len, a.accepted,
           a.bonus);
}

}  // namespace dfl
