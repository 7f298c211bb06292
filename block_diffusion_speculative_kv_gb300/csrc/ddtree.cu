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
// one per open parent; slot s belongs to lane s % 32, and a lane's slots are
// scanned by that lane at every pop.  Keys are 64-bit:
// order-preserving score bits, then the complemented creation counter, so
// equal scores pop in creation order.  A pop is a warp-wide maximum of the
// lanes' bests (redux.sync on the high word, and on the low word only when the
// high word ties); the popped slot advances to its next rank in place (or
// closes) and a new slot opens for the popped node's first child.  A pop has
// no divergent single-lane branches: the new keys are computed by every lane
// and written by predicated stores.  Candidate scores are the parent score plus
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
  int* tok;         // [B+1]
  int* par;         // [B+1]
  int* dep;         // [B+1]
  int* rnk;         // [B+1]
  uint64_t* key;    // [B+1] slot keys (0 = closed)
  uint32_t* info;   // [B+1] slot (parent, depth, rank)
  float* psc;       // [B+1] slot parent score
  uint32_t* stage;  // [32][W]
};

__host__ __device__ inline size_t build_warp_bytes(int D, int K, int B) {
  const int W = (B + 1 + 31) / 32;
  size_t b = 0;
  b += align_up(sizeof(uint64_t) * (B + 1), 16);
  b += align_up(sizeof(float) * D * K, 16);
  b += align_up(sizeof(int) * D * K, 16);
  b += 4 * align_up(sizeof(int) * (B + 1), 16);
  b += align_up(sizeof(uint32_t) * (B + 1), 16);
  b += align_up(sizeof(float) * (B + 1), 16);
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
    sm.key = reinterpret_cast<uint64_t*>(base + off); off += align_up(sizeof(uint64_t) * (B + 1), 16);
    sm.lp = reinterpret_cast<float*>(base + off); off += align_up(sizeof(float) * D * K, 16);
    sm.ids = reinterpret_cast<int*>(base + off); off += align_up(sizeof(int) * D * K, 16);
    sm.tok = reinterpret_cast<int*>(base + off); off += align_up(sizeof(int) * (B + 1), 16);
    sm.par = reinterpret_cast<int*>(base + off); off += align_up(sizeof(int) * (B + 1), 16);
    sm.dep = reinterpret_cast<int*>(base + off); off += align_up(sizeof(int) * (B + 1), 16);
    sm.rnk = reinterpret_cast<int*>(base + off); off += align_up(sizeof(int) * (B + 1), 16);
    sm.info = reinterpret_cast<uint32_t*>(base + off); off += align_up(sizeof(uint32_t) * (B + 1), 16);
    sm.psc = reinterpret_cast<float*>(base + off); off += align_up(sizeof(float) * (B + 1), 16);
    sm.stage = reinterpret_cast<uint32_t*>(base + off);
  }
  const float* lp_r = lp_g + (size_t)req * D * K;
  const int32_t* ids_r = ids_g + (size_t)req * D * K;
  for (int i = lane; i < D * K; i += 32) { sm.lp[i] = lp_r[i]; sm.ids[i] = ids_r[i]; }
  if (lane == 0) {
    sm.tok[0] = root_tok[req]; sm.par[0] = -1; sm.dep[0] = 0; sm.rnk[0] = 0;
  }
  __syncwarp();

  // ---- Algorithm 1 ----
  // Every pop: each lane scans its own slots (independent shared loads), one
  // warp-wide argmax picks the winner, all lanes read the winner's slot and the
  // log-probabilities it needs (broadcast loads), every lane computes the same
  // new keys, and the node/slot writes go out as one predicated scattered store
  // per width - no divergent single-lane branches on the critical path.
  int n = 0, n_slots = 0;
  uint32_t seq = 0;
  if (B > 0) {
    if (lane == 0) {
      sm.key[0] = make_key(__fadd_rn(0.f, sm.lp[0]), 0u);
      sm.info[0] = pack_info(0, 1, 1);
      sm.psc[0] = 0.f;
    }
    n_slots = 1;
    seq = 1;
  }
  __syncwarp();
  while (n < B) {
    uint64_t best = 0;
    int bslot = 0;
    for (int sl = lane; sl < n_slots; sl += 32) {
      const uint64_t k = sm.key[sl];
      if (k > best) { best = k; bslot = sl; }
    }
    uint64_t kmax;
    const int w = warp_argmax_key(best, kmax);
    if (kmax == 0) break;  // no candidate left
    const int slot = __shfl_sync(0xffffffffu, bslot, w);
    const uint32_t winfo = sm.info[slot];
    const float wpsc = sm.psc[slot];
    const float wscore = from_ordered_bits(static_cast<uint32_t>(kmax >> 32));
    const int p = winfo & 0x7FF;
    const int d = (winfo >> 11) & 0x1F;
    const int r = (winfo >> 16) & 0x3F;
    const float lp_sib = sm.lp[(d - 1) * K + (r < K ? r : K - 1)];
    const float lp_child = sm.lp[(d < D ? d : D - 1) * K];
    const int tokv = sm.ids[(d - 1) * K + (r - 1)];
    ++n;
    const bool has_sib = r < K;
    const bool has_child = d < D;
    const uint64_t sib_key = has_sib ? make_key(__fadd_rn(wpsc, lp_sib), seq) : 0ull;
    seq += has_sib ? 1u : 0u;
    const uint64_t child_key = make_key(__fadd_rn(wscore, lp_child), seq);
    seq += has_child ? 1u : 0u;
    const int cslot = n_slots;
    n_slots += has_child ? 1 : 0;
    // 32-bit writes: lane 0..3 the node, lane 4 the popped slot's rank, lanes 5-6 the child slot
    {
      uint32_t* addr = nullptr;
      uint32_t val = 0;
      switch (lane) {
        case 0: addr = reinterpret_cast<uint32_t*>(sm.tok + n); val = static_cast<uint32_t>(tokv); break;
        case 1: addr = reinterpret_cast<uint32_t*>(sm.par + n); val = static_cast<uint32_t>(p); break;
        case 2: addr = reinterpret_cast<uint32_t*>(sm.dep + n); val = static_cast<uint32_t>(d); break;
        case 3: addr = reinterpret_cast<uint32_t*>(sm.rnk + n); val = static_cast<uint32_t>(r); break;
        case 4: if (has_sib) { addr = sm.info + slot; val = pack_info(p, d, r + 1); } break;
        case 5: if (has_child) { addr = sm.info + cslot; val = pack_info(n, d + 1, 1); } break;
        case 6: if (has_child) { addr = reinterpret_cast<uint32_t*>(sm.psc + cslot); val = __float_as_uint(wscore); } break;
        default: break;
      }
      if (addr) *addr = val;
    }
    // 64-bit writes: lane 0 the popped slot's new key (0 closes it), lane 1 the child's key
    if (lane == 0) sm.key[slot] = sib_key;
    if (lane == 1 && has_child) sm.key[cslot] = child_key;
    __syncwarp();
  }
  __syncwarp();

  // ---- flattened tree (coalesced, -1 past the last node) ----
  const size_t nb = (size_t)req * (B + 1);
  for (int i = lane; i <= B; i += 32) {
    const bool live = i <= n;
    tok_out[nb + i] = live ? sm.tok[i] : -1;
    parent_out[nb + i] = live ? sm.par[i] : -1;
    depth_out[nb + i] = live ? sm.dep[i] : -1;
    rank_out[nb + i] = live ? sm.rnk[i] : -1;
  }
  if (lane == 0) n_nodes_out[req] = n;

  // ---- ancestor mask, 32 rows at a time staged in shared memory ----
  uint32_t* mrow = mask_out + nb * W;
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
        j = sm.par[j];
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
