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
// predecessor pops).  So the heap is a set of slots, one per open parent; slot
// s = 32*i + l lives in register i of lane l (its 64-bit key) and in shared
// memory (parent, depth, rank, and the two log-probability terms popping it
// needs: its next sibling's score and its child's log-probability).  A key is
//   [63:32] order-preserving score bits
//   [31:11] MAX - creation counter (equal scores pop in creation order)
//   [10:5]  register index i,  [4:0] lane l
// so keys are unique and the maximum key names its own slot: a pop is two
// warp reductions (redux.sync on the high word, then on the low word among
// lanes that hold the high maximum), with no ballot or shuffle to find the
// winner.  Each lane keeps the maximum of its keys and loads that slot's record
// while the next reductions run; the winner's record comes over in shuffles.
// The popped slot advances to its next rank in place (or closes) and a new
// slot opens for the popped node's first child.  Every lane runs the same
// branch-free sequence, so no lane holds the reductions back.
// Candidate scores are the parent score plus one log-probability, a single
// fp32 add, so the result is bit-identical to a plain binary-heap
// implementation of the same rule.
#include "common.cuh"
#include "kernels.h"

namespace dfl {

namespace {

constexpr int kBuildWarps = 4;
constexpr int kBuildSmemMax = 200 * 1024;
constexpr uint32_t kSeqMax = (1u << 21) - 1;   // creation counter field

__device__ __forceinline__ uint64_t make_key(float score, uint32_t seq, int reg, int lane) {
  return (static_cast<uint64_t>(ordered_bits(score)) << 32) |
         static_cast<uint64_t>(((kSeqMax - seq) << 11) | (static_cast<uint32_t>(reg) << 5) |
                               static_cast<uint32_t>(lane));
}
__device__ __forceinline__ uint32_t pack_info(int parent, int depth, int rank) {
  return static_cast<uint32_t>(parent) | (static_cast<uint32_t>(depth) << 11) |
         (static_cast<uint32_t>(rank) << 16);
}

struct WarpSmem {
  float* lp;        // [D*K]
  const int32_t* ids;   // [D*K] the request's token ids, read from global memory
  uint32_t* node;   // [B+1][4]: tok, parent, depth, rank
  uint4* slot;      // [B+1]: info (parent | depth << 11 | rank << 16), parent score,
                    //        next sibling's score, log-prob of the first child
  uint32_t* stage;  // [32][W]
};

__host__ __device__ inline size_t build_warp_bytes(int D, int K, int B) {
  const int W = (B + 1 + 31) / 32;
  size_t b = 0;
  b += align_up(sizeof(uint32_t) * 4 * (B + 1), 16);
  b += align_up(sizeof(uint4) * (B + 1), 16);
  b += align_up(sizeof(float) * D * K, 16);
  b += align_up(sizeof(uint32_t) * 32 * W, 16);
  return b;
}

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }

// Maximum of a lane's NSL keys (pairwise tree).
template <int NSL>
__device__ __forceinline__ uint64_t max_keys(const uint64_t (&key)[NSL]) {
  uint64_t t[NSL];
#pragma unroll
  for (int i = 0; i < NSL; ++i) t[i] = key[i];
#pragma unroll
  for (int s = 1; s < NSL; s *= 2) {
#pragma unroll
    for (int i = 0; i + s < NSL; i += 2 * s) t[i] = umax64(t[i], t[i + s]);
  }
  return t[0];
}

// Algorithm 1, one pop after another, on one warp (shared-memory records in
// sm, inputs already in sm.lp / sm.ids).  Fills sm.node[0..n]; returns n.
template <int NSL>
__device__ int seq_build(const WarpSmem& sm, int D, int K, int B, int lane, int32_t root) {
  const unsigned FULL = 0xffffffffu;
  // log-probability at (depth d, 0-based rank i), 0 outside the table (the
  // callers only use such values when the matching candidate does not exist)
  auto lpat = [&](int d, int i) {
    const bool in = d >= 1 && d <= D && i < K;
    const float v = sm.lp[in ? (d - 1) * K + i : 0];   // index kept in range
    return in ? v : 0.f;
  };
  if (lane == 0) {
    sm.node[0] = static_cast<uint32_t>(root);
    sm.node[1] = 0xFFFFFFFFu;  // parent -1
    sm.node[2] = 0;
    sm.node[3] = 0;
    // slot 0: the root's children (depth 1), candidate rank 1
    sm.slot[0] = make_uint4(pack_info(0, 1, 1), __float_as_uint(0.f),
                            __float_as_uint(__fadd_rn(0.f, lpat(1, 1))),
                            __float_as_uint(lpat(2, 0)));
  }
  __syncwarp();

  // ---- Algorithm 1 ----
  uint64_t key[NSL];
#pragma unroll
  for (int i = 0; i < NSL; ++i) key[i] = 0ull;
  int n = 0, n_slots = 0;
  uint32_t seq = 0;
  if (B > 0) {
    if (lane == 0) key[0] = make_key(__fadd_rn(0.f, sm.lp[0]), 0u, 0, 0);
    n_slots = 1;
    seq = 1;
  }
  uint64_t lbest = key[0];
  // record of this lane's best slot (loaded ahead of the reductions that may pick it)
  auto load_rec = [&]() {
    const int sl = static_cast<int>((static_cast<uint32_t>(lbest) >> 5) & 63u) * 32 + lane;
    return sm.slot[lbest != 0ull ? sl : 0];
  };
  uint4 brec = load_rec();
  while (n < B) {
    const uint32_t hi = static_cast<uint32_t>(lbest >> 32);
    const uint32_t lo = static_cast<uint32_t>(lbest);
    const uint32_t mhi = __reduce_max_sync(FULL, hi);
    const uint32_t mlo = __reduce_max_sync(FULL, hi == mhi ? lo : 0u);
    if (mlo == 0u) break;  // no candidate left
    const int w = static_cast<int>(mlo & 31u);
    const int wi = static_cast<int>((mlo >> 5) & 63u);
    // the popped candidate: its slot record, from the winner lane
    const uint32_t winfo = __shfl_sync(FULL, brec.x, w);
    const float wpsc = __uint_as_float(__shfl_sync(FULL, brec.y, w));
    const float s_sib = __uint_as_float(__shfl_sync(FULL, brec.z, w));
    const float lp_child = __uint_as_float(__shfl_sync(FULL, brec.w, w));
    const float wscore = from_ordered_bits(mhi);
    const int p = winfo & 0x7FF;
    const int d = (winfo >> 11) & 0x1F;
    const int r = (winfo >> 16) & 0xFFFF;
    ++n;
    const bool has_sib = r < K;
    const bool has_child = d < D;
    const float s_child = __fadd_rn(wscore, lp_child);
    const uint64_t sib_key = has_sib ? make_key(s_sib, seq, wi, w) : 0ull;
    seq += has_sib ? 1u : 0u;
    const int cslot = n_slots;
    const int co = cslot & 31, ci = cslot >> 5;
    const uint64_t child_key = has_child ? make_key(s_child, seq, ci, co) : 0ull;
    seq += has_child ? 1u : 0u;
    n_slots += has_child ? 1 : 0;
    // records: the node (lane 0); the advanced slot (winner): rank r+1, its next
    // sibling at rank r+2; the new slot (owner): the popped node's children
    const uint4 adv = make_uint4(pack_info(p, d, r + 1), __float_as_uint(wpsc),
                                 __float_as_uint(__fadd_rn(wpsc, lpat(d, r + 1))),
                                 __float_as_uint(lp_child));
    const uint4 opn = make_uint4(pack_info(n, d + 1, 1), __float_as_uint(wscore),
                                 __float_as_uint(__fadd_rn(wscore, lpat(d + 1, 1))),
                                 __float_as_uint(lpat(d + 2, 0)));
    const bool is_w = lane == w;
    const bool is_o = has_child && lane == co;
    if (lane == 0)
      *reinterpret_cast<uint4*>(sm.node + 4 * n) =
          make_uint4(0u, static_cast<uint32_t>(p), static_cast<uint32_t>(d),
                     static_cast<uint32_t>(r));
    if (is_w && has_sib) sm.slot[wi * 32 + w] = adv;
    if (is_o) sm.slot[cslot] = opn;
#pragma unroll
    for (int i = 0; i < NSL; ++i) {
      if (is_w && i == wi) key[i] = sib_key;
      if (is_o && i == ci) key[i] = child_key;
    }
    const uint64_t rescan = max_keys<NSL>(key);
    lbest = is_w ? rescan : (is_o ? umax64(lbest, child_key) : lbest);
    brec = load_rec();
  }
  __syncwarp();
  // the nodes' tokens, looked up once the pops are done (many loads in flight)
  for (int i = lane + 1; i <= n; i += 32) {
    const uint32_t* nd = sm.node + 4 * i;
    sm.node[4 * i] = static_cast<uint32_t>(sm.ids[(nd[2] - 1) * K + (nd[3] - 1)]);
  }
  __syncwarp();
  return n;
}

// Flattened tree and ancestor mask of request req from sm.node[0..n], one warp.
__device__ void write_tree(const WarpSmem& sm, int n, int B, int req, int lane,
                           int32_t* __restrict__ n_nodes_out, int32_t* __restrict__ tok_out,
                           int32_t* __restrict__ parent_out, int32_t* __restrict__ depth_out,
                           int32_t* __restrict__ rank_out, uint32_t* __restrict__ mask_out) {
  const int W = (B + 1 + 31) / 32;
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

// The same output written by every warp of the CTA: the flat arrays by thread,
// the mask 32 rows per warp at a time (stage: a [32][W] region per warp).
__device__ void write_tree_cta(const WarpSmem& sm, uint32_t* stage_all, int n, int B, int req,
                               int32_t* __restrict__ n_nodes_out, int32_t* __restrict__ tok_out,
                               int32_t* __restrict__ parent_out, int32_t* __restrict__ depth_out,
                               int32_t* __restrict__ rank_out, uint32_t* __restrict__ mask_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int W = (B + 1 + 31) / 32;
  const size_t nb_out = (size_t)req * (B + 1);
  for (int i = tid; i <= B; i += blockDim.x) {
    const bool live = i <= n;
    const uint4 rec = live ? *reinterpret_cast<const uint4*>(sm.node + 4 * i) : make_uint4(0, 0, 0, 0);
    tok_out[nb_out + i] = live ? static_cast<int32_t>(rec.x) : -1;
    parent_out[nb_out + i] = live ? static_cast<int32_t>(rec.y) : -1;
    depth_out[nb_out + i] = live ? static_cast<int32_t>(rec.z) : -1;
    rank_out[nb_out + i] = live ? static_cast<int32_t>(rec.w) : -1;
  }
  if (tid == 0) n_nodes_out[req] = n;
  uint32_t* stage = stage_all + (size_t)warp * 32 * W;
  uint32_t* mrow = mask_out + nb_out * W;
  for (int i0 = warp * 32; i0 <= B; i0 += 32 * nw) {
    for (int t = lane; t < 32 * W; t += 32) stage[t] = 0u;
    __syncwarp();
    const int i = i0 + lane;
    if (i <= n) {
      uint32_t* st = stage + lane * W;
      int j = i;
      while (true) {
        st[j >> 5] |= 1u << (j & 31);
        if (j == 0) break;
        j = static_cast<int>(sm.node[4 * j + 1]);
      }
    }
    __syncwarp();
    const int rows = min(32, B + 1 - i0);
    for (int t = lane; t < rows * W; t += 32) mrow[(size_t)i0 * W + t] = stage[t];
    __syncwarp();
  }
}

__device__ __forceinline__ WarpSmem carve_warp_smem(unsigned char* base, int D, int K, int B) {
  WarpSmem sm;
  size_t off = 0;
  sm.node = reinterpret_cast<uint32_t*>(base + off); off += align_up(sizeof(uint32_t) * 4 * (B + 1), 16);
  sm.slot = reinterpret_cast<uint4*>(base + off); off += align_up(sizeof(uint4) * (B + 1), 16);
  sm.lp = reinterpret_cast<float*>(base + off); off += align_up(sizeof(float) * D * K, 16);
  sm.ids = nullptr;
  sm.stage = reinterpret_cast<uint32_t*>(base + off);
  return sm;
}

// One request per warp (blockDim.x / 32 requests per CTA); NSL = key registers
// per lane, 32 * NSL >= B + 1 slots.
template <int NSL>
__global__ void __launch_bounds__(kBuildWarps * 32)
ddtree_build_kernel(int n_req, int D, int K, int B, const float* __restrict__ lp_g,
                    const int32_t* __restrict__ ids_g, const int32_t* __restrict__ root_tok,
                    int32_t* __restrict__ n_nodes_out, int32_t* __restrict__ tok_out,
                    int32_t* __restrict__ parent_out, int32_t* __restrict__ depth_out,
                    int32_t* __restrict__ rank_out, uint32_t* __restrict__ mask_out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int req = blockIdx.x * (blockDim.x >> 5) + wib;
  pdl_wait();
  pdl_trigger();
  if (req >= n_req) return;
  WarpSmem sm = carve_warp_smem(smem_raw + build_warp_bytes(D, K, B) * wib, D, K, B);
  const float* lp_r = lp_g + (size_t)req * D * K;
  sm.ids = ids_g + (size_t)req * D * K;
  for (int i = lane; i < D * K; i += 32) sm.lp[i] = lp_r[i];
  __syncwarp();
  const int n = seq_build<NSL>(sm, D, K, B, lane, root_tok[req]);
  write_tree(sm, n, B, req, lane, n_nodes_out, tok_out, parent_out, depth_out, rank_out,
             mask_out);
}

// ---------------------------------------------------------------------------
// Parallel construction for distinct scores.  When every depth's list is
// non-increasing and <= 0, a candidate never outscores its parent or its
// previous sibling, so the heap pops nodes in globally descending score order
// and the tree is the B best prefixes.  When no two of those scores are equal
// (and the B-th is strictly above every prefix left out) the creation-order
// rule never applies and the pop order is the descending score order.  One
// CTA finds that set depth by depth: the candidates of depth d are the children
// of the depth d-1 nodes still kept, a child below the current B-th best score
// is pruned, and a radix select over the order-preserving score bits keeps the
// best B.  Any equality met on the way (or an input outside the conditions)
// hands the request to the exact one-pop-at-a-time path.
// ---------------------------------------------------------------------------
constexpr int kFastThreads = 256;
constexpr int kFastMaxB = 1024;
constexpr int kFastMaxCand = 8192;   // candidate slots of one depth
constexpr int kFastSmemMax = 227 * 1024;

struct FastSmem {
  uint32_t* pkey[2];   // kept nodes: order-preserving score bits   [B]
  int* ppar[2];        //             parent (kept index, -1 root)  [B]
  int* pdr[2];         //             depth << 8 | rank             [B]
  uint32_t* ckey;      // candidates of one depth                   [B*K]
  int* cpar;
  int* cdr;
  int* newpos;         // old kept index -> new, later kept index -> node number [B]
  int* front;          // kept indices of the last depth            [B]
  uint32_t* skey;      // final sort                                [pow2 >= B]
  int* sidx;
  int* hist;           // [256]
  int* misc;           // [8]
  uint32_t* stage;     // mask staging, [kFastThreads / 32][32][W]
};

__host__ __device__ inline int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// cap: candidate slots of one depth (children above the current cut)
__host__ __device__ inline size_t fast_scratch_bytes(int cap, int B) {
  const size_t BK = (size_t)cap, N2 = pow2_at_least(B > 0 ? B : 1);
  const size_t W = (B + 1 + 31) / 32;
  return align_up(sizeof(int) * (6 * (size_t)B + 3 * BK + 2 * (size_t)B + 2 * N2 + 256 + 8), 16) +
         sizeof(uint32_t) * (kFastThreads / 32) * 32 * W;
}

__device__ __forceinline__ FastSmem carve_fast_smem(unsigned char* base, int cap, int B) {
  FastSmem f;
  int* q = reinterpret_cast<int*>(base);
  const int BK = cap, N2 = pow2_at_least(B > 0 ? B : 1);
  for (int b = 0; b < 2; ++b) {
    f.pkey[b] = reinterpret_cast<uint32_t*>(q); q += B;
    f.ppar[b] = q; q += B;
    f.pdr[b] = q; q += B;
  }
  f.ckey = reinterpret_cast<uint32_t*>(q); q += BK;
  f.cpar = q; q += BK;
  f.cdr = q; q += BK;
  f.newpos = q; q += B;
  f.front = q; q += B;
  f.skey = reinterpret_cast<uint32_t*>(q); q += N2;
  f.sidx = q; q += N2;
  f.hist = q; q += 256;
  f.misc = q;
  f.stage = reinterpret_cast<uint32_t*>(
      base + align_up(sizeof(int) * (6 * (size_t)B + 3 * (size_t)BK + 2 * (size_t)B + 2 * (size_t)N2 +
                                     256 + 8),
                      16));
  return f;
}

// Returns n (sm.node[0..n] filled) or -1 when the exact sequential path must
// decide.  Every thread of the CTA calls it; all branches are CTA-uniform.
__device__ int fast_build(const WarpSmem& sm, const FastSmem& f, int D, int K, int B, int cap,
                          int32_t root) {
  const int tid = threadIdx.x, T = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5;
  int* misc = f.misc;   // [0] count, [1] fallback, [2] kept, [3] frontier, [4..6] select, [7] min
  if (tid == 0) misc[1] = 0;
  __syncthreads();
  for (int i = tid; i < D * K; i += T) {
    const float v = sm.lp[i];
    bool bad = !(v <= 0.f);
    if (i % K != 0) bad = bad || !(sm.lp[i - 1] >= v);
    if (bad) misc[1] = 1;
  }
  __syncthreads();
  if (misc[1]) return -1;

  int cur = 0, n_p = 0, n_front = 1;
  bool full = false;
  uint32_t tau = 0;
  if (tid == 0) f.front[0] = -1;
  for (int d = 1; d <= D; ++d) {
    if (tid == 0) misc[0] = 0;
    __syncthreads();
    // candidates: children of the depth d-1 nodes still kept.  A depth's list
    // is non-increasing, so the children of a kept node that clear the cut
    // are a prefix of its ranks: count them by binary search, then lay them
    // out by prefix sums (offsets in newpos, free until the compaction).
    const uint32_t* pk = f.pkey[cur];
    const float* lpd = sm.lp + (d - 1) * K;
    int* offs = f.newpos;
    for (int i = tid; i < n_front; i += T) {
      const int fi = f.front[i];
      const float ps = fi < 0 ? 0.f : from_ordered_bits(pk[fi]);
      int lo = 0;
      if (!full) {
        lo = K;
      } else {
        int hi = K;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (ordered_bits(__fadd_rn(ps, lpd[mid])) > tau) lo = mid + 1;
          else hi = mid;
        }
        if (lo < K && ordered_bits(__fadd_rn(ps, lpd[lo])) == tau) misc[1] = 1;
      }
      offs[i] = lo;
    }
    __syncthreads();
    if (misc[1]) return -1;
    if (warp == 0) {
      // exclusive scan of the counts: lane l sums a contiguous segment
      const int seg = (n_front + 31) / 32;
      const int b0 = min(lane * seg, n_front), b1 = min(b0 + seg, n_front);
      int sum = 0;
      for (int i = b0; i < b1; ++i) sum += offs[i];
      int incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      int run = incl - sum;
      for (int i = b0; i < b1; ++i) {
        const int c = offs[i];
        offs[i] = run;
        run += c;
      }
      if (lane == 31) misc[0] = incl;
    }
    __syncthreads();
    const int n_c = misc[0];
    if (n_c > cap) return -1;   // more survivors than slots: the exact path decides
    for (int q = tid; q < n_c; q += T) {
      int lo = 0, hi = n_front - 1;   // the frontier node whose range holds q
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offs[mid] <= q) lo = mid;
        else hi = mid - 1;
      }
      const int fi = f.front[lo];
      const int r = q - offs[lo];
      const float ps = fi < 0 ? 0.f : from_ordered_bits(pk[fi]);
      f.ckey[q] = ordered_bits(__fadd_rn(ps, lpd[r]));
      f.cpar[q] = fi;
      f.cdr[q] = (d << 16) | (r + 1);
    }
    __syncthreads();
    if (n_c == 0) break;
    const int total = n_p + n_c;
    if (total <= B) {
      // everything fits: append, the new depth becomes the frontier
      for (int i = tid; i < n_c; i += T) {
        f.pkey[cur][n_p + i] = f.ckey[i];
        f.ppar[cur][n_p + i] = f.cpar[i];
        f.pdr[cur][n_p + i] = f.cdr[i];
        f.front[i] = n_p + i;
      }
      if (tid == 0) misc[7] = -1;   // 0xFFFFFFFF
      __syncthreads();
      n_p = total;
      n_front = n_c;
      if (n_p == B) {
        for (int i = tid; i < n_p; i += T)
          atomicMin(reinterpret_cast<unsigned int*>(&misc[7]), f.pkey[cur][i]);
        __syncthreads();
        full = true;
        tau = static_cast<uint32_t>(misc[7]);
      }
      continue;
    }
    // radix select of the B-th largest key over kept + candidates
    uint32_t prefix = 0, pmask = 0;
    int need = B;
    bool whole_bin = false;   // the chosen bin is taken whole: no cut inside it
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = tid; i < 256; i += T) f.hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < total; i += T) {
        const uint32_t key = i < n_p ? f.pkey[cur][i] : f.ckey[i - n_p];
        if ((key & pmask) == prefix) atomicAdd(&f.hist[(key >> shift) & 255], 1);
      }
      __syncthreads();
      if (warp == 0) {
        int c[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) { c[j] = f.hist[255 - 8 * lane - j]; sum += c[j]; }
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int o = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += o;
        }
        int run = incl - sum;   // keys in higher bins than this lane's
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run < need && run + c[j] >= need) {
            misc[4] = 255 - 8 * lane - j;
            misc[5] = run;
            misc[6] = c[j];
          }
          run += c[j];
        }
      }
      __syncthreads();
      prefix |= static_cast<uint32_t>(misc[4]) << shift;
      pmask |= 0xFFu << shift;
      need -= misc[5];
      if (misc[6] == need) {   // every key of the bin is kept: the bits below need no pass
        whole_bin = true;
        break;
      }
    }
    // equal scores straddling the cut: creation order decides
    if (!whole_bin && misc[6] > 1) return -1;
    const uint32_t cut = prefix;   // the kept keys are exactly those >= cut
    // compaction into the other buffer; accepted candidates form the next frontier
    const int nxt = cur ^ 1;
    if (tid == 0) { misc[2] = 0; misc[3] = 0; misc[7] = -1; }
    __syncthreads();
    for (int i = tid; i < total; i += T) {
      const bool old = i < n_p;
      const uint32_t key = old ? f.pkey[cur][i] : f.ckey[i - n_p];
      int slot = -1;
      if (key >= cut) {
        atomicMin(reinterpret_cast<unsigned int*>(&misc[7]), key);   // the new B-th best
        slot = atomicAdd(&misc[2], 1);
        f.pkey[nxt][slot] = key;
        f.ppar[nxt][slot] = old ? f.ppar[cur][i] : f.cpar[i - n_p];
        f.pdr[nxt][slot] = old ? f.pdr[cur][i] : f.cdr[i - n_p];
        if (!old) f.front[atomicAdd(&misc[3], 1)] = slot;
      }
      if (old) f.newpos[i] = slot;
    }
    __syncthreads();
    n_p = misc[2];
    n_front = misc[3];
    // parents to their new places (a kept node's parent is kept)
    for (int i = tid; i < n_p; i += T) {
      const int par = f.ppar[nxt][i];
      f.ppar[nxt][i] = par < 0 ? -1 : f.newpos[par];
    }
    __syncthreads();
    cur = nxt;
    full = true;
    tau = static_cast<uint32_t>(misc[7]);   // the smallest kept key (>= cut)
    if (n_front == 0) break;
  }

  // pop order = descending score: a kept node's position is the number of
  // kept keys above it (one pass, no sorting network); equal keys are left to
  // the exact sequential construction
  for (int i = tid; i < n_p; i += T) {
    const uint32_t ki = f.pkey[cur][i];
    int gt = 0, eq = 0;
    for (int j = 0; j < n_p; ++j) {
      const uint32_t kj = f.pkey[cur][j];
      gt += kj > ki ? 1 : 0;
      eq += kj == ki ? 1 : 0;
    }
    if (eq > 1) misc[1] = 1;
    f.sidx[gt < n_p ? gt : n_p - 1] = i;
    f.newpos[i] = gt + 1;   // kept index -> node number
  }
  __syncthreads();
  if (misc[1]) return -1;
  for (int i = tid; i < n_p; i += T) {
    const int idx = f.sidx[i];
    const int dr = f.pdr[cur][idx];
    const int dd = dr >> 16, rr = dr & 0xFFFF;
    const int par = f.ppar[cur][idx];
    *reinterpret_cast<uint4*>(sm.node + 4 * (i + 1)) =
        make_uint4(static_cast<uint32_t>(sm.ids[(dd - 1) * K + (rr - 1)]),
                   static_cast<uint32_t>(par < 0 ? 0 : f.newpos[par]), static_cast<uint32_t>(dd),
                   static_cast<uint32_t>(rr));
  }
  if (tid == 0) {
    sm.node[0] = static_cast<uint32_t>(root);
    sm.node[1] = 0xFFFFFFFFu;
    sm.node[2] = 0;
    sm.node[3] = 0;
  }
  __syncthreads();
  return n_p;
}

// One request per CTA: the parallel construction, else warp 0 runs the exact
// sequential one; warp 0 writes the tree.
template <int NSL>
__global__ void __launch_bounds__(kFastThreads)
ddtree_build_fast_kernel(int n_req, int D, int K, int B, int cap, const float* __restrict__ lp_g,
                         const int32_t* __restrict__ ids_g, const int32_t* __restrict__ root_tok,
                         int32_t* __restrict__ n_nodes_out, int32_t* __restrict__ tok_out,
                         int32_t* __restrict__ parent_out, int32_t* __restrict__ depth_out,
                         int32_t* __restrict__ rank_out, uint32_t* __restrict__ mask_out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int req = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_wait();
  pdl_trigger();
  if (req >= n_req) return;
  WarpSmem sm = carve_warp_smem(smem_raw, D, K, B);
  const FastSmem fs = carve_fast_smem(smem_raw + build_warp_bytes(D, K, B), cap, B);
  const float* lp_r = lp_g + (size_t)req * D * K;
  sm.ids = ids_g + (size_t)req * D * K;
  for (int i = threadIdx.x; i < D * K; i += blockDim.x) sm.lp[i] = lp_r[i];
  __syncthreads();
  const int32_t root = root_tok[req];
  int n = fast_build(sm, fs, D, K, B, cap, root);
  if (n < 0) {
    // (uniform: every thread saw the same flag)
    if (warp == 0) {
      n = seq_build<NSL>(sm, D, K, B, lane, root);
      if (lane == 0) fs.misc[0] = n;
    }
    __syncthreads();
    n = fs.misc[0];
  }
  write_tree_cta(sm, fs.stage, n, B, req, n_nodes_out, tok_out, parent_out, depth_out, rank_out,
                 mask_out);
}

template <int NSL>
void launch_build_t(const TreeBuildLaunch& a, cudaStream_t st) {
  // candidate slots per depth: B * K when that fits, else as many as the
  // shared memory holds (a depth with more survivors takes the exact path)
  int cap = (long long)a.B * a.K < kFastMaxCand ? a.B * a.K : kFastMaxCand;
  while (cap > 1024 &&
         build_warp_bytes(a.D, a.K, a.B) + fast_scratch_bytes(cap, a.B) > (size_t)kFastSmemMax)
    cap /= 2;
  const size_t fast_smem = build_warp_bytes(a.D, a.K, a.B) + fast_scratch_bytes(cap, a.B);
  const bool fast = a.B >= 1 && a.B <= kFastMaxB && cap >= a.K &&
                    fast_smem <= (size_t)kFastSmemMax;
  TraceScope ts("ddtree_build", st);
  if (fast) {
    static bool attr_fast = false;  // per instantiation, per process
    if (!attr_fast) {
      cudaFuncSetAttribute(ddtree_build_fast_kernel<NSL>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, kFastSmemMax);
      attr_fast = true;
    }
    const size_t smem = fast_smem;
    launch_k(ddtree_build_fast_kernel<NSL>, dim3(a.n_req), dim3(kFastThreads), smem, st, a.n_req,
             a.D, a.K, a.B, cap, a.topk_logp, a.topk_ids, a.root_tok, a.n_nodes, a.tok, a.parent,
             a.depth, a.rank, a.mask);
    return;
  }
  static bool attr_set = false;  // per instantiation, per process
  if (!attr_set) {
    cudaFuncSetAttribute(ddtree_build_kernel<NSL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kBuildSmemMax);
    attr_set = true;
  }
  // as many requests per CTA (up to kBuildWarps) as the shared memory holds
  const size_t per_warp = build_warp_bytes(a.D, a.K, a.B);
  int wpc = static_cast<int>(kBuildSmemMax / per_warp);
  wpc = wpc < 1 ? 1 : (wpc > kBuildWarps ? kBuildWarps : wpc);
  const size_t smem = per_warp * wpc;
  dim3 grid(ceil_div(a.n_req, wpc));
  launch_k(ddtree_build_kernel<NSL>, grid, dim3(wpc * 32), smem, st, a.n_req, a.D, a.K,
           a.B, a.topk_logp, a.topk_ids, a.root_tok, a.n_nodes, a.tok, a.parent, a.depth, a.rank,
           a.mask);
}

void launch_build(const TreeBuildLaunch& a, cudaStream_t st) {
  const int slots = a.B + 1;
  if (slots <= 32) launch_build_t<1>(a, st);
  else if (slots <= 64) launch_build_t<2>(a, st);
  else if (slots <= 96) launch_build_t<3>(a, st);
  else if (slots <= 160) launch_build_t<5>(a, st);
  else if (slots <= 288) launch_build_t<9>(a, st);
  else if (slots <= 544) launch_build_t<17>(a, st);
  else launch_build_t<33>(a, st);
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

// The vanilla DFlash chain in the tree layout: one CTA per request writes the
// node arrays and the lower-triangular mask (row i: bits 0..i) of all B + 1
// rows; rows past node n are -1 / zero.
__global__ void chain_tree_kernel(int D, int K, int B, const int32_t* __restrict__ topk_ids,
                                  const int32_t* __restrict__ root_tok,
                                  int32_t* __restrict__ n_nodes, int32_t* __restrict__ tok,
                                  int32_t* __restrict__ parent, int32_t* __restrict__ depth,
                                  int32_t* __restrict__ rank, uint32_t* __restrict__ mask) {
  const int req = blockIdx.x;
  const int W1 = B + 1;
  const int words = (W1 + 31) / 32;
  const int n = min(D, B);
  pdl_wait();
  pdl_trigger();
  const size_t nb = (size_t)req * W1;
  for (int i = threadIdx.x; i < W1; i += blockDim.x) {
    const bool live = i <= n;
    tok[nb + i] = !live ? -1 : i == 0 ? root_tok[req] : topk_ids[((size_t)req * D + i - 1) * K];
    parent[nb + i] = live ? i - 1 : -1;
    depth[nb + i] = live ? i : -1;
    rank[nb + i] = !live ? -1 : i == 0 ? 0 : 1;
  }
  uint32_t* mrow = mask + nb * words;
  for (int e = threadIdx.x; e < W1 * words; e += blockDim.x) {
    const int i = e / words, lo = (e % words) * 32;
    uint32_t bits = 0u;
    if (i <= n && i >= lo) {
      const int top = min(i - lo, 31);   // bits 0..top of this word
      bits = top == 31 ? 0xffffffffu : (2u << top) - 1u;
    }
    mrow[e] = bits;
  }
  if (threadIdx.x == 0) n_nodes[req] = n;
}

void launch_chain_tree(const TreeBuildLaunch& a, cudaStream_t st) {
  if (a.n_req <= 0) return;
  TraceScope ts("chain_tree", st);
  launch_k(chain_tree_kernel, dim3(a.n_req), dim3(256), 0, st, a.D, a.K, a.B, a.topk_ids,
           a.root_tok, a.n_nodes, a.tok, a.parent, a.depth, a.rank, a.mask);
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
