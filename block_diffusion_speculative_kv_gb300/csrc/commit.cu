// Steady-state bookkeeping between two draft cycles: the accepted path becomes
// context of the drafter.
//
// "DFlash: Block Diffusion for Flash Speculative Decoding", section 3.4.3:
// the target's hidden features of the verified tokens are injected into the
// drafter's cache as context, and the cache is reused across cycles; the
// DDTree page, section 3.4.5: after verification only the accepted path
// stays.  Per request r, with a = accept_len[r]:
//   - the a + 1 tokens of the accepted path (the root, i.e. this cycle's
//     anchor, and the accepted nodes in depth order) sit at positions
//     ctx_len[r] .. ctx_len[r] + a; their feature rows are gathered from the
//     target's per-node features into the next injection's rows,
//     row_off[r] .. row_off[r] + a (row_off the prefix sums of a + 1);
//   - pos0[r] = ctx_len[r], then ctx_len[r] += a + 1, and the bonus token is
//     the next anchor.
// The drafter's own block keys and values never enter the cache (they live in
// the workspace for one pass), so rejected draft positions leave nothing to
// roll back: the cache only ever receives accepted context.
#include "common.cuh"
#include "kernels.h"

namespace dfl {

namespace {

constexpr int kCommitThreads = 256;

__global__ void __launch_bounds__(kCommitThreads)
commit_kernel(int n_req, int D, int B, int row_bytes, const uint8_t* __restrict__ tree_feats,
              long long tree_row_bytes, const int32_t* __restrict__ accept_len,
              const int32_t* __restrict__ accepted, const int32_t* __restrict__ bonus,
              int32_t* __restrict__ ctx_len, int32_t* __restrict__ anchor,
              int32_t* __restrict__ row_off, int32_t* __restrict__ pos0,
              uint8_t* __restrict__ feats) {
  __shared__ int s_part[kCommitThreads / 32];
  __shared__ int s_off;
  const int r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  pdl_trigger();
  auto tau_of = [&](int j) { return min(max(accept_len[j], 0), D) + 1; };
  // row offset of request r: the accepted-path lengths of the requests before it
  int part = 0;
  for (int j = tid; j < r; j += kCommitThreads) part += tau_of(j);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
  if (lane == 0) s_part[warp] = part;
  __syncthreads();
  if (tid == 0) {
    int off = 0;
    for (int w = 0; w < kCommitThreads / 32; ++w) off += s_part[w];
    s_off = off;
  }
  __syncthreads();
  const int off = s_off;
  const int tau = tau_of(r);
  // gather the feature rows of the path (16-byte pieces)
  const int pieces = row_bytes / 16;
  for (int e = tid; e < tau * pieces; e += kCommitThreads) {
    const int i = e / pieces, q = e - i * pieces;
    int node = i == 0 ? 0 : accepted[(size_t)r * D + i - 1];
    node = min(max(node, 0), B);
    const uint4* src = reinterpret_cast<const uint4*>(
        tree_feats + ((size_t)r * (B + 1) + node) * tree_row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(feats + (size_t)(off + i) * row_bytes);
    dst[q] = __ldg(src + q);
  }
  if (tid == 0) {
    row_off[r] = off;
    if (r == n_req - 1) row_off[n_req] = off + tau;
    const int c = ctx_len[r];
    pos0[r] = c;
    ctx_len[r] = c + tau;
    anchor[r] = bonus[r];
  }
}

}  // namespace

void launch_commit(const CommitLaunch& a, cudaStream_t st) {
  if (a.n_req <= 0) return;
  TraceScope ts("commit", st);
  launch_k(commit_kernel, dim3(a.n_req), dim3(kCommitThreads), 0, st, a.n_req, a.D, a.B,
           a.row_bytes, static_cast<const uint8_t*>(a.tree_feats), a.tree_row_bytes,
           a.accept_len, a.accepted, a.bonus, a.ctx_len, a.anchor, a.row_off, a.pos0,
           static_cast<uint8_t*>(a.feats));
}

}  // namespace dfl
