// Internal launch interface between the C ABI layer (abi.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

#include "dflash.h"

namespace dfl {

// ---- log-softmax + top-K (topk.cu) ----
// Temperature sampling of a top-K pass (inv_t == 0: plain top-K).
struct SampleSpec {
  float inv_t = 0.f, t = 0.f;
  uint64_t seed = 0;
  long long row0 = 0;
};
// Validates a dflash_sampling (NULL or temperature 0: plain top-K).
dflash_status parse_sampling(const dflash_sampling* s, SampleSpec* out);

struct TopkLaunch {
  const void* logits;
  int rows, vocab;
  long long ld;
  int dtype;      // DFLASH_F32 / DFLASH_BF16
  int K;          // <= 32
  int splits;     // <= 32; 1 = one CTA per row, no partial records
  float* part;    // [rows][splits][2 + 2*32] when splits > 1
  int* counters;  // [rows], zero on entry, left zero on exit
  int32_t* ids;
  float* logp;
  // temperature sampling (inv_t > 0): rank Gumbel scores of counter rows
  // row0 + r under seed; inv_t = 1/T, t = T.  Zero-initialised: plain top-K.
  float inv_t, t;
  uint64_t seed;
  long long row0;
  int* status;    // workspace status word for a bounded wait that runs out, or null
};
int topk_splits(int rows, int vocab);
// K <= 8 without sampling, 16-byte aligned rows (topk_stream.cu): the streamed
// pass; launch_topk takes it whenever topk_stream_supported holds.
bool topk_stream_supported(const TopkLaunch& a);
int topk_stream_workers();   // pieces the streamed pass works on at once (its warps)
void launch_topk_stream(const TopkLaunch& a, cudaStream_t st);
// K in (32, 1024] (topk_large.cu): two passes, partial records in `part` of
// topk_large_part_bytes bytes (no zeroing needed); plain top-K only.
int topk_large_splits(int vocab);
size_t topk_large_part_bytes(int rows, int vocab, int K);
size_t topk_large_merge_smem(int vocab, int K);
dflash_status launch_topk_large(const TopkLaunch& a, void* part, cudaStream_t st);
size_t topk_part_bytes(int rows, int splits);
void launch_topk(const TopkLaunch& a, cudaStream_t st);

// ---- DDTree (ddtree.cu) ----
struct TreeBuildLaunch {
  int n_req, D, K, B;
  const float* topk_logp;
  const int32_t* topk_ids;
  const int32_t* root_tok;
  int32_t* n_nodes;
  int32_t* tok;
  int32_t* parent;
  int32_t* depth;
  int32_t* rank;
  uint32_t* mask;
};
size_t tree_build_smem_bytes(int D, int K, int B);
void launch_tree_build(const TreeBuildLaunch& a, cudaStream_t st);
// The chain of topk_ids[.][.][0] in the same layout (topk_logp unused).
void launch_chain_tree(const TreeBuildLaunch& a, cudaStream_t st);

// The accepted path into the next injection's inputs (commit.cu).
struct CommitLaunch {
  int n_req, D, B;
  int row_bytes;              // bytes of one feature row (a multiple of 16)
  const void* tree_feats;     // [n_req][B+1] rows of tree_row_bytes
  long long tree_row_bytes;
  const int32_t* accept_len;
  const int32_t* accepted;
  const int32_t* bonus;
  int32_t* ctx_len;
  int32_t* anchor;
  int32_t* row_off;
  int32_t* pos0;
  void* feats;                // [n_req * (D+1)] rows of row_bytes
};
void launch_commit(const CommitLaunch& a, cudaStream_t st);

struct TreeAcceptLaunch {
  int n_req, D, B;
  const int32_t* n_nodes;
  const int32_t* tok;
  const int32_t* parent;
  const int32_t* target;
  int32_t* accept_len;
  int32_t* accepted;
  int32_t* bonus;
};
void launch_tree_accept(const TreeAcceptLaunch& a, cudaStream_t st);

// ---- block prologue and rotary tables (prologue.cu) ----
// Rotary frequencies theta^(-2i/head_dim), i < head_dim/2, in double precision.
struct RopeFreqs {
  double f[64];
};
RopeFreqs rope_freqs(float theta, int head_dim);
// (cos, sin) of pos * f[i]: the angle is formed and reduced modulo 2*pi in
// double (three FP64 operations), its sine and cosine taken in fp32.
__device__ __forceinline__ float2 rope_cs(int pos, int i, const RopeFreqs& fr) {
  const double two_pi = 6.283185307179586476925;
  const double a = static_cast<double>(pos) * fr.f[i];
  const double k = rint(a * (1.0 / two_pi));
  const float r = static_cast<float>(fma(-k, two_pi, a));
  float s, c;
  sincosf(r, &s, &c);
  return make_float2(c, s);
}

struct BlockPrologueLaunch {
  bool bf16;
  const void* embed;   // [vocab][d]
  const void* gain;    // [d] first attention-norm gain
  const int* anchor;   // [n_req]
  const int* ctx_len;  // [n_req]
  int n_req, L, d, vocab, mask_id, head_dim;
  RopeFreqs freqs;
  float* x;            // [n_req*L][d] fp32
  void* xn;            // [n_req*L][d] T
  float* ssq;          // [ceil(d/128)][n_req*L]
  float2* rope;        // [n_req*L][head_dim/2]
  int* status;
};
void launch_block_prologue(const BlockPrologueLaunch& a, cudaStream_t st);
void launch_inject_rope(const int* row_off, const int* pos0, int n_req, int n_rows, int head_dim,
                        const RopeFreqs& freqs, float2* rope, cudaStream_t st);

}  // namespace dfl
