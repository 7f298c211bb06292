// Attention launch interface (attention.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace dfl {

// bf16 split-KV attention of one layer.  qkv: [n_req*L][qkv_ld] with Q at
// column 0, the block's K at n_q*hd and V at (n_q+n_kv)*hd; cache_k/v:
// [n_req][n_kv][cap][hd]; out: [n_req*L][out_ld], head h at column h*hd.
struct AttnParams {
  const __nv_bfloat16* qkv;
  long long qkv_ld;
  const __nv_bfloat16* cache_k;
  const __nv_bfloat16* cache_v;
  const int* ctx_len;
  int cap;
  int n_req, n_q, n_kv, G, L;
  int chunk;      // context keys per CTA (multiple of 64)
  int n_chunks;   // chunks per (request, KV head); the last also takes the block keys
  float scale_log2;
  int anchor_sees_block;
  float* part_o;   // [n_req][n_kv][n_chunks][G*L][hd]
  float* part_ml;  // [n_req][n_kv][n_chunks][G*L][2]
  __nv_bfloat16* out;
  long long out_ld;
  // tree attention only (0 otherwise): query tiles per request, and the
  // output's rows per request (B + 1)
  int n_qt;
  int out_rows;
};

struct AttnParamsF32 {
  const float* qkv;
  long long qkv_ld;
  const float* cache_k;
  const float* cache_v;
  const int* ctx_len;
  int cap;
  int n_req, n_q, n_kv, L;
  int anchor_sees_block;
  float* out;
  long long out_ld;
};

int attn_chunk(int max_ctx, int n_kv, int n_req);
size_t attn_smem_bytes(int G, int L, int HD);
dflash_status launch_attention_bf16(const AttnParams& p, int head_dim, cudaStream_t st);
// the merge of the split partials alone (grid: row blocks of 4, KV heads, blockIdx.z units)
void launch_attn_combine(const AttnParams& p, int head_dim, dim3 cgrid, cudaStream_t st);
dflash_status launch_attention_f32(const AttnParamsF32& p, int head_dim, cudaStream_t st);
// The same block attention on the tensor cores (tree_attention.cu): head_dim
// 128, G <= 4, L <= 32, p.chunk a multiple of 128 keys.  The block keys ride in
// the chunk holding each request's context end; the last of a (request, KV
// head)'s chunks to finish merges their partials.  arrivals: n_req * n_kv ints,
// zero before the call and left at zero; status: the workspace status word.
dflash_status launch_block_attention_tc(const AttnParams& p, int* arrivals, int* status,
                                        cudaStream_t st);

}  // namespace dfl
