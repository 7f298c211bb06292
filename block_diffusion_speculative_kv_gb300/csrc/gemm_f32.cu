// fp32 GEMM on the CUDA cores, for models whose dtype is fp32 (the tensor-core
// path is bf16-only; tf32 would not meet fp32 accuracy).  acc = X . W^T with
// the same fused epilogues as the tensor-core path (epilogue.cuh).
//
// One CTA per (128-column tile, 16-row chunk), 128 threads: thread f owns
// column f of the tile and accumulates its 16 rows.  K is walked in 32-wide
// slabs staged in shared memory (W transposed so a warp reads 32 consecutive
// columns; X broadcast), with bounds checks for ragged N, M and K.
#include "common.cuh"
#include "epilogue.cuh"
#include "gemm.h"

namespace dfl {

namespace {

constexpr int kKs = 32;

__global__ void __launch_bounds__(128)
gemm_f32_kernel(const float* __restrict__ X, long long ldx, const float* __restrict__ W,
                int M_rows, int N_feat, int K, const EpiParams e) {
  __shared__ float sW[kKs][kTileN + 1];
  __shared__ float sX[kChunk][kKs + 1];
  __shared__ float buf[kChunk * kBufLd];
  __shared__ float s_scale[kChunk];
  __shared__ float s_red[4 * kChunk];

  const int f = threadIdx.x;
  const int ftile = blockIdx.x;
  const int row0 = blockIdx.y * kChunk;
  const int col0 = ftile * kTileN;
  const int nrows = min(kChunk, M_rows - row0);
  pdl_wait();
  pdl_trigger();

  float acc[kChunk];
#pragma unroll
  for (int r = 0; r < kChunk; ++r) acc[r] = 0.f;

  for (int k0 = 0; k0 < K; k0 += kKs) {
    // W slab: 128 rows x 32 k, read row-wise (coalesced along k), stored transposed
    for (int i = threadIdx.x; i < kTileN * kKs; i += 128) {
      const int rr = i / kKs, kk = i % kKs;
      const int col = col0 + rr, k = k0 + kk;
      sW[kk][rr] = (col < N_feat && k < K) ? W[(size_t)col * K + k] : 0.f;
    }
    for (int i = threadIdx.x; i < kChunk * kKs; i += 128) {
      const int rr = i / kKs, kk = i % kKs;
      const int row = row0 + rr, k = k0 + kk;
      sX[rr][kk] = (row < M_rows && k < K) ? X[(size_t)row * ldx + k] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < kKs; ++kk) {
      const float w = sW[kk][f];
#pragma unroll
      for (int r = 0; r < kChunk; ++r) acc[r] = fmaf(sX[r][kk], w, acc[r]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int r = 0; r < kChunk; ++r) buf[r * kBufLd + f] = acc[r];
  epi_row_scales(e, row0, nrows, s_scale, threadIdx.x, 128);
  for (int i = threadIdx.x; i < 4 * kChunk; i += 128) s_red[i] = 0.f;
  __syncthreads();
  EpiPre pre;
  epi_preload<float>(e, col0, row0, nrows, f, pre);
  epi_apply_chunk<float>(e, buf, col0, row0, nrows, f, s_scale, row0, s_red, kChunk,
                         threadIdx.x >> 5, pre);
  if (e.kind == EPI_RESID) {
    __syncthreads();
    epi_resid_flush(e, ftile, row0, nrows, s_red, kChunk, 4, threadIdx.x, 128);
  }
}

}  // namespace

dflash_status launch_gemm_f32(const float* X, long long ldx, const float* W, int M_rows,
                              int N_feat, int K, const EpiParams& epi, cudaStream_t st) {
  if (M_rows <= 0) return DFLASH_OK;
  dim3 grid(ceil_div(N_feat, kTileN), ceil_div(M_rows, kChunk));
  TraceScope ts("gemm_f32", st);
  launch_k(gemm_f32_kernel, grid, dim3(128), 0, st, X, ldx, W, M_rows, N_feat, K, epi);
  return check_launch("gemm_f32");
}

}  // namespace dfl
