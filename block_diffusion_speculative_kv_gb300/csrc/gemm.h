// GEMM launch interface (tcgen05 bf16 path and the fp32 CUDA-core path).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "epilogue.cuh"

namespace dfl {

// Work decomposition of one tensor-core GEMM launch (see gemm_tc.cu).
struct TcPlan {
  int n_tile, n_rtiles, n_ftiles, kblocks;
  long long total_units;
  int grid;
  int max_slots;
  size_t part_bytes;  // split-tile partial sums: [grid][max_slots][n_tile][128] fp32
  int stages;
  int smem_bytes;
};

int tc_row_tile(int M_rows);
TcPlan tc_plan(int M_rows, int N_feat, int K, int grid_max);

// 2-D TMA map of a K-major bf16 matrix [rows][K] (row stride in elements),
// box = 64 x box_rows, 128-byte swizzle.  False if the driver entry point is
// unavailable or the arguments are rejected.
bool encode_kmajor_map(CUtensorMap* map, const void* base, int rows, int K,
                       long long row_stride_elems, int box_rows);

dflash_status launch_gemm_tc(const CUtensorMap& tmW, const CUtensorMap& tmX, const TcPlan& pl,
                             int M_rows, int N_feat, int K, float* part, int* counters,
                             int* status, const EpiParams& epi, cudaStream_t st);

// fp32 CUDA-core GEMM with the same epilogues: X [M_rows][K] fp32 (row stride
// ldx), W [N_feat][K] fp32.  One CTA per (128-column tile, 16-row chunk).
dflash_status launch_gemm_f32(const float* X, long long ldx, const float* W, int M_rows,
                              int N_feat, int K, const EpiParams& epi, cudaStream_t st);

}  // namespace dfl
