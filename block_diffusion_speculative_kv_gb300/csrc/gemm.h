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
TcPlan tc_plan(int M_rows, int N_feat, int K, int grid, int tk_kpad = 0);

// 2-D TMA map of a K-major bf16 matrix [rows][K] (row stride in elements),
// box = 64 x box_rows, 128-byte swizzle.  False if the driver entry point is
// unavailable or the arguments are rejected.
bool encode_kmajor_map(CUtensorMap* map, const void* base, int rows, int K,
                       long long row_stride_elems, int box_rows);

// One phase of a GEMM chain: acc = X . W^T, then the epilogue.
struct GemmPhase {
  const CUtensorMap* tmW;  // weight map [N][K], box 64 x 128 (encode_kmajor_map)
  const void* X;           // activations [M_rows][K] bf16, row stride ldx elements
  long long ldx;
  int N, K;
  EpiParams epi;
};

constexpr int kMaxPhases = 4;

// Runs n_phases dependent GEMMs over the same M_rows activation rows in one
// launch (gemm_tc.cu), one CTA per SM.  Phase k may read what phases < k wrote.
// part: split-tile partial sums, at least the largest tc_plan(...).part_bytes
// over the phases with grid = num_sms(); counters: gemm_counter_ints() ints,
// zero before the first launch and left at zero by every launch.
dflash_status launch_gemm_chain(const GemmPhase* ph, int n_phases, int M_rows, float* part,
                                int* counters, int* status, cudaStream_t st);
int gemm_counter_ints();

// fp32 CUDA-core GEMM with the same epilogues: X [M_rows][K] fp32 (row stride
// ldx), W [N_feat][K] fp32.  One CTA per (128-column tile, 16-row chunk).
dflash_status launch_gemm_f32(const float* X, long long ldx, const float* W, int M_rows,
                              int N_feat, int K, const EpiParams& epi, cudaStream_t st);

}  // namespace dfl
