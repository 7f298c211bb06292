// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Computes acc = X . W^T for every dense contraction of the drafter pass
// (fusion, injection, QKV, O, gate/up, down, LM head) and applies a fused
// epilogue (epilogue.cuh).  W is [N_feat][K] bf16 (a weight matrix), X is
// [M_rows][K] bf16 (activations).
//
// Mapping.  The MMA's M side (128 TMEM lanes) is a 128-row slice of W, its N
// side is a tile of n_tile activation rows (16 at batch 1, up to 256), so a
// tile of output is D[128 features][n_tile rows] in TMEM.  Work units are
// (tile, 64-wide K block) pairs; the grid is one CTA per SM and CTA c owns the
// contiguous unit range [c*U/G, (c+1)*U/G) (stream-K), so every SM streams the
// same number of weight bytes whatever the matrix shape.  A tile whose K range
// is split over several CTAs is reduced by the last CTA to arrive (an atomic
// counter; no CTA ever waits for another), adding the partial sums in a fixed
// order so results do not depend on timing.
//
// Roles (6 warps): warp 0 lane 0 issues TMA loads into a multi-stage shared
// memory ring (weights evict-first, activations evict-last in L2); warp 1
// owns the TMEM allocation and its lane 0 issues tcgen05.mma (128 x n_tile x 16,
// four per 64-wide K block) and tcgen05.commit to release ring slots; warps
// 2-5 drain TMEM (tcgen05.ld, 32 lanes each) and run the epilogue.  A CTA's
// tiles alternate between two TMEM accumulators, so the MMAs of the next tile
// never wait for the epilogue of the previous one.  Every
// mbarrier wait is bounded in time; on expiry the CTA records
// DFLASH_ERR_TIMEOUT in the status word, drains its outstanding copies and
// MMAs (again bounded), frees TMEM and exits.
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "epilogue.cuh"
#include "gemm.h"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kABytes = kTileN * 128;  // 128 weight rows x 64 bf16
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct TcParams {
  int M_rows, N_feat, K;
  int n_tile;
  int n_rtiles, kblocks;
  long long total_units;
  int stages;
  float* part;     // [grid][max_slots][n_tile][128]
  int max_slots;
  int* counters;   // [grid]
  int* status;
  EpiParams epi;
};

__host__ __device__ __forceinline__ int cta_of_unit(long long u, long long U, int G) {
  return static_cast<int>(((u + 1) * G - 1) / U);
}

struct SmemLayout {
  uint32_t a_off, b_off, bar_off, buf_off, scale_off, red_off, total;
};

__host__ __device__ inline SmemLayout smem_layout(int stages, int n_tile) {
  SmemLayout L;
  const uint32_t b_bytes = n_tile * 128;
  L.a_off = 0;
  L.b_off = stages * kABytes;
  L.bar_off = L.b_off + stages * b_bytes;
  const uint32_t bar_bytes = (2 * stages + 5) * 8 + 16 + 16;
  L.buf_off = (L.bar_off + bar_bytes + 15) / 16 * 16;
  L.scale_off = L.buf_off + kChunk * kBufLd * 4;
  L.red_off = L.scale_off + n_tile * 4;
  L.total = L.red_off + 4 * n_tile * 4 + 1024;  // + alignment slack for the 1024-B base
  return L;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
               const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const SmemLayout SL = smem_layout(p.stages, p.n_tile);
  const uint32_t b_bytes = p.n_tile * 128;
  uint8_t* sA = smem + SL.a_off;
  uint8_t* sB = smem + SL.b_off;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SL.bar_off);
  uint64_t* empty = full + p.stages;
  uint64_t* accf = empty + p.stages;   // [2] accumulator a holds a finished tile
  uint64_t* acce = accf + 2;           // [2] accumulator a has been drained
  uint64_t* drain = acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 4);  // [0] abort, [1] last
  float* buf = reinterpret_cast<float*>(smem + SL.buf_off);
  float* s_scale = reinterpret_cast<float*>(smem + SL.scale_off);
  float* s_red = reinterpret_cast<float*>(smem + SL.red_off);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int c = blockIdx.x;
  const long long U = p.total_units;
  const long long u_begin = (long long)c * U / G;
  const long long u_end = (long long)(c + 1) * U / G;
  const int KB = p.kblocks;
  // two accumulators of n_tile columns: the MMAs of a CTA's next tile run while
  // the epilogue drains the previous one
  const uint32_t tmem_cols = 2 * p.n_tile < 32 ? 32u : static_cast<uint32_t>(2 * p.n_tile);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&accf[a], 1);
      ptx::mbar_init(&acce[a], kEpiThreads);
    }
    ptx::mbar_init(drain, 1);
    flags[0] = 0;
    flags[1] = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmW);
    ptx::prefetch_tmap(&tmX);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const bool producer = (warp == 0 && lane == 0);
  if (!producer) {
    pdl_wait();
    pdl_trigger();
  }

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t pol_w = ptx::policy_evict_first();
      const uint64_t pol_x = ptx::policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase_mask = 0;  // bit s: stage s has an issued copy
      uint32_t last_phase[32];
      // Weights are never written by a kernel: the first ring slots' weight
      // tiles are requested before waiting for the previous kernel, the
      // activation tiles (its output) after.
      const int pre = static_cast<int>(
          (u_end - u_begin) < p.stages ? (u_end - u_begin) : p.stages);
      for (int i = 0; i < pre; ++i) {
        const long long u = u_begin + i;
        const int t = static_cast<int>(u / KB);
        const int kb = static_cast<int>(u - (long long)t * KB);
        const int ftile = t / p.n_rtiles;
        ptx::mbar_arrive_expect_tx(&full[i], kABytes + b_bytes);
        ptx::tma_load_2d(sA + i * kABytes, &tmW, &full[i], kb * 64, ftile * kTileN, pol_w);
      }
      pdl_wait();
      pdl_trigger();
      for (int i = 0; i < pre; ++i) {
        const long long u = u_begin + i;
        const int t = static_cast<int>(u / KB);
        const int kb = static_cast<int>(u - (long long)t * KB);
        const int ftile = t / p.n_rtiles;
        const int rtile = t - ftile * p.n_rtiles;
        ptx::tma_load_2d(sB + i * b_bytes, &tmX, &full[i], kb * 64, rtile * p.n_tile, pol_x);
        issued_phase_mask |= 1u << i;
        last_phase[i] = 0;
      }
      stage = pre % p.stages;
      phase = (pre == p.stages) ? 1u : 0u;
      for (long long u = u_begin + pre; u < u_end; ++u) {
        const int t = static_cast<int>(u / KB);
        const int kb = static_cast<int>(u - (long long)t * KB);
        const int ftile = t / p.n_rtiles;
        const int rtile = t - ftile * p.n_rtiles;
        if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, kTimeoutNs, flags)) {
          record_status(p.status, DFLASH_ERR_TIMEOUT);
          flags[0] = 1;
          break;
        }
        ptx::mbar_arrive_expect_tx(&full[stage], kABytes + b_bytes);
        ptx::tma_load_2d(sA + stage * kABytes, &tmW, &full[stage], kb * 64, ftile * kTileN,
                         pol_w);
        ptx::tma_load_2d(sB + stage * b_bytes, &tmX, &full[stage], kb * 64, rtile * p.n_tile,
                         pol_x);
        issued_phase_mask |= 1u << stage;
        last_phase[stage] = phase;
        if (++stage == p.stages) { stage = 0; phase ^= 1u; }
      }
      if (flags[0]) {
        // drain: every issued copy must land before the CTA may exit
        for (int s = 0; s < p.stages; ++s)
          if (issued_phase_mask & (1u << s))
            ptx::mbar_wait_bounded(&full[s], last_phase[s], kTimeoutNs, nullptr);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(128, p.n_tile);
      int stage = 0;
      uint32_t phase = 0;
      int tile_i = 0;   // tiles of this CTA so far: accumulator tile_i & 1
      bool issued_any = false;
      long long u = u_begin;
      while (u < u_end && !flags[0]) {
        const int t = static_cast<int>(u / KB);
        const int kb0 = static_cast<int>(u - (long long)t * KB);
        const int n = static_cast<int>((KB - kb0) < (u_end - u) ? (KB - kb0) : (u_end - u));
        const int acc = tile_i & 1;
        const uint32_t acc_phase = static_cast<uint32_t>(tile_i >> 1) & 1u;
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * p.n_tile);
        if (!ptx::mbar_wait_bounded(&acce[acc], acc_phase ^ 1u, kTimeoutNs, flags)) {
          record_status(p.status, DFLASH_ERR_TIMEOUT);
          flags[0] = 1;
          break;
        }
        ptx::tc_fence_after();
        bool ok = true;
        for (int i = 0; i < n; ++i) {
          if (!ptx::mbar_wait_bounded(&full[stage], phase, kTimeoutNs, flags)) {
            record_status(p.status, DFLASH_ERR_TIMEOUT);
            flags[0] = 1;
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t a_desc = ptx::sw128_kmajor_desc(ptx::smem_addr(sA + stage * kABytes));
          const uint64_t b_desc = ptx::sw128_kmajor_desc(ptx::smem_addr(sB + stage * b_bytes));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            ptx::mma_bf16(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc,
                          (i > 0 || k > 0) ? 1u : 0u);
          ptx::mma_commit(&empty[stage]);
          issued_any = true;
          if (++stage == p.stages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        ptx::mma_commit(&accf[acc]);
        ++tile_i;
        u += n;
      }
      if (flags[0] && issued_any) {
        // drain: wait for the MMAs already issued before TMEM is released
        ptx::mma_commit(drain);
        ptx::mbar_wait_bounded(drain, 0u, kTimeoutNs, nullptr);
      }
    }
  } else {
    // ---------------- epilogue warps ----------------
    const int ew = warp & 3;            // TMEM lane quarter this warp may access
    const int f = ew * 32 + lane;       // tile column (weight row) of this thread
    const int etid = threadIdx.x - 64;  // 0..127
    int tile_i = 0;
    long long u = u_begin;
    while (u < u_end) {
      const int acc = tile_i & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(tile_i >> 1) & 1u;
      const int t = static_cast<int>(u / KB);
      const int kb0 = static_cast<int>(u - (long long)t * KB);
      const int n = static_cast<int>((KB - kb0) < (u_end - u) ? (KB - kb0) : (u_end - u));
      const int ftile = t / p.n_rtiles;
      const int rtile = t - ftile * p.n_rtiles;
      const int row0 = rtile * p.n_tile;
      const int nrows = min(p.n_tile, p.epi.M_rows - row0);
      const int c_first = cta_of_unit((long long)t * KB, U, G);
      const int c_last = cta_of_unit((long long)t * KB + KB - 1, U, G);
      const int nslots = c_last - c_first + 1;
      const bool single = nslots == 1;

      const bool ok = ptx::mbar_wait_bounded(&accf[acc], acc_phase, kTimeoutNs, flags);
      if (!ok) {
        record_status(p.status, DFLASH_ERR_TIMEOUT);
        flags[0] = 1;
      }
      if (ptx::named_bar_or(1, kEpiThreads, !ok)) break;
      ptx::tc_fence_after();

      if (single) {
        epi_row_scales(p.epi, row0, nrows, s_scale, etid, kEpiThreads);
        for (int i = etid; i < 4 * p.n_tile; i += kEpiThreads) s_red[i] = 0.f;
      }
      float* my_part = p.part + ((size_t)c_first * p.max_slots + (c - c_first)) *
                                    (size_t)p.n_tile * kTileN;
      for (int c0 = 0; c0 < nrows; c0 += kChunk) {
        float v[16];
        __syncwarp();
        ptx::tmem_ld_32x16(tmem_base + (static_cast<uint32_t>(ew * 32) << 16) +
                               static_cast<uint32_t>(acc * p.n_tile + c0), v);
        if (single) {
#pragma unroll
          for (int j = 0; j < 16; ++j) buf[j * kBufLd + f] = v[j];
          ptx::named_bar_sync(1, kEpiThreads);
          epi_apply_chunk<T>(p.epi, buf, ftile * kTileN, row0 + c0, min(kChunk, nrows - c0), f,
                             s_scale, row0, s_red, p.n_tile, ew);
          ptx::named_bar_sync(1, kEpiThreads);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) my_part[(size_t)(c0 + j) * kTileN + f] = v[j];
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&acce[acc]);

      if (single) {
        if (p.epi.kind == EPI_RESID) {
          ptx::named_bar_sync(1, kEpiThreads);
          epi_resid_flush(p.epi, ftile, row0, nrows, s_red, p.n_tile, 4, etid, kEpiThreads);
        }
      } else {
        __threadfence();
        ptx::named_bar_sync(1, kEpiThreads);
        if (etid == 0) {
          const int prev = atomicAdd(&p.counters[c_first], 1);
          flags[1] = (prev == nslots - 1) ? 1 : 0;
        }
        ptx::named_bar_sync(1, kEpiThreads);
        if (flags[1]) {
          __threadfence();
          epi_row_scales(p.epi, row0, nrows, s_scale, etid, kEpiThreads);
          for (int i = etid; i < 4 * p.n_tile; i += kEpiThreads) s_red[i] = 0.f;
          const float* slots = p.part + (size_t)c_first * p.max_slots * p.n_tile * kTileN;
          for (int c0 = 0; c0 < nrows; c0 += kChunk) {
            const int nr = min(kChunk, nrows - c0);
            // fixed slot order; four slots' loads (16 rows each) are in flight together
            float acc[kChunk];
#pragma unroll
            for (int j = 0; j < kChunk; ++j) acc[j] = 0.f;
            for (int s0 = 0; s0 < nslots; s0 += 4) {
              float v[4][kChunk];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float* src = slots + ((size_t)(s0 + q) * p.n_tile + c0) * kTileN + f;
#pragma unroll
                for (int j = 0; j < kChunk; ++j)
                  v[q][j] = (s0 + q < nslots && j < nr) ? __ldcg(src + (size_t)j * kTileN) : 0.f;
              }
#pragma unroll
              for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int j = 0; j < kChunk; ++j) acc[j] += v[q][j];
            }
#pragma unroll
            for (int j = 0; j < kChunk; ++j) buf[j * kBufLd + f] = acc[j];
            ptx::named_bar_sync(1, kEpiThreads);
            epi_apply_chunk<T>(p.epi, buf, ftile * kTileN, row0 + c0, nr, f, s_scale, row0, s_red,
                               p.n_tile, ew);
            ptx::named_bar_sync(1, kEpiThreads);
          }
          if (p.epi.kind == EPI_RESID)
            epi_resid_flush(p.epi, ftile, row0, nrows, s_red, p.n_tile, 4, etid, kEpiThreads);
          if (etid == 0) p.counters[c_first] = 0;
        }
        ptx::named_bar_sync(1, kEpiThreads);
      }
      ++tile_i;
      u += n;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    ptx::tmem_dealloc(tmem_base, tmem_cols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

template <typename T>
void set_smem_attr_once(int bytes) {
  static int done = 0;
  if (done < bytes) {
    cudaFuncSetAttribute(gemm_tc_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    done = bytes;
  }
}

}  // namespace

bool encode_kmajor_map(CUtensorMap* map, const void* base, int rows, int K,
                       long long row_stride_elems, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_stride_elems) * 2};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int tc_row_tile(int M_rows) {
  int n = 16;
  while (n < M_rows && n < 256) n <<= 1;
  return n;
}

TcPlan tc_plan(int M_rows, int N_feat, int K, int grid_max) {
  TcPlan pl{};
  pl.n_tile = tc_row_tile(M_rows);
  pl.n_rtiles = ceil_div(M_rows, pl.n_tile);
  pl.n_ftiles = ceil_div(N_feat, kTileN);
  pl.kblocks = K / 64;
  pl.total_units = (long long)pl.n_ftiles * pl.n_rtiles * pl.kblocks;
  pl.grid = static_cast<int>(pl.total_units < grid_max ? pl.total_units : grid_max);
  if (pl.grid < 1) pl.grid = 1;
  const int n_tiles = pl.n_ftiles * pl.n_rtiles;
  int ms = 1;
  for (int t = 0; t < n_tiles; ++t) {
    const int a = cta_of_unit((long long)t * pl.kblocks, pl.total_units, pl.grid);
    const int b = cta_of_unit((long long)t * pl.kblocks + pl.kblocks - 1, pl.total_units, pl.grid);
    if (b - a + 1 > ms) ms = b - a + 1;
  }
  pl.max_slots = ms;
  pl.part_bytes = (size_t)pl.grid * ms * pl.n_tile * kTileN * sizeof(float);
  const int b_bytes = pl.n_tile * 128;
  // Weight streaming is bound by the bytes in flight: under load a TMA request
  // takes ~4 us, so keeping HBM busy takes ~27 MB in flight across the GPU,
  // i.e. the deepest ring that fits in shared memory.
  int stages = 1;
  while (stages < 24 && smem_layout(stages + 1, pl.n_tile).total <= 227u * 1024u) ++stages;
  pl.stages = stages;
  pl.smem_bytes = smem_layout(stages, pl.n_tile).total;
  (void)b_bytes;
  return pl;
}

dflash_status launch_gemm_tc(const CUtensorMap& tmW, const CUtensorMap& tmX, const TcPlan& pl,
                             int M_rows, int N_feat, int K, float* part, int* counters,
                             int* status, const EpiParams& epi, cudaStream_t st) {
  TcParams p{};
  p.M_rows = M_rows;
  p.N_feat = N_feat;
  p.K = K;
  p.n_tile = pl.n_tile;
  p.n_rtiles = pl.n_rtiles;
  p.kblocks = pl.kblocks;
  p.total_units = pl.total_units;
  p.stages = pl.stages;
  p.part = part;
  p.max_slots = pl.max_slots;
  p.counters = counters;
  p.status = status;
  p.epi = epi;
  set_smem_attr_once<__nv_bfloat16>(pl.smem_bytes);
  TraceScope ts("gemm_tc", st);
  launch_k(gemm_tc_kernel<__nv_bfloat16>, dim3(pl.grid), dim3(kThreads), pl.smem_bytes, st, tmW,
           tmX, p);
  return check_launch("gemm_tc");
}

}  // namespace dfl
