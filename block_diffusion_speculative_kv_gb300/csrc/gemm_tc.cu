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
// is split over several CTAs is finished by the CTA holding its first K blocks
// (they end that CTA's range, so it is among the last to get there): the
// others post fp32 partial sums and a release-add on the tile's counter, and
// it adds them, in a fixed order, to its own accumulator.
//
// Chains.  One launch runs up to kMaxPhases dependent GEMMs ("phases", e.g.
// W_o -> W_gate|up -> W_down -> next layer's W_qkv), each GEMM's activations
// being an earlier phase's output.  Weights depend on nothing, so the weight
// stream runs through all phases without a break; only the activation tiles
// of phase k wait, on a grid-wide counter that every CTA bumps (release) once
// its epilogue work for phase k-1 is done.  The ring holds the weight tiles
// already fetched meanwhile, so the hand-over between phases costs no stream
// time as long as it is shorter than the ring's worth of streaming.
//
// Roles (7 warps): warp 0 lane 0 loads weight tiles into a multi-stage shared
// memory ring (evict-first in L2); warp 6 lane 0 loads the matching activation
// tiles (evict-last); both arrive on the stage's full barrier.  Warp 1 owns the
// TMEM allocation and its lane 0 issues tcgen05.mma (128 x n_tile x 16, four
// per 64-wide K block) and tcgen05.commit to release ring slots; warps 2-5
// drain TMEM (tcgen05.ld, 32 lanes each) and run the epilogue.  A CTA's tiles
// alternate between two TMEM accumulators, so the MMAs of the next tile never
// wait for the epilogue of the previous one.  Every wait (mbarrier or phase
// counter) is bounded in time; on expiry the CTA records DFLASH_ERR_TIMEOUT in
// the status word, drains its outstanding copies and MMAs (again bounded),
// frees TMEM and exits.
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "epilogue.cuh"
#include "gemm.h"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int kThreads = 224;
constexpr int kEpiThreads = 128;
constexpr int kABytes = kTileN * 128;  // 128 weight rows x 64 bf16
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct TcPhase {
  int N_feat, K, n_rtiles, kblocks;
  int grid;        // CTAs sharing the units: min(launch grid, total_units)
  long long total_units;
  int max_slots;
  int* counters;   // split-tile arrival counters of this phase [grid]
  EpiParams epi;
};

struct TcParams {
  int M_rows, n_tile, stages, n_phases;
  float* part;     // split-tile partial sums [grid][max_slots][n_tile][128]
  int* sync;       // [kMaxPhases] phase-done counters, then the exit counter
  int* status;
  TcPhase ph[kMaxPhases];
};

struct TcMaps {
  CUtensorMap w[kMaxPhases];
  CUtensorMap x[kMaxPhases];
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

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Release-add: everything this CTA wrote before the preceding barrier is
// visible to whoever acquires the new value.
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("fence.acq_rel.gpu;\n\tred.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v)
               : "memory");
}
// Wait until *p >= target (bounded; false on expiry or abort).
__device__ __forceinline__ bool wait_counter(const int* p, int target, const volatile int* abort) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (ld_acquire(p) >= target) return true;
    if (abort && *abort) return false;
    if (global_ns() - t0 > kTimeoutNs) return false;
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ TcMaps maps, const TcParams p) {
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
  // two accumulators of n_tile columns: the MMAs of a CTA's next tile run while
  // the epilogue drains the previous one
  const uint32_t tmem_cols = 2 * p.n_tile < 32 ? 32u : static_cast<uint32_t>(2 * p.n_tile);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      ptx::mbar_init(&full[s], 2);   // weight producer + activation producer
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
    for (int k = 0; k < p.n_phases; ++k) {
      ptx::prefetch_tmap(&maps.w[k]);
      ptx::prefetch_tmap(&maps.x[k]);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Weights are never written by a kernel: the weight stream starts before the
  // previous kernel completes; everything else waits for it.
  if (!(warp == 0 && lane == 0)) pdl_wait();
  pdl_trigger();

  if (warp == 0 || warp == 6) {
    // ---------------- TMA producers (weights: warp 0, activations: warp 6) ----------------
    if (lane == 0) {
      const bool wprod = warp == 0;
      const uint64_t pol = wprod ? ptx::policy_evict_first() : ptx::policy_evict_last();
      const uint32_t bytes = wprod ? static_cast<uint32_t>(kABytes) : b_bytes;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0;   // bit s: stage s has an issued copy
      uint32_t last_phase = 0;    // bit s: parity of that copy's phase
      for (int k = 0; k < p.n_phases && !flags[0]; ++k) {
        const TcPhase& P = p.ph[k];
        const long long U = P.total_units;
        const int Gk = P.grid;
        const long long u_begin = c < Gk ? (long long)c * U / Gk : 0;
        const long long u_end = c < Gk ? (long long)(c + 1) * U / Gk : 0;
        const int KB = P.kblocks;
        if (!wprod && k > 0) {
          if (!wait_counter(&p.sync[k - 1], G, flags)) {
            record_status(p.status, DFLASH_ERR_TIMEOUT);
            flags[0] = 1;
            break;
          }
          // the tiles about to be read by TMA (async proxy) were written with
          // ordinary stores by other CTAs
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        const CUtensorMap* map = wprod ? &maps.w[k] : &maps.x[k];
        uint8_t* dst0 = wprod ? sA : sB;
        const uint32_t stride = wprod ? static_cast<uint32_t>(kABytes) : b_bytes;
        for (long long u = u_begin; u < u_end; ++u) {
          const int t = static_cast<int>(u / KB);
          const int kb = static_cast<int>(u - (long long)t * KB);
          const int ftile = t / P.n_rtiles;
          const int rtile = t - ftile * P.n_rtiles;
          if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, kTimeoutNs, flags)) {
            record_status(p.status, DFLASH_ERR_TIMEOUT);
            flags[0] = 1;
            break;
          }
          ptx::mbar_arrive_expect_tx(&full[stage], bytes);
          ptx::tma_load_2d(dst0 + stage * stride, map, &full[stage], kb * 64,
                           wprod ? ftile * kTileN : rtile * p.n_tile, pol);
          issued_mask |= 1u << stage;
          last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == p.stages) { stage = 0; phase ^= 1u; }
        }
      }
      if (flags[0]) {
        // drain: every issued copy must land before the CTA may exit
        for (int s = 0; s < p.stages; ++s)
          if (issued_mask & (1u << s))
            ptx::mbar_wait_bounded(&full[s], (last_phase >> s) & 1u, kTimeoutNs, nullptr);
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
      for (int k = 0; k < p.n_phases && !flags[0]; ++k) {
        const TcPhase& P = p.ph[k];
        const long long U = P.total_units;
        const int Gk = P.grid;
        const long long u_end = c < Gk ? (long long)(c + 1) * U / Gk : 0;
        const int KB = P.kblocks;
        long long u = c < Gk ? (long long)c * U / Gk : 0;
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
            for (int kk = 0; kk < 4; ++kk)
              ptx::mma_bf16(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc,
                            (i > 0 || kk > 0) ? 1u : 0u);
            ptx::mma_commit(&empty[stage]);
            issued_any = true;
            if (++stage == p.stages) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          ptx::mma_commit(&accf[acc]);
          ++tile_i;
          u += n;
        }
      }
      if (flags[0] && issued_any) {
        // drain: wait for the MMAs already issued before TMEM is released
        ptx::mma_commit(drain);
        ptx::mbar_wait_bounded(drain, 0u, kTimeoutNs, nullptr);
      }
    }
  } else {
    // ---------------- epilogue warps (2-5) ----------------
    const int ew = warp & 3;            // TMEM lane quarter this warp may access
    const int f = ew * 32 + lane;       // tile column (weight row) of this thread
    const int etid = threadIdx.x - 64;  // 0..127
    int tile_i = 0;
    bool stop = false;
    for (int k = 0; k < p.n_phases && !stop; ++k) {
      const TcPhase& P = p.ph[k];
      const EpiParams& E = P.epi;
      const long long U = P.total_units;
      const int Gk = P.grid;
      const long long u_end = c < Gk ? (long long)(c + 1) * U / Gk : 0;
      const int KB = P.kblocks;
      long long u = c < Gk ? (long long)c * U / Gk : 0;
      if (k > 0) {
        // the epilogue reads what earlier phases wrote (row norms, residual)
        bool ok = true;
        if (etid == 0) ok = wait_counter(&p.sync[k - 1], G, flags);
        if (ptx::named_bar_or(1, kEpiThreads, !ok)) {
          record_status(p.status, DFLASH_ERR_TIMEOUT);
          flags[0] = 1;
          break;
        }
      }
      // With one row tile, the RMS row scales of the phase are computed once,
      // ahead of its first accumulator.
      const bool scales_once = P.n_rtiles == 1;
      if (scales_once) {
        epi_row_scales(E, 0, min(p.n_tile, E.M_rows), s_scale, etid, kEpiThreads);
        ptx::named_bar_sync(1, kEpiThreads);
      }
      while (u < u_end) {
        const int acc = tile_i & 1;
        const uint32_t acc_phase = static_cast<uint32_t>(tile_i >> 1) & 1u;
        const uint32_t tacc = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) +
                              static_cast<uint32_t>(acc * p.n_tile);
        const int t = static_cast<int>(u / KB);
        const int kb0 = static_cast<int>(u - (long long)t * KB);
        const int n = static_cast<int>((KB - kb0) < (u_end - u) ? (KB - kb0) : (u_end - u));
        const int ftile = t / P.n_rtiles;
        const int rtile = t - ftile * P.n_rtiles;
        const int row0 = rtile * p.n_tile;
        const int nrows = min(p.n_tile, E.M_rows - row0);
        const int c_first = cta_of_unit((long long)t * KB, U, Gk);
        const int c_last = cta_of_unit((long long)t * KB + KB - 1, U, Gk);
        const int nslots = c_last - c_first + 1;
        // A tile split over several CTAs is finished by c_first: the tile's
        // first K blocks close c_first's unit range, so it is among the last to
        // finish its share.  The others post partial sums (slot c - c_first)
        // and a release-add; c_first adds them, in slot order, to its own
        // accumulator read straight from TMEM.
        const bool single = nslots == 1;
        const bool reducer = !single && c == c_first;

        const bool ok = ptx::mbar_wait_bounded(&accf[acc], acc_phase, kTimeoutNs, flags);
        if (!ok) {
          record_status(p.status, DFLASH_ERR_TIMEOUT);
          flags[0] = 1;
        }
        if (ptx::named_bar_or(1, kEpiThreads, !ok)) {
          stop = true;
          break;
        }
        ptx::tc_fence_after();

        if (!single && !reducer) {
          float* my_part = p.part + ((size_t)c_first * P.max_slots + (c - c_first)) *
                                        (size_t)p.n_tile * kTileN;
          for (int c0 = 0; c0 < nrows; c0 += kChunk) {
            float v[16];
            __syncwarp();
            ptx::tmem_ld_32x16(tacc + static_cast<uint32_t>(c0), v);
#pragma unroll
            for (int j = 0; j < 16; ++j) my_part[(size_t)(c0 + j) * kTileN + f] = v[j];
          }
          ptx::tc_fence_before();
          ptx::mbar_arrive(&acce[acc]);
          ptx::named_bar_sync(1, kEpiThreads);
          if (etid == 0) red_release_add(&P.counters[c_first], 1);
        } else {
          if (!scales_once) epi_row_scales(E, row0, nrows, s_scale, etid, kEpiThreads);
          for (int i = etid; i < 4 * p.n_tile; i += kEpiThreads) s_red[i] = 0.f;
          if (reducer) {
            bool got = true;
            if (etid == 0) got = wait_counter(&P.counters[c_first], nslots - 1, flags);
            if (ptx::named_bar_or(1, kEpiThreads, !got)) {
              record_status(p.status, DFLASH_ERR_TIMEOUT);
              flags[0] = 1;
              stop = true;
              break;
            }
          }
          const float* slots = p.part + (size_t)c_first * P.max_slots * p.n_tile * kTileN;
          for (int c0 = 0; c0 < nrows; c0 += kChunk) {
            const int nr = min(kChunk, nrows - c0);
            float sum[kChunk];
            __syncwarp();
            ptx::tmem_ld_32x16(tacc + static_cast<uint32_t>(c0), sum);
            // slots 1.. in order; four slots' loads (16 rows each) in flight together
            for (int s0 = 1; s0 < nslots; s0 += 4) {
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
                for (int j = 0; j < kChunk; ++j) sum[j] += v[q][j];
            }
#pragma unroll
            for (int j = 0; j < kChunk; ++j) buf[j * kBufLd + f] = sum[j];
            ptx::named_bar_sync(1, kEpiThreads);
            epi_apply_chunk<T>(E, buf, ftile * kTileN, row0 + c0, nr, f, s_scale, row0, s_red,
                               p.n_tile, ew);
            ptx::named_bar_sync(1, kEpiThreads);
          }
          ptx::tc_fence_before();
          ptx::mbar_arrive(&acce[acc]);
          if (E.kind == EPI_RESID)
            epi_resid_flush(E, ftile, row0, nrows, s_red, p.n_tile, 4, etid, kEpiThreads);
          if (reducer && etid == 0) P.counters[c_first] = 0;   // for the next launch
          ptx::named_bar_sync(1, kEpiThreads);
        }
        ++tile_i;
        u += n;
      }
      if (stop) break;
      // this CTA's share of phase k is written: publish it
      ptx::named_bar_sync(1, kEpiThreads);
      if (etid == 0) red_release_add(&p.sync[k], 1);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    ptx::tmem_dealloc(tmem_base, tmem_cols);
  }
  // The last CTA out resets the phase counters for the next launch (every CTA
  // has passed all of its waits by now).
  if (threadIdx.x == 0) {
    __threadfence();
    const int prev = atomicAdd(&p.sync[kMaxPhases], 1);
    if (prev == G - 1) {
      for (int k = 0; k < kMaxPhases; ++k) p.sync[k] = 0;
      p.sync[kMaxPhases] = 0;
      __threadfence();
    }
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

TcPlan tc_plan(int M_rows, int N_feat, int K, int grid) {
  TcPlan pl{};
  pl.n_tile = tc_row_tile(M_rows);
  pl.n_rtiles = ceil_div(M_rows, pl.n_tile);
  pl.n_ftiles = ceil_div(N_feat, kTileN);
  pl.kblocks = K / 64;
  pl.total_units = (long long)pl.n_ftiles * pl.n_rtiles * pl.kblocks;
  pl.grid = static_cast<int>(pl.total_units < grid ? pl.total_units : grid);
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
  // the deepest ring that fits: it also carries the weight stream across the
  // hand-over between the phases of a chain
  int stages = 1;
  while (stages < 24 && smem_layout(stages + 1, pl.n_tile).total <= 227u * 1024u) ++stages;
  pl.stages = stages;
  pl.smem_bytes = smem_layout(stages, pl.n_tile).total;
  return pl;
}

dflash_status launch_gemm_chain(const GemmPhase* ph, int n_phases, int M_rows, float* part,
                                int* counters, int* status, cudaStream_t st) {
  if (n_phases < 1 || n_phases > kMaxPhases)
    return set_error(DFLASH_ERR_INVALID_ARG, "GEMM chain: 1..%d phases", kMaxPhases);
  const int G = num_sms();
  TcMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  TcParams p{};
  p.M_rows = M_rows;
  p.n_phases = n_phases;
  p.part = part;
  p.sync = counters + kMaxPhases * G;
  p.status = status;
  int smem = 0;
  for (int k = 0; k < n_phases; ++k) {
    const TcPlan pl = tc_plan(M_rows, ph[k].N, ph[k].K, G);
    p.n_tile = pl.n_tile;
    p.stages = pl.stages;
    smem = pl.smem_bytes;
    TcPhase& P = p.ph[k];
    P.N_feat = ph[k].N;
    P.K = ph[k].K;
    P.n_rtiles = pl.n_rtiles;
    P.kblocks = pl.kblocks;
    P.grid = pl.grid;
    P.total_units = pl.total_units;
    P.max_slots = pl.max_slots;
    P.counters = counters + k * G;
    P.epi = ph[k].epi;
    maps.w[k] = *ph[k].tmW;
    if (!encode_kmajor_map(&maps.x[k], ph[k].X, M_rows, ph[k].K, ph[k].ldx, pl.n_tile))
      return set_error(DFLASH_ERR_CUDA, "cannot encode the activation TMA descriptor");
  }
  set_smem_attr_once<__nv_bfloat16>(smem);
  TraceScope ts("gemm_tc", st);
  static_assert(sizeof(TcParams) + sizeof(TcMaps) <= 32000, "kernel parameter space");
  launch_k(gemm_tc_kernel<__nv_bfloat16>, dim3(G), dim3(kThreads), smem, st, maps, p);
  return check_launch("gemm_tc");
}

int gemm_counter_ints() { return kMaxPhases * num_sms() + kMaxPhases + 1; }

}  // namespace dfl
