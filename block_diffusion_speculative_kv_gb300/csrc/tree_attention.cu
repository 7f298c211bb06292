// Tree attention of the verification pass and the depth position ids.
//
// "Accelerating Speculative Decoding with Block Diffusion Draft Trees",
// section 3.4.5: the draft tree is flattened (node 0 is the root, the bonus
// token), every node gets the position id of its depth, and one forward pass
// of the target model scores all nodes under the ancestor-only mask: node i
// attends to the whole past context (the KV cache), to the root, to its
// ancestors and to itself, and to no other tree node.  This file is one
// target-layer attention of that pass, with grouped-query heads:
//
//   out[i, h] = softmax_j( q[i, h] . key_j / sqrt(hd) ) value_j
//   over key_j in { cache slot t < ctx_len } U { tree node j : mask[i] has bit j }
//
// and the rotation of the tree's queries and keys at position ctx_len + depth.
//
// Decomposition: query tiles of 32 nodes x the G <= 4 query heads of a KV head
// (row r = head (r / 32), node 32 qt + r % 32: the 128 rows of one tensor-core
// MMA), the context split into chunks of 128-key tiles so the grid is about
// one wave, and the tree's own keys as the last tiles of the last chunk.  Each
// CTA posts an unnormalised partial (O, max, sum) of its rows; the last CTA of
// a (query tile, KV head) to finish merges every chunk's partial, in chunk
// order, and writes the bf16 rows (an arrival counter, no waiting).  Nodes are
// numbered in pop order, so an ancestor has a smaller number than its
// descendant: the tree tiles of query tile qt hold keys 0 .. 32 qt + 31 only.
//
// Block mode (the drafter's attention of "DFlash: Block Diffusion for Flash
// Speculative Decoding", section 3.4.4, for batches): the L <= 32 block rows
// take the place of a query tile's nodes (rows L .. 31 of each head are dead),
// every block key is visible to every row (the anchor row only its own key
// when the anchor is isolated), each request's context ends at its own length,
// and the block keys ride in the chunk holding that end; later chunks exit.
//
// Per CTA, on the 5th-generation tensor cores (accumulators in TMEM):
//   S_t  = Q K_t^T      A = Q (K-major), B = K tile (K-major), S in TMEM
//   O   += P_t V_t      A = P (K-major, written by the softmax warps),
//                       B = V tile read MN-major (head dims contiguous), O in TMEM
// Warp 8 lane 0 loads (TMA; context tiles before the grid dependency wait),
// warp 9 lane 0 issues the MMAs, S_{t+1} before P_t V_t so that the softmax of
// tile t+1 overlaps the second product of tile t (two S buffers).  Warps 0-7
// are the softmax: warp w owns TMEM lane quarter w % 4 (rows 32 (w % 4) ..)
// and key half w / 4 of every tile; the two warps of a quarter trade their
// row maxima through shared memory.  O is rescaled lazily, only when a row's
// maximum rises by more than 8 (base-2 units) over the reference used so far,
// so every exponential stays below 2^8; O, the sum and the reported max share
// that reference.  Every wait is bounded (2 s); on expiry the CTA records
// DFLASH_ERR_TIMEOUT in the status word, waits for its copies and MMAs in
// flight, frees TMEM and returns.
#include <cmath>

#include "attention.h"
#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "ptx.cuh"

#include <math_constants.h>

namespace dfl {

namespace {

constexpr int kHd = 128;
constexpr int kTk = 128;                       // keys per tile
constexpr int kNodesPerTile = 32;              // x G <= 4 heads = the MMA's 128 rows
constexpr int kHalf = 128 * 128;               // one 64-column half of a 128-row bf16 tile
constexpr int kTileB = 2 * kHalf;              // 32 KB: 128 rows x 128 bf16
constexpr int kThreads = 320;                  // 8 softmax warps, loader, MMA issuer
constexpr int kBarOff = kTileB + 2 * 2 * kTileB + kTileB;   // Q, 2 x (K, V), P
constexpr int kSmem = 1024 + kBarOff + 4096;
constexpr float kLazy = 8.f;
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct TreeTcMaps {
  CUtensorMap kc, vc;   // cache [n_req*n_kv*cap][hd], box 64 x 128
  CUtensorMap kt, vt;   // the nodes' keys and values [n_req*B1][kv_ld], box 64 x 128
  CUtensorMap q;        // the nodes' queries [n_req*B1][q_ld], box 64 x 32
};

struct TreeTcParams {
  AttnParams a;                 // head counts, chunking, partials (with n_qt)
  const uint32_t* mask;         // [n_req][B+1][mask_w]
  int mask_w;
  const int32_t* n_nodes;       // [n_req]: nodes 0 .. n_nodes[r] are live
  int B1;                       // B + 1
  int n_ctx_tiles;              // context tiles per chunk (the chunk is n_ctx_tiles * 128 keys)
  int* status;
  int* arrivals;                // [n_req * n_qt][n_kv]: chunks done, zero between calls
  // Block attention of the drafter ("DFlash" page, 3.4.4) instead of a tree:
  // the B1 = L block rows of a request see every block key (the anchor row only
  // itself when anchor_iso), the context ends at the request's ctx_len, the
  // block keys ride in the chunk that holds that end and later chunks have no
  // work.  Partials are indexed (head, block row), G L rows per chunk.
  int block;
  int anchor_iso;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait of the loader and the MMA issuer, which share warp schedulers
// with softmax warps: they back off between polls.
__device__ __forceinline__ bool wait_backoff(uint64_t* bar, uint32_t parity,
                                             const volatile int* abort) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    __nanosleep(64);
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (abort && *abort) return false;
    if (global_ns() - t0 > kTimeoutNs) return false;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
tree_attn_tc_kernel(const __grid_constant__ TreeTcMaps maps, const TreeTcParams tp) {
  const AttnParams& p = tp.a;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                // [2 halves][128 rows][64] bf16
  uint8_t* sKV = sQ + kTileB;        // slot s: K at sKV + 2s*kTileB, V after it (separate rings)
  uint8_t* sP = sKV + 4 * kTileB;    // [2 key halves][128 rows][64 keys]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* k_full = bar;            // [2] K tile landed
  uint64_t* k_empty = bar + 2;       // [2] S of the tile done: the K slot is free
  uint64_t* v_full = bar + 4;        // [2] V tile landed
  uint64_t* v_empty = bar + 6;       // [2] P V of the tile done: the V slot is free
  uint64_t* q_full = bar + 8;
  uint64_t* s_ready = bar + 9;       // [2]
  uint64_t* s_free = bar + 11;       // [2]
  uint64_t* p_ready = bar + 13;
  uint64_t* pv_done = bar + 14;
  uint64_t* drain = bar + 15;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 16);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);
  float* xchg = reinterpret_cast<float*>(bar + 20);   // [2 tiles][8 warps][32] maxima, then sums

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk_id = blockIdx.x, g = blockIdx.y;
  const int rq = blockIdx.z, req = rq / p.n_qt, qt = rq % p.n_qt;
  const int QR = p.G * kNodesPerTile;
  const int node0 = qt * kNodesPerTile;
  const int k_begin = chunk_id * p.chunk;
  // Tree: context tiles fixed by the host's max_ctx (per-request lengths are
  // masked), the tree keys in the last chunk.  Block: the request's own
  // context tiles of the chunk, the block keys in chunk cb (read before the
  // grid dependency wait: the lengths are set kernels back, like the cache).
  int nct = tp.n_ctx_tiles, cb = p.n_chunks - 1, bctx = 0;
  if (tp.block) {
    bctx = min(max(p.ctx_len[req], 0), p.cap);
    cb = min(bctx > 0 ? (bctx - 1) / p.chunk : 0, p.n_chunks - 1);
    if (chunk_id > cb) return;   // no keys here, and no partial to post
    nct = min(max((bctx - k_begin + kTk - 1) / kTk, 0), tp.n_ctx_tiles);
  }
  const bool last_chunk = chunk_id == cb;
  const int n_parts = cb + 1;                        // chunks that post a partial
  const int rph = tp.block ? tp.B1 : kNodesPerTile;  // partial rows per head
  const int QRp = p.G * rph;
  const size_t part_row0 = (((size_t)rq * p.n_kv + g) * p.n_chunks + chunk_id) * QRp;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&k_full[s], 1);
      ptx::mbar_init(&k_empty[s], 1);
      ptx::mbar_init(&v_full[s], 1);
      ptx::mbar_init(&v_empty[s], 1);
      ptx::mbar_init(&s_ready[s], 1);
      ptx::mbar_init(&s_free[s], 8);
    }
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(p_ready, 8);
    ptx::mbar_init(pv_done, 1);
    ptx::mbar_init(drain, 1);
    *abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(tslot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = *tslot;
  // TMEM columns: S buffers at 0 and kTk, O at 2 kTk
  const uint32_t tO = tbase + 2 * kTk;

  // request-dependent sizes (read after the dependency wait by everyone)
  int last = -1, tree_end = 0, ntt = 0, ctx = 0;
  auto sizes = [&]() {
    last = tp.block ? tp.B1 - 1 : min(max(tp.n_nodes[req], 0), tp.B1 - 1);
    ctx = tp.block ? bctx : min(max(p.ctx_len[req], 0), p.cap);
    tree_end = (last_chunk && node0 <= last) ? min(node0 + kNodesPerTile - 1, last) + 1 : 0;
    ntt = (tree_end + kTk - 1) / kTk;
  };

  if (warp == 8) {
    // ---------------- loads: lane 0 the K tiles (and Q), lane 1 the V tiles ----------------
    if (lane < 2) {
      const bool kl = lane == 0;
      if (kl) {
        ptx::prefetch_tmap(&maps.kc);
        ptx::prefetch_tmap(&maps.kt);
        ptx::prefetch_tmap(&maps.q);
      } else {
        ptx::prefetch_tmap(&maps.vc);
        ptx::prefetch_tmap(&maps.vt);
      }
      // a tree's query tiles of a KV head share its tiles; a block reads them once
      const uint64_t pol = tp.block ? ptx::policy_evict_first() : ptx::policy_evict_last();
      const int slab = (req * p.n_kv + g) * p.cap;
      uint64_t* full = kl ? k_full : v_full;
      uint64_t* empty = kl ? k_empty : v_empty;
      const CUtensorMap* mc = kl ? &maps.kc : &maps.vc;
      const CUtensorMap* mt = kl ? &maps.kt : &maps.vt;
      uint32_t issued = 0, last_par = 0;
      auto load = [&](int t) {
        const int s = t & 1;
        const uint32_t par = static_cast<uint32_t>(t >> 1) & 1u;
        if (!wait_backoff(&empty[s], par ^ 1u, abort)) {
          if (!*abort) record_status(tp.status, DFLASH_ERR_TIMEOUT);
          *abort = 1;
          return false;
        }
        uint8_t* dst = sKV + (2 * s + (kl ? 0 : 1)) * kTileB;
        ptx::mbar_arrive_expect_tx(&full[s], kTileB);
        if (t < nct) {
          const int y = slab + k_begin + t * kTk;
          for (int h = 0; h < 2; ++h) ptx::tma_load_2d(dst + h * kHalf, mc, &full[s], 64 * h, y, pol);
        } else {
          const int y = req * tp.B1 + (t - nct) * kTk;
          for (int h = 0; h < 2; ++h)
            ptx::tma_load_2d(dst + h * kHalf, mt, &full[s], g * kHd + 64 * h, y, pol);
        }
        issued |= 1u << s;
        last_par = (last_par & ~(1u << s)) | (par << s);
        return true;
      };
      // the cache is written kernels back: its first tiles go out before the wait
      int t = 0;
      for (; t < 2 && t < nct; ++t)
        if (!load(t)) break;
      pdl_wait();
      pdl_trigger();
      sizes();
      const int ntiles = nct + ntt;
      if (!*abort && node0 <= last && ntiles > 0) {
        if (kl) {
          ptx::mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(p.G) * 2u * 32u * 128u);
          for (int hh = 0; hh < p.G; ++hh)
            for (int h = 0; h < 2; ++h)
              ptx::tma_load_2d(sQ + h * kHalf + hh * kNodesPerTile * 128, &maps.q, q_full,
                               (g * p.G + hh) * kHd + 64 * h, req * tp.B1 + node0, pol);
        }
        for (; t < ntiles && !*abort; ++t)
          if (!load(t)) break;
      }
      // every issued copy must land before the CTA exits (tiles requested
      // before the wait are issued even when this CTA turns out to have none)
      for (int s = 0; s < 2; ++s)
        if (issued & (1u << s))
          ptx::mbar_wait_bounded(&full[s], (last_par >> s) & 1u, kTimeoutNs, nullptr);
    } else {
      pdl_wait();
      pdl_trigger();
    }
  } else if (warp == 9) {
    // ---------------- MMA issue ----------------
    pdl_wait();
    pdl_trigger();
    sizes();
    const int ntiles = nct + ntt;
    if (lane == 0 && node0 <= last && ntiles > 0) {
      const uint32_t aQ = ptx::smem_addr(sQ), aP = ptx::smem_addr(sP);
      bool ok = wait_backoff(q_full, 0u, abort);
      const uint32_t idesc_s = ptx::idesc_bf16_f32(128, kTk);
      // O += P V: B = V tile read MN-major (the instruction's transpose bit for B)
      const uint32_t idesc_pv = ptx::idesc_bf16_f32(128, kHd) | (1u << 16);
      auto issue_s = [&](int t) {
        const int s = t & 1;
        const uint32_t par = static_cast<uint32_t>(t >> 1) & 1u;
        if (!wait_backoff(&k_full[s], par, abort)) return false;
        if (!wait_backoff(&s_free[s], par ^ 1u, abort)) return false;
        ptx::tc_fence_after();
        const uint32_t aK = ptx::smem_addr(sKV + 2 * s * kTileB);
#pragma unroll
        for (int kk = 0; kk < kHd / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          ptx::mma_bf16(tbase + s * kTk, ptx::sw128_kmajor_desc(aQ + off), ptx::sw128_kmajor_desc(aK + off),
                        idesc_s, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(&s_ready[s]);
        ptx::mma_commit(&k_empty[s]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int t = 0; t < ntiles && ok; ++t) {
        if (t + 1 < ntiles && !issue_s(t + 1)) { ok = false; break; }
        if (!ptx::mbar_wait_bounded(p_ready, static_cast<uint32_t>(t) & 1u, kTimeoutNs, abort)) {
          ok = false;
          break;
        }
        const int s = t & 1;
        if (!wait_backoff(&v_full[s], static_cast<uint32_t>(t >> 1) & 1u, abort)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t aV = ptx::smem_addr(sKV + (2 * s + 1) * kTileB);
#pragma unroll
        for (int j = 0; j < kTk / 16; ++j)
          ptx::mma_bf16(tO, ptx::sw128_kmajor_desc(aP + (j >> 2) * kHalf + (j & 3) * 32),
                        ptx::sw128_mnmajor_desc(aV + j * 2048, kHalf, 1024), idesc_pv,
                        (t > 0 || j > 0) ? 1u : 0u);
        ptx::mma_commit(pv_done);
        ptx::mma_commit(&v_empty[s]);
      }
      if (!ok) {
        if (!*abort) record_status(tp.status, DFLASH_ERR_TIMEOUT);
        *abort = 1;
      }
      // the MMAs already issued finish before TMEM is released
      ptx::mma_commit(drain);
      ptx::mbar_wait_bounded(drain, 0u, kTimeoutNs, nullptr);
    }
  } else {
    // ---------------- softmax (warps 0-7) ----------------
    pdl_wait();
    pdl_trigger();
    sizes();
    const int ntiles = nct + ntt;
    const int q = warp & 3;                      // TMEM lane quarter
    const int kh = warp >> 2;                    // key half of every tile
    const int r = q * 32 + lane;                 // query row
    const int node = node0 + (r & (kNodesPerTile - 1));
    const bool live = r < QR && node <= last;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int pair_bar = 1 + q;                  // warps q and q + 4
    const float sc = p.scale_log2;
    const uint32_t* mrow =
        tp.block ? nullptr : tp.mask + ((size_t)req * tp.B1 + (live ? node : 0)) * tp.mask_w;
    const bool iso = tp.block && tp.anchor_iso && node == 0;   // the anchor sees block key 0 only
    float m_ref = -CUDART_INF_F, l = 0.f;
    bool ok = node0 <= last && ntiles > 0;
    for (int t = 0; t < ntiles && ok; ++t) {
      const int s = t & 1;
      const bool tree = t >= nct;
      const int key0 = tree ? (t - nct) * kTk : k_begin + t * kTk;
      const int kend = tree ? tree_end : min(ctx, k_begin + nct * kTk);
      const int nk = min(kTk, kend - key0);      // valid keys of this tile (may be <= 0)
      bool got = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(
                                             &s_ready[s], static_cast<uint32_t>(t >> 1) & 1u,
                                             kTimeoutNs, abort));
      if (got) ptx::tc_fence_after();
      const uint32_t sa = tbase + s * kTk + lane_off + 64 * kh;   // this thread's 64 scores
      // ancestor bits of keys 64 kh .. 64 kh + 63 (context tiles: all keys)
      uint32_t mb[2] = {0xFFFFFFFFu, 0xFFFFFFFFu};
      if (tree && tp.block) {
        mb[0] = iso ? (kh == 0 ? 1u : 0u) : 0xFFFFFFFFu;
        mb[1] = iso ? 0u : 0xFFFFFFFFu;
      } else if (tree) {
        const int w0 = (key0 + 64 * kh) >> 5;
        mb[0] = live && w0 < tp.mask_w ? mrow[w0] : 0u;
        mb[1] = live && w0 + 1 < tp.mask_w ? mrow[w0 + 1] : 0u;
      }
      // this thread's 64 scores, read twice from TMEM (once for the row maximum,
      // once for P; both loads of a pass under one wait), -inf where masked.  A
      // context tile whose 128 keys are all valid needs no mask (warp-uniform);
      // a dead row's values are never reported.
      const bool plain = !tree && nk >= kTk;
      auto scores = [&](uint32_t (&u0)[32], uint32_t (&u1)[32]) {
        ptx::tmem_ld_32x32(sa, u0);
        ptx::tmem_ld_32x32(sa + 32, u1);
        ptx::tmem_wait_ld();
        if (!plain) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (!(live && 64 * kh + j < nk && ((mb[0] >> j) & 1u))) u0[j] = 0xff800000u;
            if (!(live && 64 * kh + 32 + j < nk && ((mb[1] >> j) & 1u))) u1[j] = 0xff800000u;
          }
        }
      };
      // Optimistic pass: P against the row's current reference m_ref.  Lazy
      // rescaling tolerates scores up to kLazy above it, so the tile's exact
      // maximum is needed only when one breaks that bound (a pair-wide vote);
      // then the pair trades maxima, raises the reference and recomputes P.
      uint32_t pk[32];
      float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      auto make_p = [&](const uint32_t (&u0)[32], const uint32_t (&u1)[32], float base) {
        const float2 sc2 = make_float2(sc, sc), nb2 = make_float2(-base, -base);
        rs2[0] = make_float2(0.f, 0.f);
        rs2[1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const uint32_t a = e < 16 ? u0[(2 * e) & 31] : u1[(2 * e) & 31];
          const uint32_t b = e < 16 ? u0[(2 * e + 1) & 31] : u1[(2 * e + 1) & 31];
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(a), __uint_as_float(b)), sc2, nb2);
          const float2 pe = make_float2(ex2(x.x), ex2(x.y));
          rs2[e & 1] = __fadd2_rn(rs2[e & 1], pe);
          __nv_bfloat162 h2 = __floats2bfloat162_rn(pe.x, pe.y);
          pk[e] = *reinterpret_cast<uint32_t*>(&h2);
        }
      };
      float lm = -CUDART_INF_F;   // this thread's maximum raw score over its 64 keys
      if (got) {
        uint32_t u0[32], u1[32];
        scores(u0, u1);
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(__uint_as_float(u0[i]), __uint_as_float(u1[i]));
#pragma unroll
        for (int j = 8; j < 32; ++j)
          mx8[j & 7] = fmaxf(mx8[j & 7], fmaxf(__uint_as_float(u0[j]), __uint_as_float(u1[j])));
        lm = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        make_p(u0, u1, m_ref == -CUDART_INF_F ? 0.f : m_ref);
      }
      const bool need = lm > -CUDART_INF_F &&
                        (m_ref == -CUDART_INF_F || lm * sc > m_ref + kLazy);
      bool raise = false;
      float f = 1.f;
      if (ptx::named_bar_or(pair_bar, 64, need || !got)) {
        float* xs = xchg + (t & 1) * 256;
        xs[warp * 32 + lane] = lm;
        if (ptx::named_bar_or(pair_bar, 64, !got)) { ok = false; break; }
        const float mx = fmaxf(lm, xs[(warp ^ 4) * 32 + lane]) * sc;
        const float m_new = fmaxf(m_ref, mx);
        raise = m_new > m_ref + kLazy || (m_ref == -CUDART_INF_F && m_new > m_ref);
        f = (raise && m_ref != -CUDART_INF_F) ? ex2(m_ref - m_new) : (raise ? 0.f : 1.f);
        l *= f;
        if (raise) m_ref = m_new;
        if (__any_sync(0xffffffffu, raise)) {
          uint32_t u0[32], u1[32];
          scores(u0, u1);
          make_p(u0, u1, m_ref == -CUDART_INF_F ? 0.f : m_ref);
        }
      }
      l += (rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y);
      // S_t is read: its TMEM buffer may take S_{t+2}
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&s_free[s]);
      // P_{t-1} V_{t-1} must be done: P is rewritten below and O may be rescaled
      if (t > 0) {
        got = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(
                                          pv_done, static_cast<uint32_t>(t - 1) & 1u, kTimeoutNs,
                                          abort));
        if (!got) { ok = false; }
        else ptx::tc_fence_after();
      }
      if (ptx::named_bar_or(pair_bar, 64, !ok)) { ok = false; break; }
      if (t > 0 && __any_sync(0xffffffffu, raise)) {
        // this warp's 64 columns of its rows of O
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          ptx::tmem_ld_32x32(tO + lane_off + 64 * kh + 32 * c, o);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
          ptx::tmem_st_32x32(tO + lane_off + 64 * kh + 32 * c, o);
        }
        ptx::tmem_wait_st();
      }
      // this thread's half row of P: 16-byte chunks of 8 keys, 128-byte swizzle
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4*>(sP + kh * kHalf + r * 128 + ((ch ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      // V rows past the tile's valid keys (stale, or another request's) are
      // zeroed: their P is 0, but 0 * NaN would not be
      const int nkz = max(nk, 0);
      if (nkz < kTk && ptx::mbar_wait_bounded(&v_full[s], static_cast<uint32_t>(t >> 1) & 1u,
                                               kTimeoutNs, abort)) {
        // (the V tile has its own ring: the zeros must land after its copy)
        uint8_t* dV = sKV + (2 * s + 1) * kTileB;
        const int nz = (kTk - nkz) * 2 * 8;        // 16-byte chunks
        for (int i = tid; i < nz; i += 256) {
          const int row = nkz + i / 16, h = (i >> 3) & 1, ch = i & 7;
          *reinterpret_cast<uint4*>(dV + h * kHalf + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(p_ready);
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(
                                       pv_done, static_cast<uint32_t>(ntiles - 1) & 1u,
                                       kTimeoutNs, abort));
      if (ok) ptx::tc_fence_after();
    }
    // one decision for all eight softmax warps (the merge below synchronises
    // them on barrier 5), then the row sum over both key halves
    const bool bad = ptx::named_bar_or(5, 256, !ok && node0 <= last && ntiles > 0);
    float* xl = xchg + 512;
    xl[warp * 32 + lane] = l;
    ptx::named_bar_sync(pair_bar, 64);
    l += xl[(warp ^ 4) * 32 + lane];

    // ---- the output rows of this query tile ----
    // Thread (quarter q, half kh) owns row r, head dims 64 kh .. 64 kh + 63.
    // With several chunks per (query tile, KV head), every CTA posts its
    // unnormalised partial and the last to arrive merges the others' into its
    // own and writes the bf16 rows (no CTA waits for another).
    const bool has_row = r < QR && node < tp.B1;    // a row of the output exists
    __nv_bfloat16* orow =
        p.out + ((size_t)req * tp.B1 + (has_row ? node : 0)) * p.out_ld +
        (size_t)(g * p.G + (r >> 5)) * kHd + 64 * kh;
    auto write_row = [&](const float (&o)[64], float inv) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t w4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __nv_bfloat162 h2 = __floats2bfloat162_rn(o[8 * i + 2 * e] * inv, o[8 * i + 2 * e + 1] * inv);
          w4[e] = *reinterpret_cast<uint32_t*>(&h2);
        }
        *reinterpret_cast<uint4*>(orow + 8 * i) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    };
    volatile int* s_last = reinterpret_cast<volatile int*>(xchg + 800);
    if (node0 > last || ntiles == 0) {
      // every node of this query tile is past the last one: zero rows (chunk 0)
      if (chunk_id == 0 && has_row) {
#pragma unroll
        for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4*>(orow + 8 * i) = make_uint4(0, 0, 0, 0);
      }
    } else if (!bad) {
      float o[64];
      {
        uint32_t ou[2][32];
        ptx::tmem_ld_32x32(tO + lane_off + 64 * kh, ou[0]);
        ptx::tmem_ld_32x32(tO + lane_off + 64 * kh + 32, ou[1]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 64; ++j) o[j] = __uint_as_float(ou[j >> 5][j & 31]);
      }
      const float m_own = live ? m_ref : -CUDART_INF_F;
      const float l_own = live ? l : 0.f;
      bool writer = true;
      const int pr = (r >> 5) * rph + (r & 31);   // partial row (= r for a tree)
      if (n_parts > 1) {
        if (r < QR && (r & 31) < rph) {
          float4* dst = reinterpret_cast<float4*>(p.part_o + (part_row0 + pr) * kHd + 64 * kh);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          if (kh == 0) {
            p.part_ml[(part_row0 + pr) * 2 + 0] = m_own;
            p.part_ml[(part_row0 + pr) * 2 + 1] = l_own;
          }
        }
        __threadfence();
        ptx::named_bar_sync(5, 256);
        int* arrive = tp.arrivals + (size_t)rq * p.n_kv + g;
        if (tid == 0) *s_last = atomicAdd(arrive, 1) == n_parts - 1;
        ptx::named_bar_sync(5, 256);
        writer = *s_last != 0;
        if (writer) {
          __threadfence();
          if (tid == 0) *arrive = 0;   // for the next call
        }
      }
      if (writer && has_row && n_parts == 1) {
        write_row(o, live && l_own > 0.f ? 1.f / l_own : 0.f);
      } else if (writer && has_row) {
        // merge every chunk's partial of this row in chunk order, the writer's
        // own re-read (reference M): the sums do not depend on which CTA
        // finished last
        const size_t row_base = ((size_t)rq * p.n_kv + g) * p.n_chunks * QRp + pr;
        float M = -CUDART_INF_F;
        for (int c = 0; c < n_parts; ++c) {
          const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + row_base + (size_t)c * QRp);
          if (ml.y > 0.f) M = fmaxf(M, ml.x);
        }
        float L = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) o[j] = 0.f;
        for (int c = 0; c < n_parts; ++c) {
          const size_t rc = row_base + (size_t)c * QRp;
          const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + rc);
          if (!(ml.y > 0.f)) continue;
          const float w = ex2(ml.x - M);
          L += w * ml.y;
          const float4* src = reinterpret_cast<const float4*>(p.part_o + rc * kHd + 64 * kh);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 v4 = __ldcg(src + i);
            o[4 * i] += w * v4.x;
            o[4 * i + 1] += w * v4.y;
            o[4 * i + 2] += w * v4.z;
            o[4 * i + 3] += w * v4.w;
          }
        }
        // a row that saw no key (a node past the last one) is written as zeros
        write_row(o, live && L > 0.f ? 1.f / L : 0.f);
      }
    } else {
      if (!*abort) record_status(tp.status, DFLASH_ERR_TIMEOUT);
      *abort = 1;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 9) {
    __syncwarp();
    ptx::tmem_dealloc(tbase, 512);
  }
}

// Rotation of one (node, head) row at position ctx_len + depth; a warp per row,
// lanes over the first half of the head dimension.
template <typename T>
__global__ void tree_rope_kernel(int n_req, int B1, int n_heads, int head_dim, const RopeFreqs fr,
                                 const int32_t* __restrict__ ctx_len,
                                 const int32_t* __restrict__ depth, T* __restrict__ x,
                                 long long ld) {
  const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  if (w >= (long long)n_req * B1 * n_heads) return;
  const int h = static_cast<int>(w % n_heads);
  const long long node = w / n_heads;            // req * B1 + i
  const int req = static_cast<int>(node / B1);
  const int dep = depth[node];
  if (dep < 0) return;                            // past the last node
  const int pos = ctx_len[req] + dep;
  const int half = head_dim / 2;
  T* row = x + node * ld + (long long)h * head_dim;
  for (int i = lane; i < half; i += 32) {
    const float2 cs = rope_cs(pos, i, fr);
    const float a = to_f32<T>(row[i]), b = to_f32<T>(row[i + half]);
    row[i] = from_f32<T>(a * cs.x - b * cs.y);
    row[i + half] = from_f32<T>(b * cs.x + a * cs.y);
  }
}

// Context tiles per chunk: the (request, query tile, KV head) triples times
// the chunks fill about one wave of one CTA per SM.
struct TreePlan {
  int n_qt, n_chunks, tiles_per_chunk;
};
TreePlan tree_plan(int n_req, int n_kv, int B, int max_ctx) {
  TreePlan pl;
  pl.n_qt = (B + 1 + kNodesPerTile - 1) / kNodesPerTile;
  const long long triples = (long long)n_req * pl.n_qt * n_kv;
  long long want = num_sms() / (triples > 0 ? triples : 1);
  if (want < 1) want = 1;
  const int ctx_tiles = (max_ctx + kTk - 1) / kTk;
  pl.tiles_per_chunk = ctx_tiles > 0 ? static_cast<int>((ctx_tiles + want - 1) / want) : 0;
  pl.n_chunks = pl.tiles_per_chunk > 0 ? (ctx_tiles + pl.tiles_per_chunk - 1) / pl.tiles_per_chunk
                                       : 1;
  return pl;
}

void set_tc_smem_attr() {
  static bool set = false;
  if (!set) {
    cudaFuncSetAttribute(tree_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    set = true;
  }
}

}  // namespace

dflash_status launch_block_attention_tc(const AttnParams& p, int* arrivals, int* status,
                                        cudaStream_t st) {
  if (p.G < 1 || p.G > 4 || p.L < 1 || p.L > kNodesPerTile || p.chunk < kTk || p.chunk % kTk ||
      p.n_chunks < 1)
    return set_error(DFLASH_ERR_UNSUPPORTED,
                     "block attention: needs G <= 4, L <= 32 and chunks of 128-key tiles");
  const long long kv_rows = (long long)p.n_req * p.n_kv * p.cap;
  const long long blk_rows = (long long)p.n_req * p.L;
  if (kv_rows >= (1ll << 31) || blk_rows >= (1ll << 31))
    return set_error(DFLASH_ERR_UNSUPPORTED, "block attention: cache or block rows exceed 2^31");
  if (p.qkv_ld % 8 || (reinterpret_cast<uintptr_t>(p.qkv) & 15) ||
      ((reinterpret_cast<uintptr_t>(p.cache_k) | reinterpret_cast<uintptr_t>(p.cache_v)) & 15))
    return set_error(DFLASH_ERR_UNSUPPORTED,
                     "block attention: the QKV row stride must be a multiple of 8 and the QKV "
                     "and cache buffers 16-byte aligned");
  TreeTcParams tp{};
  tp.a = p;
  tp.a.n_qt = 1;
  tp.B1 = p.L;
  tp.mask_w = 1;
  tp.n_ctx_tiles = p.chunk / kTk;
  tp.status = status;
  tp.arrivals = arrivals;
  tp.block = 1;
  tp.anchor_iso = p.anchor_sees_block ? 0 : 1;
  TreeTcMaps maps;
  const __nv_bfloat16* k = p.qkv + (size_t)p.n_q * kHd;
  const __nv_bfloat16* v = p.qkv + (size_t)(p.n_q + p.n_kv) * kHd;
  if (!encode_kmajor_map(&maps.kc, p.cache_k, static_cast<int>(kv_rows), kHd, kHd, kTk) ||
      !encode_kmajor_map(&maps.vc, p.cache_v, static_cast<int>(kv_rows), kHd, kHd, kTk) ||
      !encode_kmajor_map(&maps.kt, k, static_cast<int>(blk_rows), p.n_kv * kHd, p.qkv_ld, kTk) ||
      !encode_kmajor_map(&maps.vt, v, static_cast<int>(blk_rows), p.n_kv * kHd, p.qkv_ld, kTk) ||
      !encode_kmajor_map(&maps.q, p.qkv, static_cast<int>(blk_rows), p.n_q * kHd, p.qkv_ld,
                         kNodesPerTile))
    return set_error(DFLASH_ERR_CUDA, "block attention: cannot encode the TMA descriptors");
  set_tc_smem_attr();
  {
    TraceScope ts("attn_block_tc", st);
    launch_k(tree_attn_tc_kernel, dim3(p.n_chunks, p.n_kv, p.n_req), dim3(kThreads), kSmem, st,
             maps, tp);
  }
  return check_launch("block attention");
}

}  // namespace dfl

using namespace dfl;

extern "C" {

size_t dflash_tree_attention_workspace_bytes(int n_req, int n_q, int n_kv, int head_dim, int B,
                                             int max_ctx) {
  if (n_req < 1 || n_kv < 1 || n_q < n_kv || n_q % n_kv || B < 0 || max_ctx < 0 || head_dim != 128)
    return 0;
  const int G = n_q / n_kv;
  const TreePlan pl = tree_plan(n_req, n_kv, B, max_ctx);
  const size_t rows = (size_t)n_req * pl.n_qt * n_kv * pl.n_chunks * G * kNodesPerTile;
  const size_t arrivals = (size_t)n_req * pl.n_qt * n_kv * sizeof(int);
  return 256 + align_up(arrivals, 256) + align_up(rows * head_dim * sizeof(float), 256) +
         align_up(rows * 2 * sizeof(float), 256);
}

dflash_status dflash_tree_attention(int n_req, int n_q, int n_kv, int head_dim, int B,
                                    const int32_t* ctx_len, int max_ctx, int cap,
                                    const void* cache_k, const void* cache_v, const void* q,
                                    long long q_ld, const void* k, const void* v, long long kv_ld,
                                    const uint32_t* mask, const int32_t* n_nodes, void* out,
                                    long long out_ld, void* ws, size_t ws_bytes, void* stream) {
  DFL_REQUIRE(n_req >= 0, "n_req must be >= 0");
  if (n_req == 0) return DFLASH_OK;
  DFL_REQUIRE(head_dim == 128, "tree attention: head_dim must be 128");
  DFL_REQUIRE(n_kv >= 1 && n_q >= n_kv && n_q % n_kv == 0 && n_q / n_kv <= 4,
              "tree attention: need n_q a multiple of n_kv, at most 4 query heads per KV head");
  DFL_REQUIRE(B >= 0 && B <= 1024, "need 0 <= B <= 1024");
  DFL_REQUIRE(max_ctx >= 0 && max_ctx <= cap, "need 0 <= max_ctx <= cap");
  DFL_REQUIRE(ctx_len && cache_k && cache_v && q && k && v && mask && n_nodes && out,
              "null pointer argument");
  DFL_REQUIRE(q_ld >= (long long)n_q * head_dim && kv_ld >= (long long)n_kv * head_dim &&
                  out_ld >= (long long)n_q * head_dim && q_ld % 8 == 0 && kv_ld % 8 == 0,
              "row strides too small or not multiples of 8");
  DFL_REQUIRE(((reinterpret_cast<uintptr_t>(cache_k) | reinterpret_cast<uintptr_t>(cache_v) |
                reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                reinterpret_cast<uintptr_t>(v)) & 15) == 0,
              "tree attention: cache, q, k and v must be 16-byte aligned");
  DFL_REQUIRE((long long)n_req * n_kv * cap < (1ll << 31) &&
                  (long long)n_req * (B + 1) < (1ll << 31),
              "tree attention: cache or tree rows exceed 2^31");
  const size_t need = dflash_tree_attention_workspace_bytes(n_req, n_q, n_kv, head_dim, B, max_ctx);
  if (!ws || ws_bytes < need)
    return set_error(DFLASH_ERR_WORKSPACE, "tree attention workspace needs %zu bytes, got %zu",
                     need, ws_bytes);
  const int G = n_q / n_kv;
  const int B1 = B + 1;
  const TreePlan pl = tree_plan(n_req, n_kv, B, max_ctx);
  const size_t rows = (size_t)n_req * pl.n_qt * n_kv * pl.n_chunks * G * kNodesPerTile;
  char* w = static_cast<char*>(ws);
  TreeTcParams tp{};
  AttnParams& a = tp.a;
  a.cache_k = static_cast<const __nv_bfloat16*>(cache_k);
  a.cache_v = static_cast<const __nv_bfloat16*>(cache_v);
  a.ctx_len = ctx_len;
  a.cap = cap;
  a.n_req = n_req * pl.n_qt;   // combine: blockIdx.z over (request, query tile)
  a.n_q = n_q;
  a.n_kv = n_kv;
  a.G = G;
  a.L = kNodesPerTile;
  a.chunk = pl.tiles_per_chunk * kTk;
  a.n_chunks = pl.n_chunks;
  a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(head_dim));
  const size_t arr_bytes = align_up((size_t)n_req * pl.n_qt * n_kv * sizeof(int), 256);
  tp.arrivals = reinterpret_cast<int*>(w + 256);
  a.part_o = reinterpret_cast<float*>(w + 256 + arr_bytes);
  a.part_ml = reinterpret_cast<float*>(w + 256 + arr_bytes +
                                       align_up(rows * head_dim * sizeof(float), 256));
  a.out = static_cast<__nv_bfloat16*>(out);
  a.out_ld = out_ld;
  a.n_qt = pl.n_qt;
  a.out_rows = B1;
  tp.mask = mask;
  tp.mask_w = (B1 + 31) / 32;
  tp.n_nodes = n_nodes;
  tp.B1 = B1;
  tp.n_ctx_tiles = pl.tiles_per_chunk;
  tp.status = static_cast<int*>(ws);
  TreeTcMaps maps;
  if (!encode_kmajor_map(&maps.kc, cache_k, n_req * n_kv * cap, head_dim, head_dim, kTk) ||
      !encode_kmajor_map(&maps.vc, cache_v, n_req * n_kv * cap, head_dim, head_dim, kTk) ||
      !encode_kmajor_map(&maps.kt, k, n_req * B1, static_cast<int>(kv_ld), kv_ld, kTk) ||
      !encode_kmajor_map(&maps.vt, v, n_req * B1, static_cast<int>(kv_ld), kv_ld, kTk) ||
      !encode_kmajor_map(&maps.q, q, n_req * B1, static_cast<int>(q_ld), q_ld, kNodesPerTile))
    return set_error(DFLASH_ERR_CUDA, "tree attention: cannot encode the TMA descriptors");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  set_tc_smem_attr();
  {
    TraceScope ts("tree_attn_tc", st);
    launch_k(tree_attn_tc_kernel, dim3(pl.n_chunks, n_kv, n_req * pl.n_qt), dim3(kThreads), kSmem,
             st, maps, tp);
  }
  return check_launch("tree attention");
}

dflash_status dflash_tree_rope(int n_req, int B, int n_heads, int head_dim, float theta,
                               const int32_t* ctx_len, const int32_t* depth, void* x,
                               long long ld, int dtype, void* stream) {
  DFL_REQUIRE(n_req >= 0 && B >= 0 && n_heads >= 1, "bad sizes");
  if (n_req == 0) return DFLASH_OK;
  DFL_REQUIRE(head_dim >= 2 && head_dim % 2 == 0 && head_dim <= 128, "head_dim: even, <= 128");
  DFL_REQUIRE(theta > 0.f, "rope theta must be > 0");
  DFL_REQUIRE(ld >= (long long)n_heads * head_dim, "row stride too small");
  DFL_REQUIRE(ctx_len && depth && x, "null pointer argument");
  DFL_REQUIRE(dtype == DFLASH_BF16 || dtype == DFLASH_F32, "dtype must be bf16 or f32");
  const RopeFreqs fr = rope_freqs(theta, head_dim);
  const long long warps = (long long)n_req * (B + 1) * n_heads;
  const dim3 grid(static_cast<unsigned>((warps * 32 + 255) / 256));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  TraceScope ts("tree_rope", st);
  if (dtype == DFLASH_BF16)
    launch_k(tree_rope_kernel<__nv_bfloat16>, grid, dim3(256), 0, st, n_req, B + 1, n_heads,
             head_dim, fr, ctx_len, depth, static_cast<__nv_bfloat16*>(x), ld);
  else
    launch_k(tree_rope_kernel<float>, grid, dim3(256), 0, st, n_req, B + 1, n_heads, head_dim, fr,
             ctx_len, depth, static_cast<float*>(x), ld);
  return check_launch("tree rope");
}

}  // extern "C"
