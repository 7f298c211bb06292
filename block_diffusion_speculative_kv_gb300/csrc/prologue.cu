// Small per-call kernels that start the block pass and the injection.
//
// block_prologue (step a3): x_j = E[anchor] for j = 0 and E[mask] otherwise
// ("DFlash: Block Diffusion for Flash Speculative Decoding", section 3.4.4,
// block [anchor, mask x (L-1)]), written as the fp32 residual x, the
// gain-scaled GEMM operand xn = x * g (first attention norm) and per-128-column
// sums of squares for the RMS factor; plus the rotary (cos, sin) table of the
// block positions ctx_len + j.
// inject_rope: the rotary table of the injected cache positions.
// The frequencies theta^(-2i/hd) come from the host in double precision; the
// angle pos * freq is formed and reduced modulo 2*pi in double (three FP64
// operations), then the reduced angle's sine and cosine are taken in fp32.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace dfl {

namespace {

template <typename T>
__global__ void __launch_bounds__(128)
block_prologue_kernel(const T* __restrict__ embed, const T* __restrict__ gain,
                      const int* __restrict__ anchor, const int* __restrict__ ctx_len, int n_req,
                      int L, int d, int vocab, int mask_id, int head_dim, const RopeFreqs fr,
                      float* __restrict__ x, T* __restrict__ xn, float* __restrict__ ssq,
                      float2* __restrict__ rope, int* status) {
  const int R = n_req * L;
  const int row = blockIdx.x;
  const int req = row / L, j = row % L;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // Everything read here is an input of the call (or a weight): the previous
  // kernel writes none of it, and every kernel before that one has completed
  // once this one runs.  So the loads and the arithmetic come first and only
  // the stores wait for the previous kernel (which may share these workspace
  // regions).
  int tok = (j == 0) ? anchor[req] : mask_id;
  const bool bad_tok = tok < 0 || tok >= vocab;
  if (bad_tok) tok = 0;
  // warp w takes the 128-column parts w, w+4, ...; lane l the 4 columns 4l..4l+3
  const int parts = (d + 127) / 128;
  constexpr int kParts = 8;   // parts per warp held in registers (the first 4 * 8 * 128 columns)
  const T* erow = embed + (size_t)tok * d;
  float v[kParts][4], g[kParts][4], sq[kParts];
#pragma unroll
  for (int u = 0; u < kParts; ++u) {
    const int p = warp + 4 * u;
    sq[u] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = p * 128 + lane * 4 + e;
      const bool ok = p < parts && c < d;
      v[u][e] = ok ? to_f32<T>(erow[c]) : 0.f;
      g[u][e] = ok ? to_f32<T>(gain[c]) : 0.f;
      sq[u] += v[u][e] * v[u][e];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sq[u] += __shfl_xor_sync(0xffffffffu, sq[u], off);
  }
  const int half = head_dim / 2;
  const int pos = ctx_len[req] + j;
  const int i_rope = threadIdx.x;
  const float2 cs = i_rope < half ? rope_cs(pos, i_rope, fr) : make_float2(1.f, 0.f);
  pdl_wait();
  pdl_trigger();
  if (bad_tok && threadIdx.x == 0) record_status(status, DFLASH_ERR_INVALID_ARG);
#pragma unroll
  for (int u = 0; u < kParts; ++u) {
    const int p = warp + 4 * u;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = p * 128 + lane * 4 + e;
      if (p < parts && c < d) {
        x[(size_t)row * d + c] = v[u][e];
        xn[(size_t)row * d + c] = from_f32<T>(v[u][e] * g[u][e]);
      }
    }
    if (lane == 0 && p < parts) ssq[(size_t)p * R + row] = sq[u];
  }
  if (i_rope < half) rope[(size_t)row * half + i_rope] = cs;
  // columns past the first 4 * kParts parts (d > 4096): loaded after the wait
  for (int p = warp + 4 * kParts; p < parts; p += 4) {
    float s2 = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = p * 128 + lane * 4 + e;
      if (c < d) {
        const float a = to_f32<T>(erow[c]);
        x[(size_t)row * d + c] = a;
        xn[(size_t)row * d + c] = from_f32<T>(a * to_f32<T>(gain[c]));
        s2 += a * a;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, off);
    if (lane == 0) ssq[(size_t)p * R + row] = s2;
  }
}

__global__ void inject_rope_kernel(const int* __restrict__ row_off, const int* __restrict__ pos0,
                                   int n_req, int n_rows, int head_dim, const RopeFreqs fr,
                                   float2* __restrict__ rope) {
  const int half = head_dim / 2;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  // (inputs only: computed before the wait, stored after it)
  const bool live = idx < (long long)n_rows * half;
  float2 cs = make_float2(1.f, 0.f);
  if (live) {
    const int row = static_cast<int>(idx / half), i = static_cast<int>(idx % half);
    int lo = 0, hi = n_req - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (row_off[mid] <= row) lo = mid;
      else hi = mid - 1;
    }
    const int pos = pos0[lo] + (row - row_off[lo]);
    cs = rope_cs(pos, i, fr);
  }
  pdl_wait();
  pdl_trigger();
  if (live) rope[idx] = cs;
}

}  // namespace

RopeFreqs rope_freqs(float theta, int head_dim) {
  RopeFreqs r{};
  for (int i = 0; i < head_dim / 2 && i < 64; ++i)
    r.f[i] = std::pow(static_cast<double>(theta), -2.0 * i / head_dim);
  return r;
}

void launch_block_prologue(const BlockPrologueLaunch& a, cudaStream_t st) {
  const int R = a.n_req * a.L;
  if (R <= 0) return;
  TraceScope ts("block_prologue", st);
  if (a.bf16) {
    launch_k(block_prologue_kernel<__nv_bfloat16>, dim3(R), dim3(128), 0, st,
             static_cast<const __nv_bfloat16*>(a.embed), static_cast<const __nv_bfloat16*>(a.gain),
             a.anchor, a.ctx_len, a.n_req, a.L, a.d, a.vocab, a.mask_id, a.head_dim, a.freqs, a.x,
             static_cast<__nv_bfloat16*>(a.xn), a.ssq, a.rope, a.status);
  } else {
    launch_k(block_prologue_kernel<float>, dim3(R), dim3(128), 0, st,
             static_cast<const float*>(a.embed), static_cast<const float*>(a.gain), a.anchor,
             a.ctx_len, a.n_req, a.L, a.d, a.vocab, a.mask_id, a.head_dim, a.freqs, a.x,
             static_cast<float*>(a.xn), a.ssq, a.rope, a.status);
  }
}

void launch_inject_rope(const int* row_off, const int* pos0, int n_req, int n_rows, int head_dim,
                        const RopeFreqs& freqs, float2* rope, cudaStream_t st) {
  const long long n = (long long)n_rows * (head_dim / 2);
  if (n <= 0) return;
  TraceScope ts("inject_rope", st);
  launch_k(inject_rope_kernel, dim3(static_cast<int>((n + 255) / 256)), dim3(256), 0, st,
           row_off, pos0, n_req, n_rows, head_dim, freqs, rope);
}

}  // namespace dfl
