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

__device__ __forceinline__ float2 rope_cs(int pos, int i, const RopeFreqs& fr) {
  const double two_pi = 6.283185307179586476925;
  const double a = static_cast<double>(pos) * fr.f[i];
  const double k = rint(a * (1.0 / two_pi));
  const float r = static_cast<float>(fma(-k, two_pi, a));
  float s, c;
  sincosf(r, &s, &c);
  return make_float2(c, s);
}

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
  pdl_wait();
  pdl_trigger();
  int tok = (j == 0) ? anchor[req] : mask_id;
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) record_status(status, DFLASH_ERR_INVALID_ARG);
    tok = 0;
  }
  // warp w takes the 128-column parts w, w+4, ...; lane l the 4 columns 4l..4l+3
  const int parts = (d + 127) / 128;
  constexpr int kMaxParts = 64;  // d <= 8192
  const T* erow = embed + (size_t)tok * d;
  for (int p0 = warp; p0 < parts; p0 += 4 * 8) {
    float v[8][4], g[8][4];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int p = p0 + 4 * u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = p * 128 + lane * 4 + e;
        const bool ok = p < parts && c < d;
        v[u][e] = ok ? to_f32<T>(erow[c]) : 0.f;
        g[u][e] = ok ? to_f32<T>(gain[c]) : 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int p = p0 + 4 * u;
      float sq = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = p * 128 + lane * 4 + e;
        if (p < parts && c < d) {
          x[(size_t)row * d + c] = v[u][e];
          xn[(size_t)row * d + c] = from_f32<T>(v[u][e] * g[u][e]);
        }
        sq += v[u][e] * v[u][e];
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
      if (lane == 0 && p < parts) ssq[(size_t)p * R + row] = sq;
    }
  }
  (void)kMaxParts;
  const int half = head_dim / 2;
  const int pos = ctx_len[req] + j;
  for (int i = threadIdx.x; i < half; i += blockDim.x)
    rope[(size_t)row * half + i] = rope_cs(pos, i, fr);
}

__global__ void inject_rope_kernel(const int* __restrict__ row_off, const int* __restrict__ pos0,
                                   int n_req, int n_rows, int head_dim, const RopeFreqs fr,
                                   float2* __restrict__ rope) {
  const int half = head_dim / 2;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (idx >= (long long)n_rows * half) return;
  const int row = static_cast<int>(idx / half), i = static_cast<int>(idx % half);
  int lo = 0, hi = n_req - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (row_off[mid] <= row) lo = mid;
    else hi = mid - 1;
  }
  const int pos = pos0[lo] + (row - row_off[lo]);
  rope[idx] = rope_cs(pos, i, fr);
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
