// Internal helpers shared by the kernels of the drafting library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "dflash.h"

namespace dfl {

constexpr int kWarp = 32;

// ---------------------------------------------------------------------------
// Host-side error reporting (thread-local message, see dflash_last_error).
// ---------------------------------------------------------------------------
dflash_status set_error(dflash_status st, const char* fmt, ...);
dflash_status check_launch(const char* what);

// ---------------------------------------------------------------------------
// Device-side status word: the first error recorded wins.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// Element conversions.
// ---------------------------------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Order-preserving map of a float onto uint32 (larger float -> larger code);
// -0.0 is folded onto +0.0 first.
__device__ __forceinline__ uint32_t ordered_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_ordered_bits(uint32_t h) {
  uint32_t u = (h & 0x80000000u) ? (h & 0x7FFFFFFFu) : ~h;
  return __uint_as_float(u);
}

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ size_t align_up(size_t a, size_t b) {
  return (a + b - 1) / b * b;
}

// Number of SMs of the current device (cached per device on the host).
int num_sms();

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Kernels of one call are launched so that the
// next kernel may start while the previous one finishes.  Every kernel calls
// pdl_wait() before it touches memory written by an earlier kernel of the
// stream (and before any global write), then pdl_trigger(); work done before
// pdl_wait() only reads data no kernel of the call writes (weights, the
// context part of the KV cache) into the CTA's own shared memory.  Because a
// kernel triggers only after its own wait, when a kernel starts its
// predecessor's predecessor has completed.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
bool pdl_enabled();  // DFLASH_PDL=0 in the environment turns it off

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launch tracing (dflash_set_trace_hook): host callbacks around each launch.
void trace(const char* kernel, int phase, cudaStream_t st);
struct TraceScope {
  const char* name;
  cudaStream_t st;
  TraceScope(const char* n, cudaStream_t s) : name(n), st(s) { trace(name, 0, st); }
  ~TraceScope() { trace(name, 1, st); }
};

}  // namespace dfl

// Argument check of a C-ABI entry point: on failure, record the message and
// return DFLASH_ERR_INVALID_ARG.
#define DFL_REQUIRE(cond, ...)                                            \
  do {                                                                    \
    if (!(cond)) return dfl::set_error(DFLASH_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)
