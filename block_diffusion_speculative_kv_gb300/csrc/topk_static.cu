// Log-softmax + top-K for callers that cannot provide a workspace.
//
// Some callers cannot allocate device memory at the time they need this step:
// a serving loop whose device memory is carved up once at start-up by its own
// allocator and that must not call cudaMalloc afterwards (cudaMalloc can
// synchronise the device and stall every stream), or a plugin host that hands
// out input and output buffers but exposes no way to ask for scratch.  For
// them dflash_logits_topk_noalloc runs the same kernel as dflash_logits_topk,
// with its scratch (per-row arrival counters and split-row partial records) in
// a fixed array that is part of the library image itself.
//
// The array is a file-scope __device__ object of kStaticScratchBytes bytes;
// every GPU on which the library is loaded holds one copy until the process
// exits.  Host code cannot use the array's name as a device address, so the
// first call on each device looks the address up with cudaGetSymbolAddress
// (with that device current) and caches it; make that first call before any
// stream capture.  All calls on a device share the array: calls that overlap
// on the GPU (different streams, or graphs replayed concurrently) race and
// must be serialised by the caller.  Each call clears the counters it uses
// before its kernel runs.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace dfl {

namespace {

constexpr int kStaticMaxRows = 4096;
constexpr int kStaticMaxRecords = 1024;   // rows x splits held when a row is split
constexpr size_t kRecordFloats = 2 + 2 * 32;
constexpr size_t kCounterBytes = sizeof(int) * kStaticMaxRows;
constexpr size_t kStaticScratchBytes =
    kCounterBytes + sizeof(float) * kRecordFloats * kStaticMaxRecords;

static __device__ __align__(256) unsigned char g_topk_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_addr[64] = {nullptr};

dflash_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return set_error(DFLASH_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return set_error(DFLASH_ERR_UNSUPPORTED, "device index >= 64");
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess || p == nullptr)
      return set_error(DFLASH_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return DFLASH_OK;
}

}  // namespace
}  // namespace dfl

using namespace dfl;

extern "C" dflash_status dflash_logits_topk_noalloc(int rows, int vocab, int ld, int dtype,
                                                    const void* logits, int K, int32_t* ids,
                                                    float* logp, void* stream) {
  if (rows < 0) return set_error(DFLASH_ERR_INVALID_ARG, "rows must be >= 0");
  if (rows > kStaticMaxRows)
    return set_error(DFLASH_ERR_UNSUPPORTED,
                     "dflash_logits_topk_noalloc handles at most %d rows (got %d); use "
                     "dflash_logits_topk with a workspace",
                     kStaticMaxRows, rows);
  if (vocab < 1 || ld < vocab) return set_error(DFLASH_ERR_INVALID_ARG, "need 1 <= vocab <= ld");
  if (K < 1 || K > 32 || K > vocab)
    return set_error(DFLASH_ERR_INVALID_ARG, "need 1 <= K <= min(32, vocab)");
  if (dtype != DFLASH_F32 && dtype != DFLASH_BF16)
    return set_error(DFLASH_ERR_INVALID_ARG, "dtype must be F32 or BF16");
  if (rows == 0) return DFLASH_OK;
  if (!logits || !ids || !logp) return set_error(DFLASH_ERR_INVALID_ARG, "null logits/ids/logp");
  void* base = nullptr;
  dflash_status st = scratch_address(&base);
  if (st != DFLASH_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  TopkLaunch a{};
  a.logits = logits;
  a.rows = rows;
  a.vocab = vocab;
  a.ld = ld;
  a.dtype = dtype;
  a.K = K;
  a.splits = topk_splits(rows, vocab);
  while (a.splits > 1 && (long long)rows * a.splits > kStaticMaxRecords) --a.splits;
  a.counters = static_cast<int*>(base);
  a.part = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kCounterBytes);
  a.ids = ids;
  a.logp = logp;
  // counters must start at zero whatever an earlier call left behind
  cudaError_t e = cudaMemsetAsync(a.counters, 0, sizeof(int) * (size_t)rows, s);
  if (e != cudaSuccess)
    return set_error(DFLASH_ERR_CUDA, "clearing the static counters: %s", cudaGetErrorString(e));
  launch_topk(a, s);
  return check_launch("logits_topk_noalloc");
}
