// C ABI of the drafting library: argument validation, workspace layout and
// kernel launches.  Declarations and contracts are in include/dflash.h.
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace dfl {

namespace {
thread_local char g_err[1024] = "";
}

dflash_status set_error(dflash_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

dflash_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(DFLASH_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return DFLASH_OK;
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 148;
    cached[dev] = v;
  }
  return cached[dev];
}

size_t ws_header_bytes() { return 256; }

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("DFLASH_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

namespace {
std::atomic<dflash_trace_fn> g_trace_fn{nullptr};
std::atomic<void*> g_trace_user{nullptr};
}  // namespace

void trace(const char* kernel, int phase, cudaStream_t st) {
  dflash_trace_fn fn = g_trace_fn.load(std::memory_order_acquire);
  if (fn) fn(g_trace_user.load(std::memory_order_relaxed), kernel, phase, st);
}

dflash_status parse_sampling(const dflash_sampling* s, SampleSpec* out) {
  *out = SampleSpec{};
  if (s == nullptr || s->temperature == 0.f) return DFLASH_OK;
  const float T = s->temperature;
  if (!(T >= 1e-6f && T <= 1e6f))
    return set_error(DFLASH_ERR_INVALID_ARG, "sampling temperature must be 0 or in [1e-6, 1e6]");
  out->inv_t = static_cast<float>(1.0 / static_cast<double>(T));
  out->t = T;
  out->seed = s->seed;
  out->row0 = static_cast<long long>(s->row_offset);
  return DFLASH_OK;
}

}  // namespace dfl

using namespace dfl;


extern "C" {

const char* dflash_last_error(void) { return g_err; }

void dflash_set_trace_hook(dflash_trace_fn fn, void* user) {
  g_trace_user.store(user, std::memory_order_relaxed);
  g_trace_fn.store(fn, std::memory_order_release);
}
int dflash_abi_version(void) { return DFLASH_ABI_VERSION; }

dflash_status dflash_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  DFL_REQUIRE(ws != nullptr && ws_bytes >= ws_header_bytes(), "workspace missing or too small");
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return set_error(DFLASH_ERR_CUDA, "workspace init: %s", cudaGetErrorString(e));
  return DFLASH_OK;
}

dflash_status dflash_workspace_set_wait_limit(void* ws, size_t ws_bytes, uint64_t limit_ns,
                                              void* stream) {
  DFL_REQUIRE(ws != nullptr && ws_bytes >= ws_header_bytes(), "workspace missing or too small");
  // a pageable source is staged before cudaMemcpyAsync returns
  const uint64_t v = limit_ns;
  cudaError_t e = cudaMemcpyAsync(static_cast<char*>(ws) + 8, &v, sizeof(v),
                                  cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return set_error(DFLASH_ERR_CUDA, "set wait limit: %s", cudaGetErrorString(e));
  return DFLASH_OK;
}

dflash_status dflash_read_status(void* ws, int* device_status, void* stream) {
  DFL_REQUIRE(ws != nullptr && device_status != nullptr, "null argument");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, ws, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(int), st);
  if (e != cudaSuccess) return set_error(DFLASH_ERR_CUDA, "read status: %s", cudaGetErrorString(e));
  *device_status = host;
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------
// Step a6 standalone: log-softmax + top-K over given logits.
// ---------------------------------------------------------------------------
size_t dflash_topk_workspace_bytes(int rows, int vocab, int K) {
  if (rows < 0 || vocab <= 0 || K < 1 || K > 1024) return 0;
  size_t part = topk_part_bytes(rows, 32);
  if (K > 8 && topk_large_part_bytes(rows, vocab, K) > part)
    part = topk_large_part_bytes(rows, vocab, K);
  return ws_header_bytes() + align_up(sizeof(int) * (size_t)rows, 256) + part;
}

static dflash_status logits_topk_impl(int rows, int vocab, int ld, int dtype, const void* logits,
                                      const dflash_sampling* sampling, int K, int32_t* ids,
                                      float* logp, void* ws, size_t ws_bytes, void* stream) {
  DFL_REQUIRE(rows >= 0, "rows must be >= 0");
  DFL_REQUIRE(vocab >= 1 && ld >= vocab, "need 1 <= vocab <= ld");
  DFL_REQUIRE(K >= 1 && K <= 1024 && K <= vocab, "need 1 <= K <= min(1024, vocab)");
  DFL_REQUIRE(dtype == DFLASH_F32 || dtype == DFLASH_BF16, "dtype must be F32 or BF16");
  SampleSpec smp;
  const dflash_status ps = parse_sampling(sampling, &smp);
  if (ps) return ps;
  if (smp.inv_t > 0.f && K > 32)
    return set_error(DFLASH_ERR_UNSUPPORTED, "sampling draws at most 32 tokens per row");
  if (K > 8 && topk_large_merge_smem(vocab, K) > 200 * 1024)
    return set_error(DFLASH_ERR_UNSUPPORTED, "K = %d is too large for a vocabulary of %d", K,
                     vocab);
  if (rows == 0) return DFLASH_OK;
  DFL_REQUIRE(logits && ids && logp, "null logits/ids/logp");
  const size_t need = dflash_topk_workspace_bytes(rows, vocab, K);
  if (ws == nullptr || ws_bytes < need)
    return set_error(DFLASH_ERR_WORKSPACE, "top-K workspace needs %zu bytes, got %zu", need,
                     ws_bytes);
  char* w = static_cast<char*>(ws);
  TopkLaunch a{};
  a.logits = logits; a.rows = rows; a.vocab = vocab; a.ld = ld; a.dtype = dtype; a.K = K;
  a.splits = topk_splits(rows, vocab);
  a.counters = reinterpret_cast<int*>(w + ws_header_bytes());
  a.part = reinterpret_cast<float*>(w + ws_header_bytes() +
                                    align_up(sizeof(int) * (size_t)rows, 256));
  a.ids = ids; a.logp = logp;
  a.inv_t = smp.inv_t; a.t = smp.t; a.seed = smp.seed; a.row0 = smp.row0;
  a.status = static_cast<int*>(ws);
  if (K > 8 && smp.inv_t == 0.f) {
    const dflash_status ls = launch_topk_large(a, a.part, static_cast<cudaStream_t>(stream));
    if (ls) return ls;
  } else {
    launch_topk(a, static_cast<cudaStream_t>(stream));
  }
  return check_launch("logits_topk");
}

dflash_status dflash_logits_topk(int rows, int vocab, int ld, int dtype, const void* logits,
                                 int K, int32_t* ids, float* logp, void* ws, size_t ws_bytes,
                                 void* stream) {
  return logits_topk_impl(rows, vocab, ld, dtype, logits, nullptr, K, ids, logp, ws, ws_bytes,
                          stream);
}

dflash_status dflash_logits_sample(int rows, int vocab, int ld, int dtype, const void* logits,
                                   const dflash_sampling* sampling, int K, int32_t* ids,
                                   float* logq, void* ws, size_t ws_bytes, void* stream) {
  return logits_topk_impl(rows, vocab, ld, dtype, logits, sampling, K, ids, logq, ws, ws_bytes,
                          stream);
}

// ---------------------------------------------------------------------------
// Step a7: DDTree build.  Step a8: verifier walk.
// ---------------------------------------------------------------------------
dflash_status ddtree_build(int n_req, int D, int K, int B, const float* topk_logp,
                           const int32_t* topk_ids, const int32_t* root_tok, int32_t* n_nodes,
                           int32_t* tok, int32_t* parent, int32_t* depth, int32_t* rank,
                           uint32_t* mask, void* stream) {
  DFL_REQUIRE(n_req >= 0, "n_req must be >= 0");
  DFL_REQUIRE(D >= 1 && D <= 16, "need 1 <= D <= 16");
  DFL_REQUIRE(K >= 1 && K <= 1024, "need 1 <= K <= 1024");
  DFL_REQUIRE(B >= 0 && B <= 1024, "need 0 <= B <= 1024");
  if (n_req == 0) return DFLASH_OK;
  DFL_REQUIRE(topk_logp && topk_ids && root_tok && n_nodes && tok && parent && depth && rank &&
                  mask,
              "null pointer argument");
  TreeBuildLaunch a{n_req, D, K, B, topk_logp, topk_ids, root_tok, n_nodes, tok, parent,
                    depth, rank, mask};
  launch_tree_build(a, static_cast<cudaStream_t>(stream));
  return check_launch("ddtree_build");
}

dflash_status dflash_chain_tree(int n_req, int D, int K, int B, const int32_t* topk_ids,
                                const int32_t* root_tok, int32_t* n_nodes, int32_t* tok,
                                int32_t* parent, int32_t* depth, int32_t* rank, uint32_t* mask,
                                void* stream) {
  DFL_REQUIRE(n_req >= 0, "n_req must be >= 0");
  DFL_REQUIRE(D >= 1 && D <= 16, "need 1 <= D <= 16");
  DFL_REQUIRE(K >= 1 && K <= 1024, "need 1 <= K <= 1024");
  DFL_REQUIRE(B >= 0 && B <= 1024, "need 0 <= B <= 1024");
  if (n_req == 0) return DFLASH_OK;
  DFL_REQUIRE(topk_ids && root_tok && n_nodes && tok && parent && depth && rank && mask,
              "null pointer argument");
  TreeBuildLaunch a{n_req, D, K, B, nullptr, topk_ids, root_tok, n_nodes, tok, parent,
                    depth, rank, mask};
  launch_chain_tree(a, static_cast<cudaStream_t>(stream));
  return check_launch("chain_tree");
}

dflash_status dflash_commit_accepted(int n_req, int D, int B, int feat_dim, int dtype,
                                    const void* tree_feats, long long tree_ld,
                                    const int32_t* accept_len, const int32_t* accepted,
                                    const int32_t* bonus, int32_t* ctx_len, int32_t* anchor,
                                    int32_t* row_off, int32_t* pos0, void* feats, void* stream) {
  DFL_REQUIRE(n_req >= 0, "n_req must be >= 0");
  DFL_REQUIRE(D >= 1 && D <= 16, "need 1 <= D <= 16");
  DFL_REQUIRE(B >= 0 && B <= 1024, "need 0 <= B <= 1024");
  DFL_REQUIRE(dtype == DFLASH_F32 || dtype == DFLASH_BF16, "dtype must be F32 or BF16");
  const int esz = dtype == DFLASH_F32 ? 4 : 2;
  DFL_REQUIRE(feat_dim >= 1 && ((long long)feat_dim * esz) % 16 == 0,
              "feature rows must be a multiple of 16 bytes");
  DFL_REQUIRE(tree_ld >= feat_dim && (tree_ld * esz) % 16 == 0,
              "tree_ld must be >= feat_dim and a multiple of 16 bytes");
  if (n_req == 0) return DFLASH_OK;
  DFL_REQUIRE(tree_feats && accept_len && accepted && bonus && ctx_len && anchor && row_off &&
                  pos0 && feats,
              "null pointer argument");
  DFL_REQUIRE(((reinterpret_cast<uintptr_t>(tree_feats) | reinterpret_cast<uintptr_t>(feats)) &
               15u) == 0,
              "feature buffers must be 16-byte aligned");
  CommitLaunch a{n_req, D, B, feat_dim * esz, tree_feats, tree_ld * esz, accept_len, accepted,
                 bonus, ctx_len, anchor, row_off, pos0, feats};
  launch_commit(a, static_cast<cudaStream_t>(stream));
  return check_launch("commit_accepted");
}

dflash_status ddtree_accept(int n_req, int D, int B, const int32_t* n_nodes, const int32_t* tok,
                            const int32_t* parent, const int32_t* target_tok,
                            int32_t* accept_len, int32_t* accepted, int32_t* bonus,
                            void* stream) {
  DFL_REQUIRE(n_req >= 0, "n_req must be >= 0");
  DFL_REQUIRE(D >= 1 && D <= 16, "need 1 <= D <= 16");
  DFL_REQUIRE(B >= 0 && B <= 1024, "need 0 <= B <= 1024");
  if (n_req == 0) return DFLASH_OK;
  DFL_REQUIRE(n_nodes && tok && parent && target_tok && accept_len && accepted && bonus,
              "null pointer argument");
  TreeAcceptLaunch a{n_req, D, B, n_nodes, tok, parent, target_tok, accept_len, accepted, bonus};
  launch_tree_accept(a, static_cast<cudaStream_t>(stream));
  return check_launch("ddtree_accept");
}

}  // extern "C"
