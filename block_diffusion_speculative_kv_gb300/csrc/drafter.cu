// Drafter model handle, KV injection and the block pass (steps a1-a6).
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

using namespace dfl;

struct dflash_model {
  dflash_dims dims;
  dflash_weights w;
};

extern "C" {

dflash_status dflash_model_create(const dflash_dims* dims, const dflash_weights* weights,
                                  dflash_model** out) {
  if (!dims || !weights || !out) return set_error(DFLASH_ERR_INVALID_ARG, "null argument");
  return set_error(DFLASH_ERR_UNSUPPORTED, "drafter kernels not built yet");
}

void dflash_model_destroy(dflash_model* model) { std::free(model); }

size_t dflash_workspace_bytes(const dflash_model* model, int n_req, int max_inject_rows, int L,
                              int K) {
  (void)model; (void)n_req; (void)max_inject_rows; (void)L; (void)K;
  return 0;
}

dflash_status dflash_inject_kv(const dflash_model* model, const dflash_cache* cache, int n_req,
                               int n_rows, const int32_t* row_off, const int32_t* pos0,
                               const void* feats, void* ws, size_t ws_bytes, void* stream) {
  (void)model; (void)cache; (void)n_req; (void)n_rows; (void)row_off; (void)pos0;
  (void)feats; (void)ws; (void)ws_bytes; (void)stream;
  return set_error(DFLASH_ERR_UNSUPPORTED, "drafter kernels not built yet");
}

dflash_status dflash_draft_block(const dflash_model* model, const dflash_cache* cache, int n_req,
                                 const int32_t* anchor, const int32_t* ctx_len, int max_ctx,
                                 int L, int K, int32_t* topk_ids, float* topk_logp,
                                 float* logits, void* ws, size_t ws_bytes, void* stream) {
  (void)model; (void)cache; (void)n_req; (void)anchor; (void)ctx_len; (void)max_ctx; (void)L;
  (void)K; (void)topk_ids; (void)topk_logp; (void)logits; (void)ws; (void)ws_bytes;
  (void)stream;
  return set_error(DFLASH_ERR_UNSUPPORTED, "drafter kernels not built yet");
}

}  // extern "C"
