// Drafter model handle, workspace layout, KV injection (steps a1-a2) and the
// block pass with LM head and top-K (steps a3-a6).  Contracts: include/dflash.h.
//
// Call sequence of dflash_draft_block for a model of n_layers layers
// ("DFlash: Block Diffusion for Flash Speculative Decoding", section 3.4.4):
//   block_prologue                          x, xn = x*g, RMS partials, RoPE table
//   per layer: GEMM  xn . [W_q|W_k|W_v]^T    -> QKV epilogue (RMS scale, RoPE)
//              attention over [context ; block]  (split-KV + combine)
//              GEMM  o . W_o^T               -> residual epilogue (x, xn, RMS partials)
//              GEMM  xn . [W_gate|W_up]^T    -> SwiGLU epilogue
//              GEMM  h . W_down^T            -> residual epilogue
//   GEMM  xn . W_lm^T                       -> logits of the L-1 mask rows (fp32)
//   log-softmax + top-K per row             (DDTree page, section 3.4.2)
// dflash_inject_kv (section 3.4.3): GEMM feats . W_proj^T -> f; GEMM
// f . [U_K|U_V]^T (all layers stacked) -> KV epilogue (RoPE on K, cache scatter).
#include <cstdlib>
#include <cstring>
#include <new>

#include "attention.h"
#include "common.cuh"
#include "gemm.h"
#include "kernels.h"

using namespace dfl;

struct dflash_model {
  dflash_dims dims;
  dflash_weights w;
  bool bf16;
  RopeFreqs freqs;
  CUtensorMap tm_proj, tm_ukv, tm_lm;
  CUtensorMap tm_qkv[DFLASH_MAX_LAYERS], tm_o[DFLASH_MAX_LAYERS], tm_gu[DFLASH_MAX_LAYERS],
      tm_down[DFLASH_MAX_LAYERS];
};

namespace {

size_t esize(const dflash_dims& d) { return d.dtype == DFLASH_BF16 ? 2 : 4; }

// Workspace regions of a model-sized workspace (byte offsets).
struct WsLayout {
  size_t counters, x, xn, ssq, qkv, attn_o, h, logits, gpart, apart_o, apart_ml, tpart, tkpart,
      rope_blk,
      f, rope_inj, total;
  int attn_chunks_cap;
  int attn_arrivals;   // first int of the tensor-core attention's arrival counters
};

int ssq_parts(const dflash_dims& d) { return (d.d + 127) / 128; }

WsLayout ws_layout(const dflash_model& m, int n_req, int max_inject_rows, int L, int K) {
  const dflash_dims& d = m.dims;
  const size_t es = esize(d);
  const int R = n_req * L;
  const int D = L - 1;
  const int G = d.n_q / d.n_kv;
  const int qkv_dim = (d.n_q + 2 * d.n_kv) * d.head_dim;
  const int sms = num_sms();
  WsLayout w{};
  size_t off = 256;  // status word and reserved header
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  // the GEMM chains' counters, one arrival counter per top-K row, then one per
  // (request, KV head) of the tensor-core attention.  The counters persist
  // between calls (every launch leaves them at zero), so the region's size
  // does not depend on L or the injected rows: calls with other L or injected
  // rows lay out the regions after it differently (up to 16 rows per request).
  const int R16 = 16 * n_req;
  const int NKV = n_req * d.n_kv;
  w.attn_arrivals = gemm_counter_ints() + (4096 > R16 ? 4096 : R16);
  const int n_counters = w.attn_arrivals + (4096 > NKV ? 4096 : NKV);
  w.counters = take(sizeof(int) * n_counters);
  w.x = take(sizeof(float) * (size_t)R * d.d);
  w.xn = take(es * (size_t)R * d.d);
  w.ssq = take(sizeof(float) * (size_t)ssq_parts(d) * R);
  w.qkv = take(es * (size_t)R * qkv_dim);
  w.attn_o = take(es * (size_t)R * d.n_q * d.head_dim);
  w.h = take(es * (size_t)R * d.d_ff);
  w.logits = take(sizeof(float) * (size_t)n_req * D * d.vocab);
  // GEMM partial sums: the largest plan among the GEMMs of a call
  size_t gp = 0;
  if (m.bf16) {
    // the largest need among all activation-row counts up to this call's maximum:
    // for a fixed row tile and row-tile count the partial count peaks at the
    // smallest such row count, so the row-tile sizes and the first row count of
    // every count of 256-row tiles cover every row count in between
    const int Mmax = R > max_inject_rows ? R : max_inject_rows;
    int Ms[48];
    int nm = 0;
    for (int t = 16; t <= tc_row_tile(Mmax); t <<= 1) Ms[nm++] = t;
    for (int t = 1; 256 * t < Mmax && nm < 44; ++t) Ms[nm++] = 256 * t + 1;
    Ms[nm++] = R;
    if (max_inject_rows > 0) Ms[nm++] = max_inject_rows;
    for (int mi = 0; mi < nm; ++mi) {
      const int M = Ms[mi];
      const int NK[7][2] = {{qkv_dim, d.d}, {d.d, d.n_q * d.head_dim}, {2 * d.d_ff, d.d},
                            {d.d, d.d_ff}, {d.vocab, d.d}, {d.d, d.n_feat * d.d_feat},
                            {d.n_layers * 2 * d.n_kv * d.head_dim, d.d}};
      for (auto& nk : NK) {
        const TcPlan pl = tc_plan(M, nk[0], nk[1], sms);
        if (pl.part_bytes > gp) gp = pl.part_bytes;
      }
    }
  }
  w.gpart = take(gp);
  // attention partials: enough chunks for ~2 CTAs per SM plus the block chunk
  int cap_chunks = (4 * sms + d.n_kv * n_req - 1) / (d.n_kv * n_req) + 2;
  w.attn_chunks_cap = cap_chunks;
  const size_t arows = (size_t)n_req * d.n_kv * cap_chunks * G * L;
  w.apart_o = take(m.bf16 ? sizeof(float) * arows * d.head_dim : 0);
  w.apart_ml = take(m.bf16 ? sizeof(float) * arows * 2 : 0);
  size_t tp = topk_part_bytes(n_req * D, 32);
  if (K > 8 && topk_large_part_bytes(n_req * D, d.vocab, K) > tp)
    tp = topk_large_part_bytes(n_req * D, d.vocab, K);
  w.tpart = take(tp);
  // records of the top-K fused into the LM head (batch-1 row tile)
  w.tkpart = take(m.bf16 && tc_row_tile(R) == 16 ? sizeof(float) * sms * R * kTkStride : 0);
  w.rope_blk = take(sizeof(float2) * (size_t)R * (d.head_dim / 2));
  w.f = take(es * (size_t)max_inject_rows * d.d);
  w.rope_inj = take(sizeof(float2) * (size_t)max_inject_rows * (d.head_dim / 2));
  w.total = off;
  (void)K;
  return w;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

dflash_status validate_dims(const dflash_dims& d) {
  if (d.n_layers < 1 || d.n_layers > DFLASH_MAX_LAYERS)
    return set_error(DFLASH_ERR_INVALID_ARG, "n_layers must be in [1, %d]", DFLASH_MAX_LAYERS);
  if (d.d <= 0 || d.n_q <= 0 || d.n_kv <= 0 || d.d_ff <= 0 || d.vocab <= 0 || d.n_feat <= 0 ||
      d.d_feat <= 0)
    return set_error(DFLASH_ERR_INVALID_ARG, "all sizes must be positive");
  if (d.n_q % d.n_kv != 0) return set_error(DFLASH_ERR_INVALID_ARG, "n_q %% n_kv != 0");
  if (d.head_dim != 64 && d.head_dim != 128)
    return set_error(DFLASH_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (d.mask_id < 0 || d.mask_id >= d.vocab)
    return set_error(DFLASH_ERR_INVALID_ARG, "mask_id out of range");
  if (d.dtype != DFLASH_F32 && d.dtype != DFLASH_BF16)
    return set_error(DFLASH_ERR_INVALID_ARG, "dtype must be F32 or BF16");
  if (!(d.rope_theta > 0.f) || !(d.rms_eps >= 0.f))
    return set_error(DFLASH_ERR_INVALID_ARG, "rope_theta must be > 0 and rms_eps >= 0");
  if (d.dtype == DFLASH_BF16) {
    const int q = d.n_q * d.head_dim;
    if (d.d % 128 || (d.n_feat * d.d_feat) % 128 || q % 128 || d.d_ff % 128)
      return set_error(DFLASH_ERR_UNSUPPORTED,
                       "bf16 models need d, n_feat*d_feat, n_q*head_dim, d_ff multiples of 128");
    if ((d.n_q / d.n_kv) > 4)
      return set_error(DFLASH_ERR_UNSUPPORTED, "bf16 attention supports n_q/n_kv <= 4");
  }
  return DFLASH_OK;
}

EpiParams epi_base(const dflash_model& m, int M_rows, int N_feat) {
  EpiParams e{};
  e.M_rows = M_rows;
  e.N_feat = N_feat;
  e.inv_d = 1.f / static_cast<float>(m.dims.d);
  e.eps = m.dims.rms_eps;
  e.ssq_parts = ssq_parts(m.dims);
  e.head_dim = m.dims.head_dim;
  return e;
}

struct CallCtx {
  const dflash_model* m;
  char* ws;
  WsLayout L;
  cudaStream_t st;
  int* status;
  int* counters;
};

// One GEMM of a chain: acc = X . W^T with epilogue e.  X [M][K] (row stride
// ldx, elements).
struct Step {
  const CUtensorMap* tmW;
  const void* W;
  const void* X;
  long long ldx;
  int N, K;
  EpiParams e;
};

// A chain of dependent GEMMs over the same M activation rows: one launch on
// the tensor-core path, one launch per GEMM on the fp32 path.
dflash_status run_chain(const CallCtx& c, const Step* s, int n, int M) {
  if (M <= 0) return DFLASH_OK;
  if (c.m->bf16) {
    GemmPhase ph[kMaxPhases];
    for (int i = 0; i < n; ++i) ph[i] = GemmPhase{s[i].tmW, s[i].X, s[i].ldx, s[i].N, s[i].K, s[i].e};
    return launch_gemm_chain(ph, n, M, reinterpret_cast<float*>(c.ws + c.L.gpart), c.counters,
                             c.status, c.st);
  }
  for (int i = 0; i < n; ++i) {
    const dflash_status st =
        launch_gemm_f32(static_cast<const float*>(s[i].X), s[i].ldx,
                        static_cast<const float*>(s[i].W), M, s[i].N, s[i].K, s[i].e, c.st);
    if (st) return st;
  }
  return DFLASH_OK;
}

}  // namespace

extern "C" {

dflash_status dflash_model_create(const dflash_dims* dims, const dflash_weights* weights,
                                  dflash_model** out) {
  if (!dims || !weights || !out) return set_error(DFLASH_ERR_INVALID_ARG, "null argument");
  dflash_status st = validate_dims(*dims);
  if (st != DFLASH_OK) return st;
  const dflash_weights& w = *weights;
  const void* req_ptrs[] = {w.w_proj, w.embed, w.lm_head, w.final_norm, w.u_kv};
  for (const void* p : req_ptrs)
    if (!p || !aligned16(p)) return set_error(DFLASH_ERR_INVALID_ARG, "weight pointer null or not 16-byte aligned");
  for (int l = 0; l < dims->n_layers; ++l) {
    const void* lp[] = {w.attn_norm[l], w.w_qkv[l], w.wo[l], w.mlp_norm[l], w.w_gate_up[l],
                        w.w_down[l]};
    for (const void* p : lp)
      if (!p || !aligned16(p))
        return set_error(DFLASH_ERR_INVALID_ARG, "layer %d weight pointer null or misaligned", l);
  }
  dflash_model* m = new (std::nothrow) dflash_model();
  if (!m) return set_error(DFLASH_ERR_INVALID_ARG, "out of host memory");
  m->dims = *dims;
  m->w = w;
  m->bf16 = dims->dtype == DFLASH_BF16;
  m->freqs = rope_freqs(dims->rope_theta, dims->head_dim);
  if (m->bf16) {
    const dflash_dims& d = *dims;
    const int qkv_dim = (d.n_q + 2 * d.n_kv) * d.head_dim;
    const int qd = d.n_q * d.head_dim;
    bool ok = encode_kmajor_map(&m->tm_proj, w.w_proj, d.d, d.n_feat * d.d_feat,
                                (long long)d.n_feat * d.d_feat, 128) &&
              encode_kmajor_map(&m->tm_ukv, w.u_kv, d.n_layers * 2 * d.n_kv * d.head_dim, d.d,
                                d.d, 128) &&
              encode_kmajor_map(&m->tm_lm, w.lm_head, d.vocab, d.d, d.d, 128);
    for (int l = 0; ok && l < d.n_layers; ++l) {
      ok = encode_kmajor_map(&m->tm_qkv[l], w.w_qkv[l], qkv_dim, d.d, d.d, 128) &&
           encode_kmajor_map(&m->tm_o[l], w.wo[l], d.d, qd, qd, 128) &&
           encode_kmajor_map(&m->tm_gu[l], w.w_gate_up[l], 2 * d.d_ff, d.d, d.d, 128) &&
           encode_kmajor_map(&m->tm_down[l], w.w_down[l], d.d, d.d_ff, d.d_ff, 128);
    }
    if (!ok) {
      delete m;
      return set_error(DFLASH_ERR_CUDA, "cannot encode weight TMA descriptors");
    }
  }
  *out = m;
  return DFLASH_OK;
}

void dflash_model_destroy(dflash_model* model) { delete model; }

size_t dflash_workspace_bytes(const dflash_model* model, int n_req, int max_inject_rows, int L,
                              int K) {
  if (!model || n_req < 1 || max_inject_rows < 0 || L < 2 || L > 16 || K < 1 || K > 1024)
    return 0;
  return ws_layout(*model, n_req, max_inject_rows, L, K).total;
}

// Validation of the injection's arguments (the workspace is checked by the caller).
static dflash_status check_inject(const dflash_model* model, const dflash_cache* cache, int n_req,
                           int n_rows, const int32_t* row_off, const int32_t* pos0,
                           const void* feats) {
  if (!model || !cache) return set_error(DFLASH_ERR_INVALID_ARG, "null model or cache");
  if (n_req < 1 || n_req > cache->n_req)
    return set_error(DFLASH_ERR_INVALID_ARG, "n_req must be in [1, cache->n_req]");
  if (n_rows < 0) return set_error(DFLASH_ERR_INVALID_ARG, "n_rows must be >= 0");
  if (n_rows == 0) return DFLASH_OK;
  if (!row_off || !pos0 || !feats)
    return set_error(DFLASH_ERR_INVALID_ARG, "null row_off/pos0/feats");
  const dflash_dims& d = model->dims;
  for (int l = 0; l < d.n_layers; ++l)
    if (!cache->k[l] || !cache->v[l]) return set_error(DFLASH_ERR_INVALID_ARG, "null cache layer %d", l);
  if (cache->cap < 1) return set_error(DFLASH_ERR_INVALID_ARG, "cache cap must be >= 1");
  if (model->bf16 && !aligned16(feats))
    return set_error(DFLASH_ERR_INVALID_ARG, "feats must be 16-byte aligned");
  return DFLASH_OK;
}

// Steps a1 + a2 as two GEMM steps (f = feats . W_proj^T; [K|V] of every layer
// = f . U^T, K rotated, scattered into the cache), after the RoPE table of the
// injected positions is launched.
static dflash_status inject_steps(const dflash_model* model, const dflash_cache* cache, int n_req,
                           int n_rows, const int32_t* row_off, const int32_t* pos0,
                           const void* feats, const CallCtx& c, Step (&out)[2]) {
  const dflash_dims& d = model->dims;
  float2* rope = reinterpret_cast<float2*>(c.ws + c.L.rope_inj);
  launch_inject_rope(row_off, pos0, n_req, n_rows, d.head_dim, model->freqs, rope, c.st);
  dflash_status st = check_launch("inject rope");
  if (st) return st;
  void* f = c.ws + c.L.f;
  EpiParams e1 = epi_base(*model, n_rows, d.d);
  e1.kind = EPI_STORE;
  e1.ssq_in = nullptr;
  e1.out = f;
  e1.ldo = d.d;
  EpiParams e2 = epi_base(*model, n_rows, d.n_layers * 2 * d.n_kv * d.head_dim);
  e2.kind = EPI_KV;
  e2.ssq_in = nullptr;
  e2.rope = rope;
  for (int l = 0; l < d.n_layers; ++l) {
    e2.cache_k[l] = cache->k[l];
    e2.cache_v[l] = cache->v[l];
  }
  e2.n_kv = d.n_kv;
  e2.cap = cache->cap;
  e2.n_req = n_req;
  e2.row_off = row_off;
  e2.pos0 = pos0;
  out[0] = Step{&model->tm_proj, model->w.w_proj, feats, (long long)d.n_feat * d.d_feat, d.d,
                d.n_feat * d.d_feat, e1};
  out[1] = Step{&model->tm_ukv, model->w.u_kv, f, d.d, d.n_layers * 2 * d.n_kv * d.head_dim,
                d.d, e2};
  return DFLASH_OK;
}

dflash_status dflash_inject_kv(const dflash_model* model, const dflash_cache* cache, int n_req,
                               int n_rows, const int32_t* row_off, const int32_t* pos0,
                               const void* feats, void* ws, size_t ws_bytes, void* stream) {
  dflash_status st = check_inject(model, cache, n_req, n_rows, row_off, pos0, feats);
  if (st || n_rows == 0) return st;
  const dflash_dims& d = model->dims;
  // the workspace must have been sized for at least n_rows injected rows
  const WsLayout L = ws_layout(*model, n_req, n_rows, 2, 1);
  const size_t need = L.rope_inj + sizeof(float2) * (size_t)n_rows * (d.head_dim / 2);
  if (!ws || ws_bytes < need)
    return set_error(DFLASH_ERR_WORKSPACE, "inject workspace needs %zu bytes, got %zu", need,
                     ws_bytes);
  CallCtx c{model, static_cast<char*>(ws), L, static_cast<cudaStream_t>(stream),
            static_cast<int*>(ws), reinterpret_cast<int*>(static_cast<char*>(ws) + L.counters)};
  Step chain[2];
  st = inject_steps(model, cache, n_req, n_rows, row_off, pos0, feats, c, chain);
  if (st) return st;
  return run_chain(c, chain, 2, n_rows);
}

static dflash_status check_draft(const dflash_model* model, const dflash_cache* cache, int n_req,
                          const int32_t* anchor, const int32_t* ctx_len, int max_ctx, int L,
                          int K, int32_t* topk_ids, float* topk_logp) {
  if (!model || !cache) return set_error(DFLASH_ERR_INVALID_ARG, "null model or cache");
  const dflash_dims& d = model->dims;
  if (n_req < 1 || n_req > cache->n_req)
    return set_error(DFLASH_ERR_INVALID_ARG, "n_req must be in [1, cache->n_req]");
  if (L < 2 || L > 16) return set_error(DFLASH_ERR_INVALID_ARG, "L must be in [2, 16]");
  if (K < 1 || K > 1024 || K > d.vocab)
    return set_error(DFLASH_ERR_INVALID_ARG, "K must be in [1, min(1024, vocab)]");
  if (K > 8 && topk_large_merge_smem(d.vocab, K) > 200 * 1024)
    return set_error(DFLASH_ERR_UNSUPPORTED, "K = %d is too large for this vocabulary", K);
  if (max_ctx < 0 || max_ctx > cache->cap)
    return set_error(DFLASH_ERR_INVALID_ARG, "max_ctx must be in [0, cache->cap]");
  if (!anchor || !ctx_len || !topk_ids || !topk_logp)
    return set_error(DFLASH_ERR_INVALID_ARG, "null anchor/ctx_len/topk output");
  for (int l = 0; l < d.n_layers; ++l)
    if (!cache->k[l] || !cache->v[l]) return set_error(DFLASH_ERR_INVALID_ARG, "null cache layer %d", l);
  return DFLASH_OK;
}

// Steps a3 - a6.  `pre`: GEMM steps over the same n_req * L activation rows
// that run in the first GEMM launch, ahead of layer 0's QKV projection.
static dflash_status draft_impl(const dflash_model* model, const dflash_cache* cache, int n_req,
                         const int32_t* anchor, const int32_t* ctx_len, int max_ctx, int L, int K,
                         const SampleSpec& smp, int32_t* topk_ids, float* topk_logp,
                         float* logits, const CallCtx& c, const Step* pre, int n_pre) {
  const dflash_dims& d = model->dims;
  const WsLayout& W = c.L;
  const int R = n_req * L;
  const int D = L - 1;
  const int hd = d.head_dim;
  const int qd = d.n_q * hd;
  const int qkv_dim = (d.n_q + 2 * d.n_kv) * hd;
  float* x = reinterpret_cast<float*>(c.ws + W.x);
  void* xn = c.ws + W.xn;
  float* ssq = reinterpret_cast<float*>(c.ws + W.ssq);
  void* qkv = c.ws + W.qkv;
  void* ao = c.ws + W.attn_o;
  void* hbuf = c.ws + W.h;
  float* lg = logits ? logits : reinterpret_cast<float*>(c.ws + W.logits);
  float2* rope = reinterpret_cast<float2*>(c.ws + W.rope_blk);

  BlockPrologueLaunch pa{model->bf16, model->w.embed, model->w.attn_norm[0], anchor, ctx_len,
                         n_req, L, d.d, d.vocab, d.mask_id, hd, model->freqs, x, xn, ssq, rope,
                         c.status};
  launch_block_prologue(pa, c.st);
  dflash_status st = check_launch("block prologue");
  if (st) return st;

  // attention decomposition: the last chunk also takes the block keys, so
  // there is at least one chunk even without context
  int chunk = attn_chunk(max_ctx > 0 ? max_ctx : 1, d.n_kv, n_req);
  int n_chunks = max_ctx > 0 ? (max_ctx + chunk - 1) / chunk : 1;
  if (n_chunks > W.attn_chunks_cap) {
    chunk = ((max_ctx + W.attn_chunks_cap - 1) / W.attn_chunks_cap + 63) / 64 * 64;
    n_chunks = (max_ctx + chunk - 1) / chunk;
  }
  // With (request, KV head) pairs for half the SMs or more, the tensor-core
  // kernel (128-key tiles, one CTA per SM) takes the attention: chunks for
  // about four CTAs per SM over the grid, fewer where contexts are short.  A
  // few pairs (one request) stay on the split kernel above, whose shorter
  // per-CTA latency suits a grid of many small chunks.
  const long long kv_pairs = (long long)n_req * d.n_kv;
  const bool attn_tc = model->bf16 && hd == 128 && d.n_q / d.n_kv <= 4 && L <= 32 &&
                       2 * kv_pairs >= num_sms();
  if (attn_tc) {
    long long nc = (4LL * num_sms() + kv_pairs - 1) / kv_pairs;
    if (nc > W.attn_chunks_cap) nc = W.attn_chunks_cap;
    const int mc = max_ctx > 0 ? max_ctx : 1;
    chunk = static_cast<int>((mc + nc - 1) / nc + 127) / 128 * 128;
    n_chunks = (mc + chunk - 1) / chunk;
  }

  // GEMM steps of the pass.  A chain runs the dependent GEMMs between two
  // attention calls in one launch: [QKV_0], attention_0, [O_0, gate/up_0,
  // down_0, QKV_1], attention_1, ..., [O_n-1, gate/up_n-1, down_n-1, LM head].
  auto qkv_step = [&](int l) {
    EpiParams eq = epi_base(*model, R, qkv_dim);
    eq.kind = EPI_QKV;
    eq.ssq_in = ssq;
    eq.out = qkv;
    eq.ldo = qkv_dim;
    eq.rope = rope;
    eq.rope_cols = (d.n_q + d.n_kv) * hd;
    return Step{&model->tm_qkv[l], model->w.w_qkv[l], xn, d.d, qkv_dim, d.d, eq};
  };
  // With one 16-row tile and K <= 8 the log-softmax / top-K (or the sampling)
  // rides in the LM head's epilogue and is merged inside the same launch; the
  // logits are then stored only if the caller asked for them.  Otherwise the
  // logits are stored and a top-K pass follows (the two-pass large-K one for
  // K > 8 without sampling).
  const bool sampling = smp.inv_t > 0.f;
  const bool fused_topk = model->bf16 && tc_row_tile(R) == 16 && K <= 8;
  auto lm_step = [&]() {
    EpiParams el = epi_base(*model, R, d.vocab);
    el.kind = EPI_LOGITS;
    el.ssq_in = ssq;
    el.logits = fused_topk ? logits : lg;
    el.L = L;
    el.tk_part = fused_topk ? reinterpret_cast<float*>(c.ws + W.tkpart) : nullptr;
    el.tk_K = K;
    el.tk_ids = fused_topk ? topk_ids : nullptr;
    el.tk_logp = fused_topk ? topk_logp : nullptr;
    if (fused_topk) {
      el.tk_inv_t = smp.inv_t;
      el.tk_t = smp.t;
      el.tk_seed = smp.seed;
      el.tk_row0 = smp.row0;
    }
    return Step{&model->tm_lm, model->w.lm_head, xn, d.d, d.vocab, d.d, el};
  };
  {
    Step first[kMaxPhases];
    for (int i = 0; i < n_pre; ++i) first[i] = pre[i];
    first[n_pre] = qkv_step(0);
    st = run_chain(c, first, n_pre + 1, R);
    if (st) return st;
  }
  for (int l = 0; l < d.n_layers; ++l) {
    // attention over [context ; block]
    if (model->bf16) {
      AttnParams ap{};
      ap.qkv = static_cast<const __nv_bfloat16*>(qkv);
      ap.qkv_ld = qkv_dim;
      ap.cache_k = static_cast<const __nv_bfloat16*>(cache->k[l]);
      ap.cache_v = static_cast<const __nv_bfloat16*>(cache->v[l]);
      ap.ctx_len = ctx_len;
      ap.cap = cache->cap;
      ap.n_req = n_req;
      ap.n_q = d.n_q;
      ap.n_kv = d.n_kv;
      ap.G = d.n_q / d.n_kv;
      ap.L = L;
      ap.chunk = chunk;
      ap.n_chunks = n_chunks;
      ap.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(hd));
      ap.anchor_sees_block = d.anchor_sees_block;
      ap.part_o = reinterpret_cast<float*>(c.ws + W.apart_o);
      ap.part_ml = reinterpret_cast<float*>(c.ws + W.apart_ml);
      ap.out = static_cast<__nv_bfloat16*>(ao);
      ap.out_ld = qd;
      st = attn_tc ? launch_block_attention_tc(ap, c.counters + W.attn_arrivals, c.status, c.st)
                   : launch_attention_bf16(ap, hd, c.st);
    } else {
      AttnParamsF32 ap{};
      ap.qkv = static_cast<const float*>(qkv);
      ap.qkv_ld = qkv_dim;
      ap.cache_k = static_cast<const float*>(cache->k[l]);
      ap.cache_v = static_cast<const float*>(cache->v[l]);
      ap.ctx_len = ctx_len;
      ap.cap = cache->cap;
      ap.n_req = n_req;
      ap.n_q = d.n_q;
      ap.n_kv = d.n_kv;
      ap.L = L;
      ap.anchor_sees_block = d.anchor_sees_block;
      ap.out = static_cast<float*>(ao);
      ap.out_ld = qd;
      st = launch_attention_f32(ap, hd, c.st);
    }
    if (st) return st;
    // x += o . W_o^T ; xn = x * g_mlp
    EpiParams eo = epi_base(*model, R, d.d);
    eo.kind = EPI_RESID;
    eo.ssq_in = nullptr;
    eo.x = x;
    eo.xn = xn;
    eo.gain = model->w.mlp_norm[l];
    eo.ssq_out = ssq;
    // h = silu(g) * u
    EpiParams eg = epi_base(*model, R, 2 * d.d_ff);
    eg.kind = EPI_SWIGLU;
    eg.ssq_in = ssq;
    eg.out = hbuf;
    eg.ldo = d.d_ff;
    // x += h . W_down^T ; xn = x * g_next
    EpiParams ed = epi_base(*model, R, d.d);
    ed.kind = EPI_RESID;
    ed.ssq_in = nullptr;
    ed.x = x;
    ed.xn = xn;
    ed.gain = (l + 1 < d.n_layers) ? model->w.attn_norm[l + 1] : model->w.final_norm;
    ed.ssq_out = ssq;
    // then the next layer's Q, K, V, or the LM head on the mask rows
    const Step chain[4] = {
        {&model->tm_o[l], model->w.wo[l], ao, qd, d.d, qd, eo},
        {&model->tm_gu[l], model->w.w_gate_up[l], xn, d.d, 2 * d.d_ff, d.d, eg},
        {&model->tm_down[l], model->w.w_down[l], hbuf, d.d_ff, d.d, d.d_ff, ed},
        (l + 1 < d.n_layers) ? qkv_step(l + 1) : lm_step()};
    st = run_chain(c, chain, 4, R);
    if (st) return st;
  }
  // log-softmax + top-K
  if (fused_topk) return DFLASH_OK;   // merged inside the LM-head chain
  TopkLaunch tk{};
  tk.logits = lg;
  tk.rows = n_req * D;
  tk.vocab = d.vocab;
  tk.ld = d.vocab;
  tk.dtype = DFLASH_F32;
  tk.K = K;
  tk.splits = topk_splits(tk.rows, d.vocab);
  tk.part = reinterpret_cast<float*>(c.ws + W.tpart);
  tk.counters = c.counters + gemm_counter_ints();
  tk.ids = topk_ids;
  tk.logp = topk_logp;
  tk.inv_t = smp.inv_t;
  tk.t = smp.t;
  tk.seed = smp.seed;
  tk.row0 = smp.row0;
  tk.status = c.status;
  if (K > 8 && !sampling) {
    st = launch_topk_large(tk, c.ws + W.tpart, c.st);
    if (st) return st;
  } else {
    launch_topk(tk, c.st);
  }
  return check_launch("top-K");
}

dflash_status dflash_draft_block(const dflash_model* model, const dflash_cache* cache, int n_req,
                                 const int32_t* anchor, const int32_t* ctx_len, int max_ctx,
                                 int L, int K, const dflash_sampling* sampling,
                                 int32_t* topk_ids, float* topk_logp, float* logits, void* ws,
                                 size_t ws_bytes, void* stream) {
  dflash_status st = check_draft(model, cache, n_req, anchor, ctx_len, max_ctx, L, K, topk_ids,
                                 topk_logp);
  if (st) return st;
  SampleSpec smp;
  st = parse_sampling(sampling, &smp);
  if (st) return st;
  if (smp.inv_t > 0.f && K > 32)
    return set_error(DFLASH_ERR_UNSUPPORTED, "sampling draws at most 32 tokens per position");
  const WsLayout W = ws_layout(*model, n_req, 0, L, K);
  if (!ws || ws_bytes < W.f)
    return set_error(DFLASH_ERR_WORKSPACE, "draft workspace needs %zu bytes, got %zu", W.f,
                     ws_bytes);
  CallCtx c{model, static_cast<char*>(ws), W, static_cast<cudaStream_t>(stream),
            static_cast<int*>(ws), reinterpret_cast<int*>(static_cast<char*>(ws) + W.counters)};
  return draft_impl(model, cache, n_req, anchor, ctx_len, max_ctx, L, K, smp, topk_ids,
                    topk_logp, logits, c, nullptr, 0);
}

dflash_status dflash_draft_cycle(const dflash_model* model, const dflash_cache* cache, int n_req,
                                 int n_rows, const int32_t* row_off, const int32_t* pos0,
                                 const void* feats, const int32_t* anchor,
                                 const int32_t* ctx_len, int max_ctx, int L, int K,
                                 const dflash_sampling* sampling, int32_t* topk_ids,
                                 float* topk_logp, float* logits, void* ws, size_t ws_bytes,
                                 void* stream) {
  dflash_status st = check_inject(model, cache, n_req, n_rows, row_off, pos0, feats);
  if (st) return st;
  st = check_draft(model, cache, n_req, anchor, ctx_len, max_ctx, L, K, topk_ids, topk_logp);
  if (st) return st;
  SampleSpec smp;
  st = parse_sampling(sampling, &smp);
  if (st) return st;
  if (smp.inv_t > 0.f && K > 32)
    return set_error(DFLASH_ERR_UNSUPPORTED, "sampling draws at most 32 tokens per position");
  const WsLayout W = ws_layout(*model, n_req, n_rows, L, K);
  if (!ws || ws_bytes < W.total)
    return set_error(DFLASH_ERR_WORKSPACE, "cycle workspace needs %zu bytes, got %zu", W.total,
                     ws_bytes);
  CallCtx c{model, static_cast<char*>(ws), W, static_cast<cudaStream_t>(stream),
            static_cast<int*>(ws), reinterpret_cast<int*>(static_cast<char*>(ws) + W.counters)};
  if (n_rows == 0)
    return draft_impl(model, cache, n_req, anchor, ctx_len, max_ctx, L, K, smp, topk_ids,
                      topk_logp, logits, c, nullptr, 0);
  Step inj[2];
  st = inject_steps(model, cache, n_req, n_rows, row_off, pos0, feats, c, inj);
  if (st) return st;
  // One GEMM launch for the injection and layer 0's QKV when they share the
  // activation row count (a chain runs over one row count).
  if (model->bf16 && n_rows == n_req * L)
    return draft_impl(model, cache, n_req, anchor, ctx_len, max_ctx, L, K, smp, topk_ids,
                      topk_logp, logits, c, inj, 2);
  st = run_chain(c, inj, 2, n_rows);
  if (st) return st;
  return draft_impl(model, cache, n_req, anchor, ctx_len, max_ctx, L, K, smp, topk_ids,
                    topk_logp, logits, c, nullptr, 0);
}

size_t dflash_linear_workspace_bytes(int M, int N, int K) {
  if (M < 0 || N <= 0 || K <= 0 || K % 64 || N % 128) return 0;
  const TcPlan pl = tc_plan(M > 0 ? M : 1, N, K, num_sms());
  const int n_counters = gemm_counter_ints() > 4096 ? gemm_counter_ints() : 4096;
  return 256 + align_up(sizeof(int) * n_counters, 256) + align_up(pl.part_bytes, 256);
}

dflash_status dflash_linear_bf16(int M, int N, int K, const void* X, const void* W, float* Y,
                                 void* ws, size_t ws_bytes, void* stream) {
  if (M < 0 || N <= 0 || K <= 0 || K % 64 || N % 128)
    return set_error(DFLASH_ERR_INVALID_ARG, "need M >= 0, K %% 64 == 0, N %% 128 == 0");
  if (M == 0) return DFLASH_OK;
  if (!X || !W || !Y || !aligned16(X) || !aligned16(W))
    return set_error(DFLASH_ERR_INVALID_ARG, "X, W, Y must be non-null, X and W 16-byte aligned");
  const size_t need = dflash_linear_workspace_bytes(M, N, K);
  if (!ws || ws_bytes < need)
    return set_error(DFLASH_ERR_WORKSPACE, "linear workspace needs %zu bytes, got %zu", need,
                     ws_bytes);
  CUtensorMap tmW;
  if (!encode_kmajor_map(&tmW, W, N, K, K, 128))
    return set_error(DFLASH_ERR_CUDA, "cannot encode TMA descriptors");
  EpiParams e{};
  e.kind = EPI_STORE_F32;
  e.M_rows = M;
  e.N_feat = N;
  e.logits = Y;
  e.ldo = N;
  char* w = static_cast<char*>(ws);
  const int n_counters = gemm_counter_ints() > 4096 ? gemm_counter_ints() : 4096;
  int* counters = reinterpret_cast<int*>(w + 256);
  float* part = reinterpret_cast<float*>(w + 256 + align_up(sizeof(int) * n_counters, 256));
  const GemmPhase ph{&tmW, X, K, N, K, e};
  return launch_gemm_chain(&ph, 1, M, part, counters, static_cast<int*>(ws),
                           static_cast<cudaStream_t>(stream));
}

}  // extern "C"
