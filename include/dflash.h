/*
 * dflash.h - C ABI of the block-diffusion speculative drafting library
 * (DFlash drafter + DDTree draft trees) for one NVIDIA GB300 (sm_103a).
 *
 * One drafter cycle is four calls, in the order the pages describe a round:
 *
 *   dflash_inject_kv    project the target's fused hidden features into every
 *                       drafter layer's KV cache
 *                       ("DFlash: Block Diffusion for Flash Speculative Decoding",
 *                       section 3.4.3, feature fusion and KV injection);
 *   dflash_draft_block  one parallel pass of the drafter over
 *                       [anchor, mask x (L-1)], LM head, log-softmax and top-K
 *                       (same page, section 3.4.4; "Accelerating Speculative
 *                       Decoding with Block Diffusion Draft Trees", section 3.4.2);
 *   ddtree_build        Algorithm 1: the best-first heap over rank tuples, with
 *                       the flattened tree, depth position ids and the ancestor
 *                       attention mask (DDTree page, sections 3.4.4-3.4.5);
 *   ddtree_accept       the verifier walk against the target's token choices
 *   dflash_tree_attention / dflash_tree_rope
 *                       the verification pass's attention over the flattened
 *                       tree (ancestor mask, depth position ids)
 *                       (DDTree page, section 3.4.5);
 *   dflash_commit_accepted
 *                       the accepted path becomes the next cycle's injected
 *                       context (sizes stay on the device, so a whole cycle
 *                       replays as one CUDA graph).
 * dflash_draft_cycle runs the first two calls as one.  With a dflash_sampling
 * the drafter draws tokens at temperature T (vanilla DFlash), and
 * dflash_chain_tree lays the drafted block out as a chain in ddtree_build's
 * layout.  dflash_logits_topk / dflash_logits_sample run step a6 alone.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Memory: every tensor argument is a DEVICE pointer unless marked "host".
 *   The caller owns all memory.  The library never allocates device memory;
 *   scratch space comes from a caller-provided workspace (see
 *   dflash_workspace_bytes).  The only host allocation is the model handle.
 * - Layout: row-major, innermost index last, densely packed unless a leading
 *   dimension is given.  "T" below is the model dtype: fp32 (DFLASH_F32) or
 *   bf16 (DFLASH_BF16, IEEE-754 binary32 truncated to its top 16 bits, round to
 *   nearest even when produced here).
 * - Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  Every
 *   call only enqueues work on it and returns; nothing synchronises.  Calls are
 *   capturable into a CUDA graph (no allocation, no host synchronisation).
 * - Errors: arguments are validated on the host before anything is enqueued; a
 *   rejected call returns non-zero, enqueues nothing and leaves outputs
 *   untouched.  DFLASH_ERR_CUDA means a launch failed (the CUDA error string is
 *   in dflash_last_error()).  Problems found on the device (a bounded wait that
 *   ran out) are recorded in the workspace status word, read with
 *   dflash_read_status.  dflash_last_error() returns a thread-local message for
 *   the last non-OK status of the calling thread.
 * - Concurrency: calls that share a workspace must be ordered on one stream.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DFLASH_ABI_VERSION 2
#define DFLASH_MAX_LAYERS 16

typedef enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = 1,   /* null pointer, bad size, unsupported shape    */
  DFLASH_ERR_UNSUPPORTED = 2,   /* valid request the library does not implement */
  DFLASH_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required   */
  DFLASH_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed            */
  DFLASH_ERR_TIMEOUT = 5        /* device-side bounded wait expired (status word)*/
} dflash_status;

typedef enum { DFLASH_F32 = 0, DFLASH_BF16 = 1 } dflash_dtype;

/* Temperature of the drafted tokens (DFlash page, 3.4.4: argmax at temperature
 * 0, a sample from softmax(logits) at temperature 1).  A top-K pass given a
 * dflash_sampling with temperature T > 0 ranks, instead of the logits l_v, the
 * Gumbel scores s_v = l_v * f32(1/T) + G_v (an fp32 multiply then an fp32
 * add), G_v = -log(-log U_v) in fp32, and keeps the K best (score desc, token
 * id asc): entry 0 is a sample from softmax(l / T), the K entries a draw
 * without replacement.  U_v: the SplitMix64 generator (Steele, Lea, Flood,
 * 2014) seeded with `seed`; element v of counter row c takes output number
 * (c << 32 | v) + 1 and U = (its top 23 bits + 1/2) / 2^23.  Output row r of a
 * call uses counter row row_offset + r.  The log-probabilities written are
 * log q(token) = logit - logsumexp(row), the logit recovered from the score as
 * (s - G) * T (exact to the fp32 rounding of s).  A NULL pointer or T == 0
 * selects the plain top-K (ranked by logit).  Requires T == 0 or
 * 1e-6 <= T <= 1e6. */
typedef struct dflash_sampling {
  float temperature;
  uint64_t seed;
  int64_t row_offset;
} dflash_sampling;

/* Drafter shape and the readings the pages leave open.
 * - Pre-norm RMSNorm: x / sqrt(mean(x^2) + rms_eps) * gain, before attention,
 *   before the MLP and before the LM head; SwiGLU MLP; no biases.
 * - Rotary embedding (rotate-half, base rope_theta) on queries and keys at
 *   absolute positions: cache slot t has position t, block row j of a request
 *   whose context holds ctx_len entries has position ctx_len + j.
 * - anchor_sees_block = 1: every block row attends to the whole context and the
 *   whole block (bidirectional block).  0: the anchor row attends only to the
 *   context and itself, as the DFlash page's attention bullet list states.
 * Supported: 1 <= n_layers <= 16; head_dim in {64, 128}; n_q % n_kv == 0;
 * bf16 models need d, d_feat*n_feat, n_q*head_dim and d_ff multiples of 128
 * (every GEMM reduction dimension a multiple of 64). */
typedef struct {
  int n_layers;
  int d;            /* hidden size; also the fused feature size            */
  int n_q;          /* query heads                                         */
  int n_kv;         /* key/value heads                                     */
  int head_dim;
  int d_ff;         /* SwiGLU inner size                                   */
  int vocab;
  int n_feat;       /* target layers whose hidden states are concatenated  */
  int d_feat;       /* target hidden size                                  */
  int dtype;        /* dflash_dtype                                        */
  float rope_theta;
  float rms_eps;
  int mask_id;      /* token id of the mask token, 0 <= mask_id < vocab    */
  int anchor_sees_block;
} dflash_dims;

/* Device pointers to the drafter weights (type T unless noted), in the packed
 * layouts the kernels stream.  [out][in] matrices are the usual y = W x form.
 *   w_proj      [d][n_feat*d_feat]        fusion projection W_proj
 *   embed       [vocab][d]                token embedding (shared with target)
 *   lm_head     [vocab][d]                LM head (shared with target)
 *   final_norm  [d]                       gain of the norm before the LM head
 *   u_kv        [n_layers][2][n_kv*head_dim][d]
 *                                         injection projections: per layer
 *                                         U_K rows, then U_V rows
 *   per layer l < n_layers:
 *   attn_norm   [d]
 *   w_qkv       [(n_q + 2*n_kv)*head_dim][d]   rows of W_q, then W_k, then W_v
 *   wo          [d][n_q*head_dim]
 *   mlp_norm    [d]
 *   w_gate_up   [2*d_ff][d]               interleaved: row 2j = gate row j,
 *                                         row 2j+1 = up row j
 *   w_down      [d][d_ff]
 * All pointers 16-byte aligned.  The weights must stay valid and unchanged for
 * the lifetime of a dflash_model built from them. */
typedef struct {
  const void* w_proj;
  const void* embed;
  const void* lm_head;
  const void* final_norm;
  const void* u_kv;
  const void* attn_norm[DFLASH_MAX_LAYERS];
  const void* w_qkv[DFLASH_MAX_LAYERS];
  const void* wo[DFLASH_MAX_LAYERS];
  const void* mlp_norm[DFLASH_MAX_LAYERS];
  const void* w_gate_up[DFLASH_MAX_LAYERS];
  const void* w_down[DFLASH_MAX_LAYERS];
} dflash_weights;

/* The drafter's injected-context KV cache (DFlash page, 3.4.3: the projected
 * features are stored in the drafter's KV cache and reused across cycles).
 * Per layer l: k[l], v[l] are T [n_req][n_kv][cap][head_dim]; slot t of a
 * request holds the entry injected for position t (keys already rotated at t).
 * Written by dflash_inject_kv, read by dflash_draft_block. */
typedef struct {
  void* k[DFLASH_MAX_LAYERS];
  void* v[DFLASH_MAX_LAYERS];
  int n_req;
  int cap;
} dflash_cache;

/* Opaque model handle: the dims, the weight pointers and the TMA descriptors
 * built for them once.  Host memory only. */
typedef struct dflash_model dflash_model;

/* Build a model handle.  Validates dims and weight pointers (non-null, 16-byte
 * aligned).  Returns DFLASH_ERR_INVALID_ARG / DFLASH_ERR_UNSUPPORTED on a bad
 * or unsupported shape, DFLASH_ERR_CUDA if the TMA descriptors cannot be
 * encoded.  *out is set only on success; free it with dflash_model_destroy. */
dflash_status dflash_model_create(const dflash_dims* dims, const dflash_weights* weights,
                                  dflash_model** out);
void dflash_model_destroy(dflash_model* model);

/* Workspace bytes for calls on this model with at most n_req requests,
 * max_inject_rows feature rows per dflash_inject_kv call, block length L <= 16
 * and top-K K <= 1024.  The same workspace also serves dflash_logits_topk for up
 * to n_req*(L-1) rows of this model's vocabulary.  0 on invalid arguments. */
size_t dflash_workspace_bytes(const dflash_model* model, int n_req, int max_inject_rows,
                              int L, int K);

/* Zero a workspace (its status word and arrival counters).  Required once before
 * first use, and again after a call reported a device-side error. */
dflash_status dflash_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Read (synchronously) and clear the device status word of a workspace:
 * *device_status receives DFLASH_OK or the first device-side error recorded. */
dflash_status dflash_read_status(void* ws, int* device_status, void* stream);

/* Set the time limit of every bounded device-side wait of the tensor-core GEMM
 * launches that use this workspace (ring slots, the phase counters of a GEMM
 * chain, split-tile partial sums, the fused top-K's arrivals).  The pages have
 * no counterpart: this is the failure-detection hook.  limit_ns = 0 restores
 * the default of 2 s; values above 60 s also mean the default.  A wait that
 * runs out records DFLASH_ERR_TIMEOUT in the status word; the CTA then waits
 * (up to 2 s) for its own copies and MMAs in flight, frees its tensor memory
 * and returns, so the context stays usable.  The outputs of that call are
 * undefined and the workspace must go through dflash_workspace_init (which
 * also restores the default limit) before its next use.  The limit is stored
 * in the workspace header (bytes 8..15) by an asynchronous copy on `stream`.
 * Errors: DFLASH_ERR_INVALID_ARG for a null or too small workspace,
 * DFLASH_ERR_CUDA if the copy cannot be queued. */
dflash_status dflash_workspace_set_wait_limit(void* ws, size_t ws_bytes, uint64_t limit_ns,
                                              void* stream);

/* Step a1 + a2: KV injection (DFlash page, 3.4.3).
 * For each request r and each of its feature rows i (global row
 * row_off[r] + i, i < row_off[r+1] - row_off[r]):
 *   f       = W_proj * feats[row]                       (fusion, no norm)
 *   K_l,pos = RoPE(U_K,l f, pos),  V_l,pos = U_V,l f    for every layer l
 * stored at cache slot pos = pos0[r] + i of request r.
 *   row_off  int32 [n_req+1] (device) prefix offsets, row_off[0] = 0,
 *            row_off[n_req] <= n_rows; rows at or past row_off[n_req] are
 *            computed but stored nowhere (a fixed n_rows can then serve a
 *            device-side row count, as dflash_commit_accepted writes it)
 *   pos0     int32 [n_req]   (device) first cache slot written per request;
 *            pos0[r] + rows of r must not exceed cache->cap (not checked on
 *            the device: the caller guarantees it)
 *   feats    T [n_rows][n_feat*d_feat] (device)
 * n_rows may be 0 (nothing is enqueued).  Overwrites only the addressed slots. */
dflash_status dflash_inject_kv(const dflash_model* model, const dflash_cache* cache,
                               int n_req, int n_rows, const int32_t* row_off,
                               const int32_t* pos0, const void* feats,
                               void* ws, size_t ws_bytes, void* stream);

/* Steps a3 - a6: one drafter pass over the block [anchor, mask x (L-1)] of each
 * request, then per-position log-softmax and top-K (DFlash page, 3.4.4; DDTree
 * page, 3.4.2: q_i = softmax(l_i)), or, with `sampling` at T > 0, the Gumbel
 * draw of dflash_sampling (output row r = request * (L-1) + position - 1).
 *   anchor    int32 [n_req] (device) the bonus token of each request
 *   ctx_len   int32 [n_req] (device) context entries of each request in the
 *             cache, 0 <= ctx_len[r] <= max_ctx <= cache->cap
 *   max_ctx   host bound on ctx_len used to size the attention grid
 *   L         block length, 2 <= L <= 16; D = L-1 draft positions
 *   K         1 <= K <= 1024 (and K <= vocab; with sampling K <= 32).  At
 *             batch 1 (n_req * L <= 16) and K <= 8 on bf16 models the top-K
 *             rides in the LM head's epilogue; otherwise the logits are
 *             stored in the workspace and a top-K pass follows
 *   topk_ids  int32 [n_req][L-1][K] (device) out: token ids by (logit desc,
 *             id asc)
 *   topk_logp fp32  [n_req][L-1][K] (device) out: logit - logsumexp(row)
 *   logits    fp32  [n_req][L-1][vocab] (device) out, optional (NULL skips)
 */
dflash_status dflash_draft_block(const dflash_model* model, const dflash_cache* cache,
                                 int n_req, const int32_t* anchor, const int32_t* ctx_len,
                                 int max_ctx, int L, int K, const dflash_sampling* sampling,
                                 int32_t* topk_ids, float* topk_logp, float* logits,
                                 void* ws, size_t ws_bytes, void* stream);

/* Steps a1 - a6 in one call: dflash_inject_kv(n_rows, row_off, pos0, feats)
 * followed by dflash_draft_block(anchor, ctx_len, max_ctx, L, K, ...), with the
 * same arguments, meanings and results as the two calls in sequence (the new
 * context entries are visible to the block pass).  When the injected row count
 * equals n_req * L (bf16 models), the injection's two GEMMs and the first
 * layer's QKV projection run in one GEMM launch.  The workspace must be sized
 * by dflash_workspace_bytes(model, n_req, >= n_rows, L, >= K).  n_rows may be
 * 0 (the block pass alone). */
dflash_status dflash_draft_cycle(const dflash_model* model, const dflash_cache* cache,
                                 int n_req, int n_rows, const int32_t* row_off,
                                 const int32_t* pos0, const void* feats,
                                 const int32_t* anchor, const int32_t* ctx_len, int max_ctx,
                                 int L, int K, const dflash_sampling* sampling,
                                 int32_t* topk_ids, float* topk_logp, float* logits, void* ws,
                                 size_t ws_bytes, void* stream);

/* Step a6 on its own: log-softmax + top-K over given logits rows (DDTree page,
 * 3.4.2 and Lemma 1 in 3.4.4: only the top-K tokens per depth are needed).
 *   logits  [rows][ld] of dtype (DFLASH_F32 or DFLASH_BF16), vocab <= ld
 *   ids     int32 [rows][K], logp fp32 [rows][K] (device) out; order is
 *           (logit desc, token id asc); logp = logit - logsumexp over the row
 * Requires 1 <= K <= 1024, K <= vocab, rows >= 0 (K > 8: a two-pass radix
 * select whose merge holds a row's per-chunk lists in shared memory, so K
 * times the number of 16384-logit chunks is bounded; DFLASH_ERR_UNSUPPORTED
 * beyond); ws of at least
 * dflash_topk_workspace_bytes(rows, vocab, K) bytes (zero-initialised once). */
size_t dflash_topk_workspace_bytes(int rows, int vocab, int K);
dflash_status dflash_logits_topk(int rows, int vocab, int ld, int dtype, const void* logits,
                                 int K, int32_t* ids, float* logp,
                                 void* ws, size_t ws_bytes, void* stream);

/* Step a6 with temperature sampling (DFlash page, 3.4.4; see dflash_sampling):
 * the same pass as dflash_logits_topk ranking Gumbel scores, so ids[r][0] is a
 * sample from softmax(logits[r] / T) and ids[r][0..K) a draw without
 * replacement; logq[r][k] = log q(ids[r][k]).  Same arguments, limits and
 * workspace as dflash_logits_topk; sampling NULL or T == 0 is
 * dflash_logits_topk. */
dflash_status dflash_logits_sample(int rows, int vocab, int ld, int dtype, const void* logits,
                                   const dflash_sampling* sampling, int K, int32_t* ids,
                                   float* logq, void* ws, size_t ws_bytes, void* stream);

/* Step a6 for callers that cannot provide a workspace.  The pages have no
 * counterpart: this variant exists for callers that cannot allocate device
 * memory when they run this step (a serving loop whose device memory is carved
 * up once at start-up and that must not call cudaMalloc afterwards, since that
 * can synchronise the device; a plugin host that passes inputs and outputs but
 * offers no scratch).  Same arguments and results as dflash_logits_topk,
 * without ws, for K <= 32 (always the single-pass kernel, which dflash_logits_topk
 * uses for K <= 8 only): the scratch lives in a fixed array inside the library
 * image (about 286 KB on every device that loads the library, held until the
 * process exits).  Limits: rows <= 4096 and K <= 32, larger requests return
 * DFLASH_ERR_UNSUPPORTED (rows) or DFLASH_ERR_INVALID_ARG (K).  The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress) and caches it; make that first call
 * before any stream capture.  Every call on a device shares the array and
 * clears its counters first, so calls that overlap on the GPU race: order them
 * on one stream.  Allocates nothing. */
dflash_status dflash_logits_topk_noalloc(int rows, int vocab, int ld, int dtype,
                                         const void* logits, int K, int32_t* ids, float* logp,
                                         void* stream);

/* Step a7: DDTree tree construction, Algorithm 1 (DDTree page, 3.4.4), plus the
 * flattened tree and its ancestor-only mask (3.4.5).  Per request r:
 *   topk_logp fp32 [n_req][D][K] log q of the rank-k token at depth d+1,
 *             descending along k; topk_ids int32 [n_req][D][K] its token id
 *   root_tok  int32 [n_req] the bonus token (tree root)
 * Outputs (device), width W1 = B+1 nodes per request, node 0 = root, nodes
 * 1..n in pop order:
 *   n_nodes   int32 [n_req]        n = min(B, number of prefixes available)
 *   tok       int32 [n_req][B+1]   token of the node (root: root_tok)
 *   parent    int32 [n_req][B+1]   parent node index (root: -1)
 *   depth     int32 [n_req][B+1]   depth = position id (root: 0)
 *   rank      int32 [n_req][B+1]   1-based rank of the node's token (root: 0)
 *   mask      uint32 [n_req][B+1][ceil((B+1)/32)] bit j of row i set iff node
 *             j is node i or an ancestor of it
 * Entries past node n are -1 (mask rows 0).  Scores: the candidate score is the
 * parent's score plus logp, one fp32 add; the heap pops the highest score and,
 * on equal scores, the candidate created first (each pop creates its next
 * sibling before its first child).  Requires 0 <= B <= 1024, 1 <= K <= 1024,
 * 1 <= D <= 16.  Needs no workspace. */
dflash_status ddtree_build(int n_req, int D, int K, int B, const float* topk_logp,
                           const int32_t* topk_ids, const int32_t* root_tok,
                           int32_t* n_nodes, int32_t* tok, int32_t* parent,
                           int32_t* depth, int32_t* rank, uint32_t* mask, void* stream);

/* The vanilla DFlash draft as a tree (DFlash page, 3.4.1 and 3.4.4): the chain
 * root -> drafted token of position 1 -> ... -> position D, in ddtree_build's
 * output layout so that tree attention and ddtree_accept serve both drafters.
 * Node d (1 <= d <= n = min(D, B)) holds topk_ids[r][d-1][0] (the argmax, or
 * the sample of a dflash_sampling call), parent d-1, depth d, rank 1; mask row
 * i has bits 0..i.  The walk over a chain accepts the longest prefix the
 * target agrees with.  topk_ids int32 [n_req][D][K]; outputs as ddtree_build
 * (entries past node n are -1, mask rows 0).  Requires 1 <= D <= 16,
 * 1 <= K <= 1024, 0 <= B <= 1024.  Needs no workspace. */
dflash_status dflash_chain_tree(int n_req, int D, int K, int B, const int32_t* topk_ids,
                                const int32_t* root_tok, int32_t* n_nodes, int32_t* tok,
                                int32_t* parent, int32_t* depth, int32_t* rank, uint32_t* mask,
                                void* stream);

/* Steady state between two cycles (DFlash page, 3.4.3: verified tokens are
 * injected as context and the cache is reused across cycles; DDTree page,
 * 3.4.5: only the accepted path stays).  Per request r with a = accept_len[r]
 * (ddtree_accept's outputs for this cycle's tree of budget B and depth D):
 *   the accepted path is node 0 (this cycle's anchor) then accepted[r][0..a),
 *   at positions ctx_len[r] .. ctx_len[r] + a;
 *   feats row row_off[r] + i = tree_feats[r][node i of the path], i <= a
 *   (the target's hidden features of the tree nodes, rows of feat_dim
 *   elements, tree_ld elements apart, [n_req][B+1]);
 *   row_off = prefix sums of a + 1 ([n_req+1]); pos0[r] = ctx_len[r];
 *   then ctx_len[r] += a + 1 and anchor[r] = bonus[r].
 * So a following dflash_draft_cycle with n_rows = n_req * (D+1) and these
 * row_off / pos0 / feats appends exactly the accepted path to the cache and
 * drafts from the bonus token; every size is on the device, so the cycle can
 * be captured in a CUDA graph and replayed.  The drafter's block keys and
 * values never enter the cache, so rejected positions need no rollback.
 * Requires 1 <= D <= 16, 0 <= B <= 1024, feature rows and tree_ld multiples
 * of 16 bytes, 16-byte aligned buffers; dtype DFLASH_BF16 or DFLASH_F32.  The
 * caller guarantees ctx_len[r] + D + 1 <= the cache capacity (not checked on
 * the device).  Needs no workspace. */
dflash_status dflash_commit_accepted(int n_req, int D, int B, int feat_dim, int dtype,
                                     const void* tree_feats, long long tree_ld,
                                     const int32_t* accept_len, const int32_t* accepted,
                                     const int32_t* bonus, int32_t* ctx_len, int32_t* anchor,
                                     int32_t* row_off, int32_t* pos0, void* feats, void* stream);

/* Step a8: greedy verifier walk (DDTree page, 3.4.5).  From the root, while the
 * current node has a child whose token equals target_tok[current], move to it.
 *   target_tok int32 [n_req][B+1]  the target's choice at every node
 *   accept_len int32 [n_req]       accepted draft tokens (tau = accept_len + 1)
 *   accepted   int32 [n_req][D]    accepted node indices, -1 padded
 *   bonus      int32 [n_req]       target_tok at the node where the walk stops
 * Tree arrays as produced by ddtree_build with the same B. */
dflash_status ddtree_accept(int n_req, int D, int B, const int32_t* n_nodes,
                            const int32_t* tok, const int32_t* parent,
                            const int32_t* target_tok, int32_t* accept_len,
                            int32_t* accepted, int32_t* bonus, void* stream);

/* Verification-side tree attention (DDTree page, 3.4.5): one target-model
 * attention layer over the flattened draft tree.  Per request r, tree node i
 * (0 <= i <= n_nodes[r]; node 0 is the root) attends, head h reading KV head
 * h / (n_q / n_kv), to
 *   - the request's context: cache slots t < ctx_len[r] of cache_k / cache_v
 *     ([n_req][n_kv][cap][head_dim] bf16, as the drafter's cache), and
 *   - the tree nodes j whose bit j is set in mask row i (its ancestors and
 *     itself; the mask ddtree_build writes, [n_req][B+1][ceil((B+1)/32)]),
 * with softmax(q . key / sqrt(head_dim)) weights.
 *   q    bf16 [n_req][B+1][q_ld]: query heads at columns h * head_dim,
 *        already rotated at position ctx_len + depth (dflash_tree_rope)
 *   k, v bf16 [n_req][B+1][kv_ld]: the nodes' own keys (rotated) and values,
 *        KV head g at column g * head_dim
 *   out  bf16 [n_req][B+1][out_ld]: rows of nodes past n_nodes[r] are zero
 * Requires head_dim == 128, n_q a multiple of n_kv with at most 4 query heads
 * per KV head, 0 <= B <= 1024, 0 <= ctx_len[r] <= max_ctx <= cap, strides that
 * are multiples of 8 elements and 16-byte aligned cache, q, k and v.  Device
 * pointers; ws of dflash_tree_attention_workspace_bytes(...) bytes, zeroed once
 * (dflash_workspace_init) before the first call: it holds arrival counters that
 * every call leaves at zero.  Calls sharing a workspace must not overlap. */
size_t dflash_tree_attention_workspace_bytes(int n_req, int n_q, int n_kv, int head_dim, int B,
                                             int max_ctx);
dflash_status dflash_tree_attention(int n_req, int n_q, int n_kv, int head_dim, int B,
                                    const int32_t* ctx_len, int max_ctx, int cap,
                                    const void* cache_k, const void* cache_v, const void* q,
                                    long long q_ld, const void* k, const void* v, long long kv_ld,
                                    const uint32_t* mask, const int32_t* n_nodes, void* out,
                                    long long out_ld, void* ws, size_t ws_bytes, void* stream);

/* Depth position ids of the flattened tree (DDTree page, 3.4.5): rotates heads
 * 0 .. n_heads-1 of x[r][i] (rows of ld elements, dtype DFLASH_BF16 or
 * DFLASH_F32, in place) at position ctx_len[r] + depth[r][i] with the
 * rotate-half RoPE of base theta; rows with depth < 0 (past the last node) are
 * left alone.  depth is ddtree_build's [n_req][B+1] output. */
dflash_status dflash_tree_rope(int n_req, int B, int n_heads, int head_dim, float theta,
                               const int32_t* ctx_len, const int32_t* depth, void* x,
                               long long ld, int dtype, void* stream);

/* The dense contraction every step above is built on, exposed on its own:
 * Y[M][N] = X[M][K] . W[N][K]^T with bf16 X and W and fp32 Y, on the tcgen05
 * tensor cores (the same kernel, work split and reduction the drafter's GEMMs
 * use, with a plain fp32 store as epilogue).  Requires K % 64 == 0, N % 128 ==
 * 0, X, W 16-byte aligned; M >= 0.  ws of dflash_linear_workspace_bytes(M, N,
 * K) bytes, zero-initialised once. */
size_t dflash_linear_workspace_bytes(int M, int N, int K);
dflash_status dflash_linear_bf16(int M, int N, int K, const void* X, const void* W, float* Y,
                                 void* ws, size_t ws_bytes, void* stream);

/* Launch tracing.  When a hook is set, the library calls it on the host right
 * before (phase 0) and right after (phase 1) it enqueues each kernel, with the
 * kernel's name and the stream, so a caller can record CUDA events around
 * every kernel (also while a stream is being captured into a graph).  One hook
 * per process; NULL removes it.  The hook must not call back into the library. */
typedef void (*dflash_trace_fn)(void* user, const char* kernel, int phase, void* stream);
void dflash_set_trace_hook(dflash_trace_fn fn, void* user);

/* Thread-local message for the calling thread's last non-OK status. */
const char* dflash_last_error(void);
int dflash_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
