"""GPU parity of KV injection (steps a1-a2) and the drafter block pass with LM
head and top-K (steps a3-a6), through the C ABI, against the oracle on the
same seeded inputs.

Tolerances (from the pages' bar and the arithmetic): logits per row
max|l_gpu - l_ora| / max|l_ora| <= 2e-2 for bf16 models, 1e-4 for fp32;
injected cache entries the same per (layer, position).

Top-K, two checks.  (1) On identical logits: the oracle's log-softmax/top-K
of the fp32 logits the GPU itself returned must give the GPU's ids bit for
bit (ties to the smaller id) and its log-probs within 1e-5 nats.  The fused
LM-head fold ranks exactly the values it stores, so this holds the in-path
kernel to the exact bar.  (2) End to end: against the oracle's own logits
the sets may differ only by tokens whose oracle logit lies within delta of
the oracle's K-th logit, delta = 2 * (that row's max logit error) + 1e-3
nats, since each side decides on its own logits."""
import dataclasses

import numpy as np
import pytest
import torch

from block_diffusion_speculative_kv_gb300 import synth
from block_diffusion_speculative_kv_gb300.configs import WORKLOADS, DrafterShape
from block_diffusion_speculative_kv_gb300.drafter import Drafter
from oracle import drafter as od

pytestmark = pytest.mark.gpu

DEV = "cuda"


class F64:
    """Lazy float64 view of a torch tensor (bf16 has no NumPy dtype)."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, idx):
        return self.t[idx].float().cpu().numpy().astype(np.float64)

    def __array__(self, dtype=None, copy=None):
        return self.t.float().cpu().numpy().astype(np.float64)


def oracle_weights(w):
    out = {}
    for k, v in w.items():
        out[k] = [F64(t) for t in v] if isinstance(v, list) else F64(v)
    return out


def oracle_dims(s: DrafterShape):
    return dict(n_layers=s.n_layers, d=s.d, n_q=s.n_q, n_kv=s.n_kv, head_dim=s.head_dim,
                vocab=s.vocab, mask_id=s.mask_id, rope_theta=s.rope_theta, rms_eps=s.rms_eps)


def tol(s: DrafterShape):
    return 1e-4 if s.dtype == "fp32" else 2e-2


def _i32(a):
    return torch.as_tensor(np.asarray(a, dtype=np.int32), device=DEV)


# ---------------------------------------------------------------------------
# injection
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("wid,rows_per_req,pos0", [
    (0, [64], [0]),                   # fp32: the whole context in one call
    (0, [5, 3], [10, 60]),            # fp32: two requests, ragged
    (1, [16], [2032]),                # 4B shape: one cycle's worth at the tail
    (1, [7, 16, 1], [0, 100, 2047]),  # ragged rows, last slot of the cache
    # 256-row tiles (a batch's injection): 320 rows over 20 requests, and 700
    # rows in three tiles (the last ragged), split tiles finished by all their
    # contributors
    (1, [16] * 20, [97 * i % 2000 for i in range(20)]),
    (1, [100, 250, 350], [0, 500, 1600]),
])
def test_inject_matches_oracle(wid, rows_per_req, pos0):
    wl = WORKLOADS[wid]
    s = wl.shape
    n_req = len(rows_per_req)
    w = synth.drafter_weights(s, wl.seed, device=DEV)
    if wid == 0:
        w.update(synth.random_gains(s, wl.seed, device=DEV))
    n_rows = sum(rows_per_req)
    dr = Drafter(s, w, n_req=n_req, cap=wl.cap, max_inject_rows=n_rows, L=wl.L, K=wl.K)
    feats = synth.features(n_rows, s, wl.seed, device=DEV)
    row_off = np.concatenate([[0], np.cumsum(rows_per_req)])
    dr.inject_kv(feats, _i32(row_off), _i32(pos0))
    torch.cuda.synchronize()
    assert dr.read_status() == 0
    ow = oracle_weights(w)
    f = od.fuse_features(F64(feats), ow["w_proj"])
    for r in range(n_req):
        rows = slice(row_off[r], row_off[r + 1])
        pos = pos0[r] + np.arange(rows_per_req[r])
        for l in range(s.n_layers):
            K, V = od.inject_kv(f[rows], ow["uk"][l], ow["uv"][l], pos, s.n_kv, s.head_dim,
                                s.rope_theta)
            gk = dr.cache_k[l][r][:, pos].float().cpu().numpy()
            gv = dr.cache_v[l][r][:, pos].float().cpu().numpy()
            for ref, got in ((K, gk), (V, gv)):
                err = np.max(np.abs(got - ref), axis=(0, 2)) / np.max(np.abs(ref), axis=(0, 2))
                assert np.all(err <= tol(s)), (l, float(err.max()))
        # slots outside the injected range stay untouched (zero)
        mask = np.ones(wl.cap, dtype=bool)
        mask[pos] = False
        assert torch.count_nonzero(dr.cache_k[0][r][:, torch.from_numpy(mask).to(DEV)]) == 0


# ---------------------------------------------------------------------------
# the block pass
# ---------------------------------------------------------------------------

def _check_topk_on_own_logits(gpu_logits, gpu_ids, gpu_lp, K):
    o_ids, o_lp, _ = od.logits_topk(gpu_logits, K)
    bad = np.nonzero(np.any(o_ids != gpu_ids, axis=1))[0]
    assert bad.size == 0, (bad[:4].tolist(), o_ids[bad[:1]].tolist(), gpu_ids[bad[:1]].tolist())
    assert np.max(np.abs(gpu_lp - o_lp)) <= 1e-5, float(np.max(np.abs(gpu_lp - o_lp)))


def _check_logits_topk(ref_logits, gpu_logits, gpu_ids, gpu_lp, K, tolerance):
    _check_topk_on_own_logits(gpu_logits, gpu_ids, gpu_lp, K)
    rows = ref_logits.shape[0]
    err = np.max(np.abs(gpu_logits - ref_logits), axis=1)
    scale = np.max(np.abs(ref_logits), axis=1)
    assert np.all(err / scale <= tolerance), float(np.max(err / scale))
    ref_ids, ref_vals = od.topk(ref_logits, K)
    lp_ref, lse_ref = od.log_softmax(ref_logits)
    for r in range(rows):
        delta = 2.0 * err[r] + 1e-3
        kth = ref_vals[r, K - 1]
        for tok in set(ref_ids[r].tolist()) ^ set(gpu_ids[r].tolist()):
            assert abs(ref_logits[r, tok] - kth) <= delta, (r, tok)
        # the GPU's logp of its own tokens agree with the oracle's logp of them
        assert np.all(np.abs(gpu_lp[r] - lp_ref[r, gpu_ids[r]]) <= delta)
        # and are sorted
        assert np.all(np.diff(gpu_lp[r]) <= 0)


def _draft_case(wid, anchor_sees_block=True, gains=False, sample_reqs=None, K=None, ctx=None,
                tied_head=False):
    wl = WORKLOADS[wid] if isinstance(wid, int) else wid
    s = wl.shape
    K = wl.K if K is None else K
    w = synth.drafter_weights(s, wl.seed, device=DEV)
    if gains:
        w.update(synth.random_gains(s, wl.seed, device=DEV))
    if tied_head:
        w["lm_head"] = synth.tied_lm_head(s, wl.seed, device=DEV)
    ctx = synth.context_lengths(wl) if ctx is None else np.asarray(ctx, dtype=np.int32)
    max_ctx = int(ctx.max())
    dr = Drafter(s, w, n_req=wl.n_req, cap=wl.cap, max_inject_rows=0, L=wl.L, K=K,
                 anchor_sees_block=anchor_sees_block)
    ks, vs = synth.cache_prefix(s, wl.n_req, wl.cap, wl.seed, device=DEV)
    for l in range(s.n_layers):
        dr.cache_k[l].copy_(ks[l])
        dr.cache_v[l].copy_(vs[l])
    del ks, vs
    anchors = synth.anchors(wl.n_req, s.vocab, s.mask_id, wl.seed)
    D = wl.L - 1
    ids = torch.empty(wl.n_req, D, K, dtype=torch.int32, device=DEV)
    lp = torch.empty(wl.n_req, D, K, dtype=torch.float32, device=DEV)
    logits = torch.empty(wl.n_req, D, s.vocab, dtype=torch.float32, device=DEV)
    dr.draft_block(_i32(anchors), _i32(ctx), max_ctx, ids, lp, logits)
    ids2, lp2 = torch.empty_like(ids), torch.empty_like(lp)
    dr.draft_block(_i32(anchors), _i32(ctx), max_ctx, ids2, lp2)
    torch.cuda.synchronize()
    assert dr.read_status() == 0
    assert torch.equal(ids, ids2) and torch.equal(lp, lp2), "two runs differ"
    ow = oracle_weights(w)
    dims = oracle_dims(s)
    reqs = range(wl.n_req) if sample_reqs is None else sample_reqs
    for r in reqs:
        ck = [F64(dr.cache_k[l][r]) for l in range(s.n_layers)]
        cv = [F64(dr.cache_v[l][r]) for l in range(s.n_layers)]
        ref = od.drafter_block(ow, dims, ck, cv, int(ctx[r]), int(anchors[r]), wl.L,
                               anchor_sees_block=anchor_sees_block)
        _check_logits_topk(ref, logits[r].cpu().numpy().astype(np.float64),
                           ids[r].cpu().numpy(), lp[r].cpu().numpy(), K, tol(s))


def test_draft_tiny_fp32():
    _draft_case(0)


def test_draft_tiny_fp32_gains_and_anchor_isolation():
    _draft_case(0, gains=True)
    _draft_case(0, anchor_sees_block=False, gains=True)


def test_draft_qwen3_4b_shape():
    _draft_case(1)


@pytest.mark.parametrize("K", [1, 5, 16, 32])
def test_draft_qwen3_4b_shape_topk_widths(K):
    # batch 1: K <= 8 rides in the LM-head epilogue (row-per-lane fold, merged
    # in the same launch); larger K stores the logits for the two-pass top-K
    _draft_case(1, K=K)


def test_draft_qwen3_4b_shape_large_k():
    # K = 256 (Lemma 1's exact mode at B = 256): logits stored, then the
    # two-pass large-K top-K
    _draft_case(1, K=256)


def test_draft_qwen3_4b_shape_anchor_isolated():
    # the anchor row sees no other block position (tensor-core attention mask)
    _draft_case(1, anchor_sees_block=False)


def test_draft_qwen3_8b_shape_long_context():
    _draft_case(2)


@pytest.mark.parametrize("wid,ctx", [
    (1, [0]),      # no context at all: the block attends to itself only
    (1, [37]),     # a context shorter than one 64-key attention tile
    (0, [0]),      # the fp32 model without context
    (0, [5]),
])
def test_draft_empty_and_short_context(wid, ctx):
    _draft_case(wid, ctx=ctx)


@pytest.mark.parametrize("K", [8, 5])
def test_draft_fused_topk_exact_ties(K):
    # a sparse power-of-two LM head: equal logits recur, bit for bit, at ids
    # spread over every CTA's vocabulary range, so the fold's tie-break by id
    # and its cross-CTA merges decide the top-K
    _draft_case(1, K=K, tied_head=True)


def test_draft_batched_ragged_sampled():
    # 32 requests with contexts U[512, 8192]: the shortest, the longest and one more
    wl = WORKLOADS[3]
    ctx = synth.context_lengths(wl)
    pick = sorted({int(np.argmin(ctx)), int(np.argmax(ctx)), 7})
    _draft_case(3, sample_reqs=pick)


@pytest.mark.parametrize("anchor_sees_block,pick", [
    (True, [0, 1, 3, 5, 6, 11]),
    (False, [0, 4, 10]),
])
def test_draft_batched_tensor_core_attention_edges(anchor_sees_block, pick):
    # 12 requests x 8 KV heads take the batched attention path (tcgen05,
    # 128-key tiles; on 152 SMs six chunks of 384 keys for a 2048-key maximum,
    # the block keys in the chunk holding each request's context end, the last
    # chunk to finish merging the partials).  Contexts: none, inside the first
    # tile, at and around tile and chunk boundaries, and the whole cache.
    wl = dataclasses.replace(WORKLOADS[1], name="qwen3-4b-drafter-b12", n_req=12)
    ctx = [0, 1, 127, 128, 129, 383, 384, 385, 768, 1000, 2047, 2048]
    _draft_case(wl, ctx=ctx, anchor_sees_block=anchor_sees_block, sample_reqs=pick)


# ---------------------------------------------------------------------------
# inject + draft as one call
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("wid,rows_per_req", [
    (1, None),      # n_rows == n_req * L: the injection shares the first GEMM launch
    (1, [5]),       # other row counts: the two steps run one after the other
    (0, None),      # fp32 model
])
def test_draft_cycle_equals_inject_then_draft(wid, rows_per_req):
    wl = WORKLOADS[wid]
    s = wl.shape
    n_req = wl.n_req
    if rows_per_req is None:
        rows_per_req = [wl.L] * n_req
    w = synth.drafter_weights(s, wl.seed, device=DEV)
    ctx = synth.context_lengths(wl)
    max_ctx = int(ctx.max())
    n_rows = sum(rows_per_req)
    dr = Drafter(s, w, n_req=n_req, cap=wl.cap, max_inject_rows=n_rows, L=wl.L, K=wl.K)
    ks, vs = synth.cache_prefix(s, n_req, wl.cap, wl.seed, device=DEV)
    feats = synth.features(n_rows, s, wl.seed, stream=7, device=DEV)
    row_off = np.concatenate([[0], np.cumsum(rows_per_req)])
    pos0 = ctx - np.asarray(rows_per_req)          # the newest positions of each context
    anchors = _i32(synth.anchors(n_req, s.vocab, s.mask_id, wl.seed))
    D = wl.L - 1
    outs = []
    for fused in (False, True):
        for l in range(s.n_layers):
            dr.cache_k[l].copy_(ks[l])
            dr.cache_v[l].copy_(vs[l])
        ids = torch.empty(n_req, D, wl.K, dtype=torch.int32, device=DEV)
        lp = torch.empty(n_req, D, wl.K, dtype=torch.float32, device=DEV)
        if fused:
            dr.draft_cycle(feats, _i32(row_off), _i32(pos0), anchors, _i32(ctx), max_ctx, ids, lp)
        else:
            dr.inject_kv(feats, _i32(row_off), _i32(pos0))
            dr.draft_block(anchors, _i32(ctx), max_ctx, ids, lp)
        torch.cuda.synchronize()
        assert dr.read_status() == 0
        outs.append((ids, lp, [c.clone() for c in dr.cache_k], [c.clone() for c in dr.cache_v]))
    (i0, l0, k0, v0), (i1, l1, k1, v1) = outs
    assert torch.equal(i0, i1)
    assert torch.equal(l0, l1)
    for a, b in zip(k0 + v0, k1 + v1):
        assert torch.equal(a, b)
