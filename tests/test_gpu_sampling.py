"""GPU parity of the vanilla DFlash drafting path at temperature T (DFlash page,
3.4.4) and its chain tree (3.4.1) against the oracle, through the C ABI.

Both sides take the sampling decision in fp32 on the same logits: the
standalone pass on the given logits, the drafter on its own fp32 logits
(returned through the optional logits output, the values its LM-head
epilogue ranks).  The chosen ids must equal the oracle's, except where the
oracle's scores of the two choices lie within a few fp32 ulps of each other
(the two sides' log may differ in the last place).  The log-probabilities of
the chosen tokens must match the oracle's log-softmax within 2e-4 nats (the
logit is recovered from an fp32 score).  The chain tree is integer work:
bit-exact."""
import numpy as np
import pytest
import torch

from block_diffusion_speculative_kv_gb300 import binding as bd
from block_diffusion_speculative_kv_gb300 import synth
from block_diffusion_speculative_kv_gb300.configs import WORKLOADS
from block_diffusion_speculative_kv_gb300.drafter import Drafter
from oracle import ddtree as odt
from oracle import sampling as osm

pytestmark = pytest.mark.gpu

DEV = "cuda"
LOGQ_TOL = 2e-4


def _i32(a):
    return torch.as_tensor(np.asarray(a, dtype=np.int32), device=DEV)


def _check_draws(logits_f32, T, seed, row0, K, gpu_ids, gpu_logq):
    """logits_f32 [rows, vocab] (numpy fp32, the values both sides rank)."""
    mism = 0
    for r in range(logits_f32.shape[0]):
        s = osm.scores(logits_f32[r], T, seed, row0 + r)
        ids, lq = osm.gumbel_topk(logits_f32[r], T, seed, row0 + r, K)
        g = gpu_ids[r]
        tol = 8 * np.spacing(np.float32(np.max(np.abs(s[ids]))))
        if not np.array_equal(g, ids):
            mism += 1
            # only near-ties may differ: the ranked scores agree value by value
            assert np.all(np.abs(s[g].astype(np.float64) - s[ids].astype(np.float64)) <= tol), \
                (r, g, ids, s[g], s[ids])
        assert len(set(g.tolist())) == K
        l64 = logits_f32[r].astype(np.float64)
        m = l64.max()
        lse = m + np.log(np.sum(np.exp(l64 - m)))
        assert np.all(np.abs(gpu_logq[r] - (l64[g] - lse)) <= LOGQ_TOL), (r, gpu_logq[r])
    assert mism <= max(1, logits_f32.shape[0] // 10)


def _sample(x, T, seed, row0, K, vocab=None):
    rows = x.shape[0]
    vocab = x.shape[1] if vocab is None else vocab
    ids = torch.full((rows, K), -5, dtype=torch.int32, device=DEV)
    lq = torch.full((rows, K), 9.0, dtype=torch.float32, device=DEV)
    ws = torch.zeros(bd.topk_workspace_bytes(rows, vocab, K), dtype=torch.uint8, device=DEV)
    bd.logits_sample(x, (T, seed, row0), K, ids, lq, ws, vocab=vocab)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), lq.cpu().numpy()


@pytest.mark.parametrize("rows,vocab,ld,dtype,T,K", [
    (15, 151936, 151936, torch.float32, 1.0, 1),    # one drafted block, Qwen3 vocabulary
    (15, 151936, 151936, torch.float32, 0.5, 4),    # a draw of 4 without replacement
    (15, 151931, 152000, torch.bfloat16, 1.0, 1),   # bf16, padded rows, ragged tail
    (3, 1000, 1000, torch.float32, 0.75, 8),        # few rows: many splits per row
    (300, 5003, 5003, torch.float32, 1.0, 2),       # many rows: one CTA per row
])
def test_logits_sample_matches_oracle(rows, vocab, ld, dtype, T, K):
    g = torch.Generator().manual_seed(rows * 7 + K)
    x = (torch.randn(rows, ld, generator=g) * 3.0).to(dtype).to(DEV)
    seed, row0 = 0x1234ABCD5678, 1000
    ids, lq = _sample(x, T, seed, row0, K, vocab=vocab)
    xf = x[:, :vocab].float().cpu().numpy()
    _check_draws(xf, T, seed, row0, K, ids, lq)


def test_zero_logits_pick_the_largest_uniform_exactly():
    # with equal logits the sample is the argmax of U (G is increasing in U):
    # a check of the counter generator that no log rounding can blur
    rows, vocab = 15, 151936
    x = torch.zeros(rows, vocab, dtype=torch.float32, device=DEV)
    for seed, row0 in ((0, 0), (2 ** 63 + 12345, 7 * 2 ** 20)):
        ids, _ = _sample(x, 1.0, seed, row0, 1)
        for r in range(rows):
            u = osm.uniforms(seed, row0 + r, vocab)
            assert ids[r, 0] == int(np.argmax(u)), (seed, r)


def test_temperature_zero_is_the_plain_top_k():
    rows, vocab, K = 6, 30000, 8
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(rows, vocab, generator=g) * 2).to(DEV)
    ids_s, lq_s = _sample(x, 0.0, 99, 0, K)
    ids = torch.empty(rows, K, dtype=torch.int32, device=DEV)
    lp = torch.empty(rows, K, dtype=torch.float32, device=DEV)
    ws = torch.zeros(bd.topk_workspace_bytes(rows, vocab, K), dtype=torch.uint8, device=DEV)
    bd.logits_topk(x, K, ids, lp, ws)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ids_s)
    assert np.array_equal(lp.cpu().numpy(), lq_s)


def test_seed_and_row_offset_change_the_draw():
    rows, vocab = 15, 20000
    x = torch.zeros(rows, vocab, dtype=torch.float32, device=DEV)
    a, _ = _sample(x, 1.0, 5, 0, 1)
    b, _ = _sample(x, 1.0, 6, 0, 1)
    c, _ = _sample(x, 1.0, 5, 15, 1)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)
    # the draw of a row depends on its counter row only
    d, _ = _sample(x[1:], 1.0, 5, 1, 1)
    assert np.array_equal(a[1:], d)


def _drafter(wid, K):
    wl = WORKLOADS[wid]
    s = wl.shape
    w = synth.drafter_weights(s, wl.seed, device=DEV)
    ctx = synth.context_lengths(wl)
    dr = Drafter(s, w, n_req=wl.n_req, cap=wl.cap, max_inject_rows=0, L=wl.L, K=K)
    ks, vs = synth.cache_prefix(s, wl.n_req, wl.cap, wl.seed, device=DEV)
    for l in range(s.n_layers):
        dr.cache_k[l].copy_(ks[l])
        dr.cache_v[l].copy_(vs[l])
    anchors = _i32(synth.anchors(wl.n_req, s.vocab, s.mask_id, wl.seed))
    return wl, dr, anchors, ctx


@pytest.mark.parametrize("wid,K,T", [
    (1, 1, 1.0),    # bf16 batch 1: the draw rides in the LM-head epilogue
    (1, 4, 0.5),    # the same, 4 tokens without replacement
    (1, 12, 1.0),   # K > 8: logits stored, then the standalone sampling pass
    (0, 2, 1.0),    # fp32 model: standalone pass
])
def test_drafter_samples_match_oracle(wid, K, T):
    wl, dr, anchors, ctx = _drafter(wid, K)
    D = wl.L - 1
    n_req, vocab = wl.n_req, wl.shape.vocab
    seed, row0 = 777, 3 * n_req * D
    ids = torch.empty(n_req, D, K, dtype=torch.int32, device=DEV)
    lq = torch.empty(n_req, D, K, dtype=torch.float32, device=DEV)
    logits = torch.empty(n_req, D, vocab, dtype=torch.float32, device=DEV)
    dr.draft_block(anchors, _i32(ctx), int(ctx.max()), ids, lq, logits, sampling=(T, seed, row0))
    ids2, lq2 = torch.empty_like(ids), torch.empty_like(lq)
    dr.draft_block(anchors, _i32(ctx), int(ctx.max()), ids2, lq2, sampling=(T, seed, row0))
    torch.cuda.synchronize()
    assert dr.read_status() == 0
    # storing the logits or not does not change the draw
    assert torch.equal(ids, ids2) and torch.equal(lq, lq2)
    _check_draws(logits.reshape(n_req * D, vocab).cpu().numpy(), T, seed, row0, K,
                 ids.reshape(n_req * D, K).cpu().numpy(), lq.reshape(n_req * D, K).cpu().numpy())


def _tree_bufs(n_req, B):
    return bd.tree_buffers(n_req, B, device=DEV)


@pytest.mark.parametrize("n_req,D,K,B", [(3, 15, 4, 15), (2, 7, 1, 3), (1, 15, 8, 1024),
                                         (4, 3, 2, 0)])
def test_chain_tree_matches_oracle(n_req, D, K, B):
    rng = np.random.default_rng(n_req * 100 + B)
    topk = rng.integers(0, 151936, size=(n_req, D, K)).astype(np.int32)
    root = rng.integers(0, 151936, size=n_req).astype(np.int32)
    bufs = _tree_bufs(n_req, B)
    for t in bufs:
        t.fill_(123)          # stale values must be overwritten
    bd.chain_tree(_i32(topk), _i32(root), B, *bufs)
    torch.cuda.synchronize()
    n_nodes, tok, parent, depth, rank, mask = [t.cpu().numpy() for t in bufs]
    for r in range(n_req):
        ref = osm.chain_tree(int(root[r]), topk[r, :, 0].tolist(), B)
        assert n_nodes[r] == ref["n_nodes"]
        for key, got in (("tok", tok), ("parent", parent), ("depth", depth), ("rank", rank)):
            assert np.array_equal(got[r], ref[key]), key
        assert np.array_equal(mask[r].view(np.uint32), ref["mask"])


def test_sampled_chain_walk():
    # draft at T = 1 through the fused epilogue, build the chain, walk it with a
    # target that agrees with the first k drafted tokens
    wl, dr, anchors, ctx = _drafter(1, 1)
    D, n_req = wl.L - 1, wl.n_req
    ids = torch.empty(n_req, D, 1, dtype=torch.int32, device=DEV)
    lq = torch.empty(n_req, D, 1, dtype=torch.float32, device=DEV)
    dr.draft_block(anchors, _i32(ctx), int(ctx.max()), ids, lq, sampling=(1.0, 31, 0))
    B = D
    bufs = _tree_bufs(n_req, B)
    bd.chain_tree(ids, anchors, B, *bufs)
    torch.cuda.synchronize()
    n_nodes, tok, parent = bufs[0], bufs[1], bufs[2]
    drafted = ids[0, :, 0].cpu().numpy()
    for k in (0, 5, D):
        target = np.full((n_req, B + 1), -1, dtype=np.int32)
        target[0, :k] = drafted[:k]
        target[0, k] = (int(drafted[k]) + 1) % wl.shape.vocab if k < D else 42
        acc_len = torch.empty(n_req, dtype=torch.int32, device=DEV)
        accepted = torch.empty(n_req, D, dtype=torch.int32, device=DEV)
        bonus = torch.empty(n_req, dtype=torch.int32, device=DEV)
        bd.ddtree_accept(D, B, n_nodes, tok, parent, _i32(target), acc_len, accepted, bonus)
        torch.cuda.synchronize()
        ref = odt.accept_walk(tok[0].cpu().numpy(), parent[0].cpu().numpy(),
                              int(n_nodes[0]), target[0], D)
        assert int(acc_len[0]) == ref[0] == k
        assert int(bonus[0]) == ref[2] == target[0, k]
