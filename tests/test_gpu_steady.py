"""GPU checks of the steady state (DFlash page, 3.4.3; DDTree page, 3.4.5):
the commit step against the oracle's commit (integer bookkeeping and copied
feature rows: bit-exact), and cycles chained on the device (draft, tree, walk,
commit, the next cycle's injection of the accepted path) run eagerly and as
replays of one captured CUDA graph, with identical results.  After every cycle
the cache slots of the accepted path hold the oracle's injection of its
feature rows (the injection bar: per position max|dK| / max|K| <= 2e-2 for
bf16), and slots past the new context are untouched."""
import numpy as np
import pytest
import torch

from block_diffusion_speculative_kv_gb300 import binding as bd
from block_diffusion_speculative_kv_gb300 import synth
from block_diffusion_speculative_kv_gb300.configs import WORKLOADS
from block_diffusion_speculative_kv_gb300.drafter import Drafter
from oracle import cycle as oc
from oracle import drafter as od

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _i32(a):
    return torch.as_tensor(np.asarray(a, dtype=np.int32), device=DEV)


@pytest.mark.parametrize("n_req,D,B,fd,dtype", [(3, 15, 64, 64, torch.bfloat16),
                                                (5, 4, 8, 20, torch.float32),
                                                (1, 15, 256, 20480, torch.bfloat16)])
def test_commit_matches_oracle(n_req, D, B, fd, dtype):
    rng = np.random.default_rng(n_req + D)
    al = rng.integers(0, D + 1, size=n_req)
    al[0] = D                                   # a full accept
    acc = np.full((n_req, D), -1)
    for r in range(n_req):
        acc[r, :al[r]] = np.sort(rng.choice(np.arange(1, B + 1), size=al[r], replace=False))
    bonus = rng.integers(0, 1000, size=n_req)
    ctx = rng.integers(0, 500, size=n_req)
    tf = torch.randn(n_req, B + 1, fd, generator=torch.Generator().manual_seed(5)).to(dtype)
    feats = torch.full((n_req * (D + 1), fd), 3.0, dtype=dtype, device=DEV)
    row_off = torch.full((n_req + 1,), -9, dtype=torch.int32, device=DEV)
    pos0 = torch.full((n_req,), -9, dtype=torch.int32, device=DEV)
    ctx_d, anchor = _i32(ctx), torch.zeros(n_req, dtype=torch.int32, device=DEV)
    bd.commit_accepted(D, tf.to(DEV), _i32(al), _i32(acc), _i32(bonus), ctx_d, anchor, row_off,
                       pos0, feats)
    torch.cuda.synchronize()
    ro, p0, rows, ctx2, an2 = oc.commit(al, acc, bonus, ctx, tf.float().numpy())
    assert np.array_equal(row_off.cpu().numpy(), ro)
    assert np.array_equal(pos0.cpu().numpy(), p0)
    assert np.array_equal(ctx_d.cpu().numpy(), ctx2)
    assert np.array_equal(anchor.cpu().numpy(), an2)
    got = feats.float().cpu().numpy()
    assert np.array_equal(got[:ro[-1]], rows)
    assert np.all(got[ro[-1]:] == 3.0)          # rows past the path are untouched


class Loop:
    """One request stream of the 4B-shaped drafter: prefilled context, then
    cycles of draft_cycle (injecting the previous accepted path) + tree + walk
    + commit, every size on the device."""

    def __init__(self, n_cycles):
        wl = WORKLOADS[1]
        s = self.s = wl.shape
        self.wl, self.L, self.D, self.B = wl, wl.L, wl.L - 1, wl.B
        self.ctx0 = 1000
        self.cap = self.ctx0 + (n_cycles + 1) * self.L
        self.w = synth.drafter_weights(s, wl.seed, device=DEV)
        self.dr = Drafter(s, self.w, n_req=1, cap=self.cap, max_inject_rows=self.ctx0, L=self.L,
                          K=wl.K)
        fd = s.n_feat * s.d_feat
        self.prefill = synth.features(self.ctx0, s, wl.seed, stream=11, device=DEV)
        self.tree_feats = synth.features(self.B + 1, s, wl.seed, stream=12,
                                         device=DEV).reshape(1, self.B + 1, fd)
        i32 = dict(dtype=torch.int32, device=DEV)
        self.feats = torch.zeros(self.L, fd, dtype=self.prefill.dtype, device=DEV)
        self.row_off = torch.zeros(2, **i32)
        self.pos0 = torch.zeros(1, **i32)
        self.ctx_len = torch.zeros(1, **i32)
        self.anchor = torch.zeros(1, **i32)
        self.ids = torch.empty(1, self.D, wl.K, **i32)
        self.lp = torch.empty(1, self.D, wl.K, dtype=torch.float32, device=DEV)
        self.tree = bd.tree_buffers(1, self.B, DEV)
        self.al = torch.empty(1, **i32)
        self.acc = torch.empty(1, self.D, **i32)
        self.bonus = torch.empty(1, **i32)

    def reset(self):
        for c in self.dr.cache_k + self.dr.cache_v:
            c.zero_()
        # the first L positions are injected by the first cycle
        self.dr.inject_kv(self.prefill[:self.ctx0 - self.L], _i32([0, self.ctx0 - self.L]),
                          _i32([0]))
        self.feats.copy_(self.prefill[self.ctx0 - self.L:])
        self.row_off.copy_(_i32([0, self.L]))
        self.pos0.copy_(_i32([self.ctx0 - self.L]))
        self.ctx_len.copy_(_i32([self.ctx0]))
        self.anchor.copy_(_i32(synth.anchors(1, self.s.vocab, self.s.mask_id, 1)))
        torch.cuda.synchronize()

    def cycle(self):
        self.dr.draft_cycle(self.feats, self.row_off, self.pos0, self.anchor, self.ctx_len,
                            self.cap, self.ids, self.lp)
        bd.ddtree_build(self.lp, self.ids, self.anchor, self.B, *self.tree)
        target = synth.target_first_child(self.tree[0], self.tree[1], self.tree[2],
                                           self.s.vocab)
        bd.ddtree_accept(self.D, self.B, self.tree[0], self.tree[1], self.tree[2], target,
                         self.al, self.acc, self.bonus)
        bd.commit_accepted(self.D, self.tree_feats, self.al, self.acc, self.bonus, self.ctx_len,
                           self.anchor, self.row_off, self.pos0, self.feats)

    def state(self):
        torch.cuda.synchronize()
        return dict(ctx=self.ctx_len.clone(), anchor=self.anchor.clone(), al=self.al.clone(),
                    acc=self.acc.clone(), ids=self.ids.clone(), lp=self.lp.clone(),
                    k=[c.clone() for c in self.dr.cache_k], v=[c.clone() for c in self.dr.cache_v])


def test_steady_state_eager_graph_and_oracle():
    n = 4
    lp = Loop(n)
    lp.reset()
    eager = []
    for _ in range(n):
        lp.cycle()
        eager.append(lp.state())
    assert lp.dr.read_status() == 0
    # the accepted paths went into the cache: check every cycle's slots
    ow_proj = lp.w["w_proj"].float().cpu().numpy().astype(np.float64)
    tf = lp.tree_feats[0].float().cpu().numpy().astype(np.float64)
    prev_ctx = lp.ctx0
    for c, st in enumerate(eager):
        a = int(st["al"][0])
        ctx = int(st["ctx"][0])
        assert ctx == prev_ctx + a + 1
        path = [0] + [int(x) for x in st["acc"][0, :a]]
        f = od.fuse_features(tf[path], ow_proj)
        pos = prev_ctx + np.arange(a + 1)
        if c + 1 < n:   # this cycle's path is injected by the next cycle
            nxt = eager[c + 1]
            for l in range(lp.s.n_layers):
                K, V = od.inject_kv(f, lp.w["uk"][l].float().cpu().numpy().astype(np.float64),
                                    lp.w["uv"][l].float().cpu().numpy().astype(np.float64), pos,
                                    lp.s.n_kv, lp.s.head_dim, lp.s.rope_theta)
                gk = nxt["k"][l][0][:, pos].float().cpu().numpy()
                gv = nxt["v"][l][0][:, pos].float().cpu().numpy()
                for ref, got in ((K, gk), (V, gv)):
                    err = np.max(np.abs(got - ref), axis=(0, 2)) / np.max(np.abs(ref), axis=(0, 2))
                    assert np.all(err <= 2e-2), (c, l, float(err.max()))
                # nothing past the context
                assert torch.count_nonzero(nxt["k"][l][0][:, ctx:]) == 0
        prev_ctx = ctx
    taus = [int(st["al"][0]) + 1 for st in eager]
    assert min(taus) >= 1 and max(taus) <= lp.D + 1
    # the same cycles as replays of one captured graph
    lp.reset()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        lp.cycle()          # warm-up outside capture (first-call attributes)
    torch.cuda.current_stream().wait_stream(side)
    lp.reset()
    with torch.cuda.graph(g):
        lp.cycle()
    lp.reset()
    for c in range(n):
        g.replay()
        st = lp.state()
        for key in ("ctx", "anchor", "al", "acc", "ids", "lp"):
            assert torch.equal(st[key], eager[c][key]), (c, key)
        for a, b in zip(st["k"] + st["v"], eager[c]["k"] + eager[c]["v"]):
            assert torch.equal(a, b), c
