"""Failure detection on the GPU without a fault: the tensor-core GEMM's
bounded waits are made to run out, and the call must end, record
DFLASH_ERR_TIMEOUT in the workspace status word, and leave the context
usable; after dflash_workspace_init the same call is correct again.

The waits run out because the workspace's wait limit is set to 1 us, far
below what any CTA needs: its accumulator is ready only after its share of the
weights (several hundred KB per CTA at these shapes) has streamed in, so every
CTA's epilogue wait expires.  Nothing is left waiting: every wait is bounded,
and after giving up each CTA waits (up to 2 s) only for its own copies and
MMAs in flight, frees its tensor memory and returns."""
import numpy as np
import pytest
import torch

from block_diffusion_speculative_kv_gb300 import binding as bd
from block_diffusion_speculative_kv_gb300 import synth
from block_diffusion_speculative_kv_gb300.configs import WORKLOADS
from block_diffusion_speculative_kv_gb300.drafter import Drafter
from oracle import drafter as od

pytestmark = pytest.mark.gpu

TIMEOUT = 5
LIMIT_NS = 1000


def test_linear_wait_runs_out_then_recovers():
    M, N, K = 16, 4096, 4096
    g = torch.Generator(device="cuda").manual_seed(3)
    X = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g, device="cuda") / K ** 0.5).to(torch.bfloat16)
    ws = torch.zeros(bd.linear_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    Y_ok = torch.empty(M, N, device="cuda")
    bd.linear_bf16(X, W, Y_ok, ws)
    torch.cuda.synchronize()
    assert bd.read_status(ws) == 0

    bd.workspace_set_wait_limit(ws, LIMIT_NS)
    Y = torch.empty(M, N, device="cuda")
    bd.linear_bf16(X, W, Y, ws)
    torch.cuda.synchronize()
    assert bd.read_status(ws) == TIMEOUT

    # the context is intact: an ordinary operation still runs
    assert float((torch.ones(8, device="cuda") * 2).sum()) == 16.0
    bd.workspace_init(ws)                      # also restores the default limit
    for _ in range(2):
        Y2 = torch.full((M, N), float("nan"), device="cuda")
        bd.linear_bf16(X, W, Y2, ws)
        torch.cuda.synchronize()
        assert bd.read_status(ws) == 0
        assert torch.equal(Y2, Y_ok)
    x = X.double().cpu().numpy()
    w = W.double().cpu().numpy()
    err = np.abs(Y2.cpu().numpy() - x @ w.T)
    assert np.all(err <= 5e-4 * (np.abs(x) @ np.abs(w).T) + 1e-30)


def test_draft_chain_wait_runs_out_then_recovers():
    # multi-phase GEMM chains (phase counters, split tiles, the fused top-K's
    # in-launch merge) between attention launches, at the Qwen3-4B shape
    wl = WORKLOADS[1]
    s = wl.shape
    w = synth.drafter_weights(s, wl.seed, device="cuda")
    ctx = synth.context_lengths(wl)
    T = int(ctx[0])
    dr = Drafter(s, w, n_req=1, cap=wl.cap, max_inject_rows=0, L=wl.L, K=wl.K)
    ks, vs = synth.cache_prefix(s, 1, wl.cap, wl.seed, device="cuda")
    for l in range(s.n_layers):
        dr.cache_k[l].copy_(ks[l])
        dr.cache_v[l].copy_(vs[l])
    del ks, vs
    i32 = dict(dtype=torch.int32, device="cuda")
    anchor = torch.as_tensor(synth.anchors(1, s.vocab, s.mask_id, wl.seed), **i32)
    ctx_len = torch.as_tensor(ctx, **i32)
    D = wl.L - 1

    def run():
        ids = torch.full((1, D, wl.K), -1, **i32)
        lp = torch.full((1, D, wl.K), float("nan"), device="cuda")
        logits = torch.full((1, D, s.vocab), float("nan"), device="cuda")
        dr.draft_block(anchor, ctx_len, T, ids, lp, logits)
        torch.cuda.synchronize()
        return ids, lp, logits

    ids0, lp0, lg0 = run()
    assert dr.read_status() == 0

    bd.workspace_set_wait_limit(dr.ws, LIMIT_NS)
    run()
    assert dr.read_status() == TIMEOUT

    bd.workspace_init(dr.ws)
    ids1, lp1, lg1 = run()
    assert dr.read_status() == 0
    assert torch.equal(ids1, ids0) and torch.equal(lp1, lp0) and torch.equal(lg1, lg0)

    # and correct against the oracle: logits per row, top-K on its own logits
    def f64(t):
        return t.float().cpu().numpy().astype(np.float64)
    ow = {k: ([f64(t) for t in v] if isinstance(v, list) else f64(v)) for k, v in w.items()}
    dims = dict(n_layers=s.n_layers, d=s.d, n_q=s.n_q, n_kv=s.n_kv, head_dim=s.head_dim,
                vocab=s.vocab, mask_id=s.mask_id, rope_theta=s.rope_theta, rms_eps=s.rms_eps)
    ref = od.drafter_block(ow, dims, [f64(c[0]) for c in dr.cache_k],
                           [f64(c[0]) for c in dr.cache_v], T, int(anchor[0]), wl.L)
    got = f64(lg1[0])
    assert np.all(np.max(np.abs(got - ref), axis=1) / np.max(np.abs(ref), axis=1) <= 2e-2)
    o_ids, o_lp, _ = od.logits_topk(got, wl.K)
    assert np.array_equal(ids1[0].cpu().numpy(), o_ids)
    assert np.max(np.abs(lp1[0].cpu().numpy() - o_lp)) <= 1e-5


def test_set_wait_limit_rejects_small_workspace():
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(bd.DflashError) as ei:
        bd.workspace_set_wait_limit(ws, LIMIT_NS)
    assert ei.value.status == 1
