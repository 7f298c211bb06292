"""GPU parity for step a6 (log-softmax + top-K), a7 (DDTree build) and a8 (the
verifier walk), through the C ABI, against the oracle on the same seeded
inputs.  Integer outputs must be bit-exact; log-probabilities within 1e-5."""
import numpy as np
import pytest
import torch

from block_diffusion_speculative_kv_gb300 import binding as bd
from block_diffusion_speculative_kv_gb300 import synth
from block_diffusion_speculative_kv_gb300.configs import WORKLOADS
from oracle import ddtree as odt
from oracle import drafter as od

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _gpu_topk(logits_cpu, K, vocab=None, pad=0):
    rows, V = logits_cpu.shape
    if pad:
        buf = torch.zeros(rows, V + pad, dtype=logits_cpu.dtype)
        buf[:, :V] = logits_cpu
        lg = buf.to(DEV)
    else:
        lg = logits_cpu.to(DEV)
    ids = torch.empty(rows, K, dtype=torch.int32, device=DEV)
    lp = torch.empty(rows, K, dtype=torch.float32, device=DEV)
    ws = torch.zeros(bd.topk_workspace_bytes(rows, V, K), dtype=torch.uint8, device=DEV)
    for _ in range(2):   # a second call checks the arrival counters were left at zero
        bd.logits_topk(lg, K, ids, lp, ws, vocab=V)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), lp.cpu().numpy()


def _oracle_topk(logits_cpu, K):
    x = logits_cpu.float().numpy()
    ids, lp, _ = [], [], []
    for r0 in range(0, x.shape[0], 256):
        i, l, _ = od.logits_topk(x[r0:r0 + 256], K)
        ids.append(i)
        lp.append(l)
    return np.concatenate(ids), np.concatenate(lp)


@pytest.mark.parametrize("rows,V,K,dtype,pad", [
    (5, 1000, 4, torch.float32, 0),          # several splits, fp32, vector loads
    (37, 1003, 5, torch.float32, 1),         # ragged vocab, unaligned rows (scalar loads)
    (3, 151936, 8, torch.bfloat16, 0),       # full vocabulary, many splits per row
    (64, 4099, 32, torch.bfloat16, 3),       # K = 32, unaligned bf16 rows
    (1, 9, 9, torch.float32, 0),             # K = vocab
    (300, 2048, 1, torch.bfloat16, 0),       # argmax only, one CTA per row
])
def test_topk_matches_oracle(rows, V, K, dtype, pad):
    g = torch.Generator().manual_seed(rows * 7 + K)
    x = torch.randn(rows, V, generator=g) * 2.0
    x = torch.round(x * 4) / 4            # plenty of exact ties
    x = x.to(dtype)
    ids, lp = _gpu_topk(x, K, pad=pad)
    o_ids, o_lp = _oracle_topk(x, K)
    assert np.array_equal(ids, o_ids)
    assert np.allclose(lp, o_lp, atol=1e-5, rtol=0)


@pytest.mark.parametrize("rows,V,K,dtype,pad", [
    (7, 150003, 8, torch.bfloat16, 5),       # split rows, a last piece ending mid-vector
    (500, 30011, 8, torch.bfloat16, 5),      # more rows than CTAs: second pieces per CTA
    (700, 16384, 3, torch.float32, 0),       # several rows per CTA, one stage per row
    (2, 151936, 8, torch.float32, 0),        # fp32 rows split across many CTAs
])
def test_topk_streamed_pass_matches_oracle(rows, V, K, dtype, pad):
    # K <= 8 on rows whose stride is a multiple of 16 bytes: the pass that
    # streams the logits through shared memory
    g = torch.Generator().manual_seed(rows * 13 + K)
    x = torch.randn(rows, V, generator=g) * 2.0
    x = torch.round(x * 4) / 4            # exact ties inside and across pieces
    x = x.to(dtype)
    ids, lp = _gpu_topk(x, K, pad=pad)
    o_ids, o_lp = _oracle_topk(x, K)
    assert np.array_equal(ids, o_ids)
    assert np.allclose(lp, o_lp, atol=1e-5, rtol=0)


def test_topk_masked_logits():
    # most logits -inf (masked tokens): the -inf ones never outrank a finite
    # one, and a row with fewer than K finite logits completes its list with
    # the smallest -inf ids
    rows, V, K = 6, 40000, 8
    g = torch.Generator().manual_seed(5)
    x = torch.randn(rows, V, generator=g) * 2.0
    keep = torch.rand(rows, V, generator=g) < 0.05
    keep[5] = False
    keep[5, [7, 30000, 39999]] = True     # three finite logits only
    x = torch.where(keep, x, torch.full_like(x, float("-inf")))
    ids, lp = _gpu_topk(x, K)
    o_ids, o_lp = _oracle_topk(x, K)
    assert np.array_equal(ids, o_ids)
    fin = np.isfinite(o_lp)
    assert np.array_equal(np.isfinite(lp), fin)
    assert np.allclose(lp[fin], o_lp[fin], atol=1e-5, rtol=0)


@pytest.mark.parametrize("rows,V,K,dtype,pad", [
    (15, 151936, 64, torch.float32, 0),      # one drafted block, K above the small-K kernels
    (15, 151936, 1024, torch.bfloat16, 0),   # Lemma 1's exact mode at B = 1024
    (3, 5000, 1024, torch.float32, 1),       # one chunk per row, unaligned rows
    (2, 1000, 1000, torch.float32, 0),       # K = vocab: every token, sorted
    (40, 20000, 256, torch.bfloat16, 3),     # many rows, two chunks per row
    (4, 16385, 300, torch.float32, 0),       # a last chunk of one logit
])
def test_topk_large_k_matches_oracle(rows, V, K, dtype, pad):
    g = torch.Generator().manual_seed(rows * 11 + K)
    x = torch.randn(rows, V, generator=g) * 2.0
    x = torch.round(x * 8) / 8            # exact ties across chunk boundaries
    x = x.to(dtype)
    ids, lp = _gpu_topk(x, K, pad=pad)
    o_ids, o_lp = _oracle_topk(x, K)
    assert np.array_equal(ids, o_ids)
    assert np.allclose(lp, o_lp, atol=1e-5, rtol=0)


def test_topk_stress_workload_full_size():
    """The stress workload's logits: 256 requests x 16 positions x 151936 bf16,
    N(0, 2) plus a planted +8 token per row.  Ids exact, logp within 1e-5."""
    wl = WORKLOADS[4]
    logits, planted = synth.stress_logits(wl.n_req, wl.D, wl.vocab, wl.seed, device="cpu")
    ids, lp = _gpu_topk(logits, wl.K)
    o_ids, o_lp = _oracle_topk(logits, wl.K)
    assert np.array_equal(ids, o_ids)
    assert np.allclose(lp, o_lp, atol=1e-5, rtol=0)
    # sanity of the workload itself: the planted token (+8 on an N(0, 2) draw) is
    # usually the argmax and almost always inside the top-K
    pl = planted.numpy()
    assert np.mean(ids[:, 0] == pl) > 0.8
    assert np.mean((ids == pl[:, None]).any(axis=1)) > 0.9
    # the rows are normalised: the top-K mass is below one
    assert np.all(np.exp(lp.astype(np.float64)).sum(1) <= 1.0 + 1e-5)


def _gpu_tree(lp, ids, roots, B):
    n_req = lp.shape[0]
    bufs = bd.tree_buffers(n_req, B, DEV)
    bd.ddtree_build(torch.from_numpy(lp).to(DEV), torch.from_numpy(ids).to(DEV),
                    torch.from_numpy(roots).to(DEV), B, *bufs)
    torch.cuda.synchronize()
    return [b.cpu().numpy() for b in bufs], bufs


def _check_tree(gpu, ref_list, B):
    n_nodes, tok, par, dep, rnk, mask = gpu
    for r, ref in enumerate(ref_list):
        assert n_nodes[r] == ref["n_nodes"], r
        assert np.array_equal(tok[r], ref["tok"]), r
        assert np.array_equal(par[r], ref["parent"]), r
        assert np.array_equal(dep[r], ref["depth"]), r
        assert np.array_equal(rnk[r], ref["rank"]), r
        assert np.array_equal(mask[r].view(np.uint32), ref["mask"]), r


@pytest.mark.parametrize("n_req,D,K,B,ties", [
    (1, 7, 4, 16, 0.3),        # tiny workload shape
    (1, 15, 8, 64, 0.3),       # 4B workload
    (1, 15, 8, 256, 0.3),      # 8B workload
    (32, 15, 8, 64, 0.3),      # batched workload
    (9, 16, 32, 1024, 0.5),    # largest supported budget and K
    (5, 2, 2, 10, 0.0),        # budget above the number of prefixes (6)
    (3, 4, 1, 16, 0.0),        # K = 1: a single chain
    (4, 1, 8, 16, 0.0),        # D = 1: a fan
    (2, 5, 3, 0, 0.0),         # B = 0: root only
    (7, 16, 8, 31, 1.0),       # every row coarsely quantised: many exact ties
    (1, 15, 8, 256, 0.0),      # 8B workload, no ties: the parallel construction
    (4, 15, 8, 512, 0.0),      # its largest budget
    (3, 15, 8, 300, 0.0),      # a budget that is not a power of two
    (6, 15, 8, 256, 0.05),     # a few tied rows: some requests fall back
    (2, 15, 8, 1024, 0.0),     # the largest budget, parallel construction
    (3, 16, 8, 1024, 0.1),     # the same with some tied rows
    (2, 15, 64, 64, 0.0),      # Lemma 1's exact mode K = B: parallel construction
    (3, 15, 256, 256, 0.2),    # K = B = 256: the sequential heap, ranks above 63
    (2, 16, 1024, 1024, 0.3),  # K = B = 1024 (two requests per CTA in shared memory)
    (5, 15, 1024, 1024, 0.0),
])
def test_tree_build_bit_exact(n_req, D, K, B, ties):
    lp, ids = synth.random_topk_table(n_req, D, K, 50000, seed=B + D + n_req,
                                      tie_fraction=ties)
    roots = np.arange(n_req, dtype=np.int32) + 100
    gpu, _ = _gpu_tree(lp, ids, roots, B)
    refs = [odt.build_tree(lp[r], ids[r], int(roots[r]), B) for r in range(n_req)]
    _check_tree(gpu, refs, B)


@pytest.mark.parametrize("tie_fraction", [0.0, 1.0])
def test_tree_build_deep_ranks(tie_fraction):
    # nearly flat lists (gaps 1/400 of the table's): the budget goes to wide
    # levels, so ranks run into the hundreds (K = B = 1024, Lemma 1's mode)
    lp, ids = synth.random_topk_table(2, 4, 1024, 151936, seed=5, tie_fraction=tie_fraction)
    lp = (lp - lp[:, :, :1]) / 400.0 + lp[:, :, :1]
    lp = np.ascontiguousarray(lp.astype(np.float32))
    roots = np.array([7, 8], dtype=np.int32)
    gpu, _ = _gpu_tree(lp, ids, roots, 1024)
    refs = [odt.build_tree(lp[r], ids[r], int(roots[r]), 1024) for r in range(2)]
    assert max(int(ref["rank"].max()) for ref in refs) > 255
    _check_tree(gpu, refs, 1024)


@pytest.mark.parametrize("kind", ["unsorted", "positive", "zero"])
def test_tree_build_inputs_outside_the_sorted_case(kind):
    # the parallel construction assumes non-increasing, non-positive rows and
    # distinct scores; anything else must still match Algorithm 1 exactly
    lp, ids = synth.random_topk_table(3, 15, 8, 50000, seed=17, tie_fraction=0.0)
    if kind == "unsorted":
        lp[:, 4, [2, 5]] = lp[:, 4, [5, 2]]
    elif kind == "positive":
        lp[:, 2, 0] = 0.25
    else:
        lp[:, 6, 0] = 0.0
    roots = np.arange(3, dtype=np.int32)
    gpu, _ = _gpu_tree(lp, ids, roots, 256)
    refs = [odt.build_tree(lp[r], ids[r], int(roots[r]), 256) for r in range(3)]
    _check_tree(gpu, refs, 256)


def test_exact_tie_order_on_gpu():
    lp = np.full((1, 3, 2), np.float32(np.log(0.5)), dtype=np.float32)
    ids = np.array([[[10, 11], [20, 21], [30, 31]]], dtype=np.int32)
    gpu, _ = _gpu_tree(lp, ids, np.zeros(1, np.int32), 10)
    ref = odt.build_tree(lp[0], ids[0], 0, 10)
    _check_tree(gpu, [ref], 10)


def test_stress_workload_tree_and_walk():
    """Stress workload end to end: the oracle's top-K of the stress logits feeds
    both tree builders (identical top-K inputs); targets agree with the planted
    token with probability 0.95^(depth+1); the walks must match exactly."""
    wl = WORKLOADS[4]
    logits, planted = synth.stress_logits(wl.n_req, wl.D, wl.vocab, wl.seed, device="cpu")
    o_ids, o_lp = _oracle_topk(logits, wl.K)
    lp = o_lp.astype(np.float32).reshape(wl.n_req, wl.D, wl.K)
    ids = o_ids.astype(np.int32).reshape(wl.n_req, wl.D, wl.K)
    roots = synth.anchors(wl.n_req, wl.vocab, wl.vocab - 1, wl.seed)
    gpu, bufs = _gpu_tree(lp, ids, roots, wl.B)
    refs = [odt.build_tree(lp[r], ids[r], int(roots[r]), wl.B) for r in range(wl.n_req)]
    _check_tree(gpu, refs, wl.B)
    depth = np.stack([ref["depth"] for ref in refs])
    tgt = synth.target_tokens([ref["n_nodes"] for ref in refs], depth, lp, ids, wl.vocab,
                              wl.target_agree, seed=wl.seed,
                              preferred=planted.numpy().reshape(wl.n_req, wl.D))
    _check_walk(bufs, refs, tgt, wl.D, wl.B)


def _check_walk(bufs, refs, tgt, D, B):
    n_req = len(refs)
    al = torch.empty(n_req, dtype=torch.int32, device=DEV)
    acc = torch.empty(n_req, D, dtype=torch.int32, device=DEV)
    bon = torch.empty(n_req, dtype=torch.int32, device=DEV)
    bd.ddtree_accept(D, B, bufs[0], bufs[1], bufs[2], torch.from_numpy(tgt).to(DEV), al, acc,
                     bon)
    torch.cuda.synchronize()
    al, acc, bon = al.cpu().numpy(), acc.cpu().numpy(), bon.cpu().numpy()
    for r, ref in enumerate(refs):
        a, nodes, bonus = odt.accept_walk(ref["tok"], ref["parent"], ref["n_nodes"], tgt[r], D)
        assert al[r] == a and bon[r] == bonus and np.array_equal(acc[r], nodes), r
        assert 1 <= al[r] + 1 <= D + 1


@pytest.mark.parametrize("temperature", [0.0, 1.0])
def test_walk_on_synthetic_trees(temperature):
    n_req, D, K, B = 16, 15, 8, 256
    lp, ids = synth.random_topk_table(n_req, D, K, 1000, seed=3, tie_fraction=0.2)
    roots = np.zeros(n_req, np.int32)
    gpu, bufs = _gpu_tree(lp, ids, roots, B)
    refs = [odt.build_tree(lp[r], ids[r], 0, B) for r in range(n_req)]
    depth = np.stack([ref["depth"] for ref in refs])
    tgt = synth.target_tokens([ref["n_nodes"] for ref in refs], depth, lp, ids, 1000, 0.9,
                              seed=7, temperature=temperature)
    _check_walk(bufs, refs, tgt, D, B)


def test_walk_all_match_and_no_match():
    n_req, D, K, B = 2, 6, 2, 20
    lp, ids = synth.random_topk_table(n_req, D, K, 100, seed=1)
    roots = np.zeros(n_req, np.int32)
    gpu, bufs = _gpu_tree(lp, ids, roots, B)
    refs = [odt.build_tree(lp[r], ids[r], 0, B) for r in range(n_req)]
    # request 0 follows the rank-1 chain as deep as it goes; request 1 matches nothing
    tgt = np.full((n_req, B + 1), -7, dtype=np.int32)
    ref = refs[0]
    for i in range(ref["n_nodes"] + 1):
        d = ref["depth"][i]
        if d < D:
            tgt[0, i] = ids[0, d, 0]
    _check_walk(bufs, refs, tgt, D, B)
