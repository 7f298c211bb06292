"""Pins for the DDTree oracle: brute-force optimality (Prop. 2), the prefix-
probability identity (Prop. 1) by exact enumeration and Monte Carlo, the
algorithm's counting claims (Prop. 3, at most B pops and 2B pushes), the
rank-tuple example, the mask's definition and the verifier walk's reduction to
linear acceptance on a chain."""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import ddtree as odt


def _table(seed, D, K, ties=False):
    rng = np.random.default_rng(seed)
    raw = rng.normal(size=(D, K + 3)) * 1.5
    if ties:
        raw = np.round(raw * 2) / 2
    m = raw.max(1, keepdims=True)
    lp = raw - (m + np.log(np.exp(raw - m).sum(1, keepdims=True)))
    lp = -np.sort(-lp, axis=1)[:, :K]
    ids = np.stack([rng.choice(1000, size=K, replace=False) for _ in range(D)])
    return lp.astype(np.float32), ids.astype(np.int32)


def _all_prefixes(D, K):
    out = []
    for d in range(1, D + 1):
        out.extend(itertools.product(range(1, K + 1), repeat=d))
    return out


def _q(lp, rho):
    return math.exp(sum(float(lp[i, r - 1]) for i, r in enumerate(rho)))


def _node_tuples(tree):
    return [odt.rank_tuple(tree["parent"], tree["rank"], i)
            for i in range(1, tree["n_nodes"] + 1)]


# ---------------------------------------------------------------------------
# Prop. 2 by brute force over every prefix-closed tree
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("D,K,B,seed", [(2, 3, 4, 0), (2, 3, 6, 1), (3, 2, 5, 2),
                                        (3, 2, 6, 3), (2, 3, 5, 4), (3, 2, 3, 5)])
def test_heap_tree_is_optimal_by_brute_force(D, K, B, seed):
    lp, ids = _table(seed, D, K)
    prefixes = _all_prefixes(D, K)
    best = 0.0
    for size in range(1, B + 1):
        for subset in itertools.combinations(prefixes, size):
            s = set(subset)
            if all(p[:-1] in s for p in subset if len(p) > 1):
                best = max(best, sum(_q(lp, p) for p in subset))
    tree = odt.build_tree(lp, ids, root_tok=7, B=B)
    assert tree["n_nodes"] == min(B, len(prefixes))
    assert odt.expected_acceptance(tree, lp) == pytest.approx(best, rel=1e-12, abs=1e-15)


# ---------------------------------------------------------------------------
# Prop. 2/3 at the tiny workload's shape: the heap returns a top-B set of S_K
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("ties", [False, True])
def test_heap_returns_top_b_of_all_prefixes(ties):
    D, K, B = 7, 4, 16
    lp, ids = _table(21, D, K, ties=ties)
    prefixes = _all_prefixes(D, K)
    assert len(prefixes) == 21844
    # float32 score along each prefix, accumulated in prefix order
    def f32score(rho):
        s = np.float32(0.0)
        for i, r in enumerate(rho):
            s = np.float32(s + lp[i, r - 1])
        return s
    scores = sorted((f32score(p) for p in prefixes), reverse=True)
    tree = odt.build_tree(lp, ids, root_tok=1, B=B)
    got = sorted((float(f32score(t)) for t in _node_tuples(tree)), reverse=True)
    assert got == [float(s) for s in scores[:B]]
    # node scores are the float32 prefix scores and pop in non-increasing order
    for i, t in enumerate(_node_tuples(tree), start=1):
        assert tree["score"][i] == f32score(t)
    ps = tree["pop_scores"]
    assert np.all(ps[1:] <= ps[:-1])


def test_distinct_scores_pop_in_descending_order_of_all_prefixes():
    # The premise of the GPU's parallel construction: with non-increasing,
    # non-positive rows and pairwise distinct prefix scores, Algorithm 1 pops
    # exactly the B best prefixes, one after another in descending score order.
    D, K, B = 6, 3, 40
    lp, ids = _table(5, D, K, ties=False)
    prefixes = _all_prefixes(D, K)

    def f32score(rho):
        s = np.float32(0.0)
        for i, r in enumerate(rho):
            s = np.float32(s + lp[i, r - 1])
        return s
    scored = sorted(((float(f32score(p)), tuple(p)) for p in prefixes), reverse=True)
    assert len({sc for sc, _ in scored}) == len(scored)   # the table has no ties
    tree = odt.build_tree(lp, ids, root_tok=1, B=B)
    assert [tuple(t) for t in _node_tuples(tree)] == [p for _, p in scored[:B]]


def test_enumerates_every_prefix_exactly_once():
    D, K = 3, 3
    lp, ids = _table(5, D, K, ties=True)
    total = sum(K ** d for d in range(1, D + 1))
    tree = odt.build_tree(lp, ids, root_tok=0, B=total + 5)
    tuples = _node_tuples(tree)
    assert tree["n_nodes"] == total
    assert sorted(tuples) == sorted(_all_prefixes(D, K))


# ---------------------------------------------------------------------------
# Prop. 1: E_Q[alpha_T] = sum_u q(u)
# ---------------------------------------------------------------------------

def _alpha(tree_tuples, y):
    s = set(tree_tuples)
    a = 0
    for d in range(1, len(y) + 1):
        if tuple(y[:d]) in s:
            a = d
        else:
            break
    return a


def test_prop1_exact_enumeration():
    D, K, B = 3, 3, 7
    lp, ids = _table(8, D, K)
    q = np.exp(lp.astype(np.float64))
    rest = 1.0 - q.sum(1)                    # mass outside the top-K (symbol 0)
    tree = odt.build_tree(lp, ids, root_tok=0, B=B)
    tt = _node_tuples(tree)
    e = 0.0
    for y in itertools.product(range(0, K + 1), repeat=D):
        p = 1.0
        for i, r in enumerate(y):
            p *= rest[i] if r == 0 else q[i, r - 1]
        e += p * _alpha(tt, list(y))
    assert e == pytest.approx(odt.expected_acceptance(tree, lp), rel=1e-12)


def test_prop1_monte_carlo():
    D, K, B = 6, 4, 20
    lp, ids = _table(9, D, K)
    q = np.exp(lp.astype(np.float64))
    probs = np.concatenate([q, (1.0 - q.sum(1))[:, None]], axis=1)   # rank K+1 = other
    tree = odt.build_tree(lp, ids, root_tok=0, B=B)
    s = set(_node_tuples(tree))
    rng = np.random.default_rng(10)
    n = 200_000
    ys = np.stack([rng.choice(K + 1, size=n, p=probs[i]) + 1 for i in range(D)], axis=1)
    # encode prefixes as integers in base K+2 and walk depth by depth: a sample
    # survives depth d if its length-d prefix is a node of the tree
    base = K + 2
    alpha = np.zeros(n)
    alive = np.ones(n, dtype=bool)
    code = np.zeros(n, dtype=np.int64)
    for d in range(1, D + 1):
        code = code * base + ys[:, d - 1]
        nodes_d = [t for t in s if len(t) == d]
        codes_d = np.array([sum(r * base ** (d - 1 - i) for i, r in enumerate(t))
                            for t in nodes_d], dtype=np.int64)
        hit = alive & np.isin(code, codes_d)
        alpha += hit
        alive = hit
    mean, sd = alpha.mean(), alpha.std() / math.sqrt(n)
    assert abs(mean - odt.expected_acceptance(tree, lp)) < 4 * sd + 1e-12


# ---------------------------------------------------------------------------
# Algorithm 1 bookkeeping and tree structure
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("D,K,B", [(15, 8, 64), (16, 8, 512), (7, 4, 16), (15, 8, 256),
                                   (4, 1, 16), (1, 8, 16)])
def test_counts_closure_and_order(D, K, B):
    lp, ids = _table(D * 100 + B, D, K, ties=True)
    tree = odt.build_tree(lp, ids, root_tok=5, B=B)
    n = tree["n_nodes"]
    assert n == min(B, sum(K ** d for d in range(1, D + 1)))
    assert tree["pops"] == n and tree["pushes"] <= 2 * B and tree["max_heap"] <= B + 1
    par, dep, rk, tk = tree["parent"], tree["depth"], tree["rank"], tree["tok"]
    assert tk[0] == 5 and dep[0] == 0 and par[0] == -1
    for i in range(1, n + 1):
        assert 0 <= par[i] < i
        assert dep[i] == dep[par[i]] + 1 <= D
        assert 1 <= rk[i] <= K
        assert tk[i] == ids[dep[i] - 1, rk[i] - 1]
        # siblings of lower rank were popped earlier (prefix closure of S_K)
        if rk[i] > 1:
            assert any(par[j] == par[i] and rk[j] == rk[i] - 1 for j in range(1, i))
    assert np.all(tree["pop_scores"][1:] <= tree["pop_scores"][:-1])
    assert np.all(tk[n + 1:] == -1) and np.all(par[n + 1:] == -1)


def test_rank_tuple_example(golden_dir):
    with open(os.path.join(golden_dir, "rank_tuple_example.json")) as f:
        g = json.load(f)
    ids = np.arange(30).reshape(3, 10) * 7 + 1        # ids[depth][rank-1]
    rho = tuple(g["rho"])
    want = tuple(int(ids[i, k]) for i, k in enumerate(g["ranks_zero_based_per_depth"]))
    assert odt.prefix_tokens(ids, rho) == want


def test_node_tokens_follow_rank_tuples():
    lp, ids = _table(3, 5, 4)
    tree = odt.build_tree(lp, ids, root_tok=9, B=30)
    for i in range(1, tree["n_nodes"] + 1):
        rho = odt.rank_tuple(tree["parent"], tree["rank"], i)
        path, j = [], i
        while j > 0:
            path.append(int(tree["tok"][j]))
            j = int(tree["parent"][j])
        assert odt.prefix_tokens(ids, rho) == tuple(reversed(path))


def test_greedy_chain_when_top1_dominates():
    # rank-1 far ahead at every depth: the first D pops are the greedy chain
    D, K = 6, 4
    lp = np.tile(np.array([-0.01, -9.0, -9.5, -10.0], dtype=np.float32), (D, 1))
    ids = np.arange(D * K, dtype=np.int32).reshape(D, K)
    tree = odt.build_tree(lp, ids, root_tok=0, B=D)
    assert list(tree["depth"][1:]) == list(range(1, D + 1))
    assert list(tree["rank"][1:]) == [1] * D


def test_zero_budget_and_tie_order():
    lp, ids = _table(4, 3, 3)
    t0 = odt.build_tree(lp, ids, root_tok=2, B=0)
    assert t0["n_nodes"] == 0 and t0["mask"].shape == (1, 1) and t0["mask"][0, 0] == 1
    # all-equal scores at one depth: ties pop in creation order (rank order)
    lp = np.full((1, 4), -1.0, dtype=np.float32)
    ids = np.array([[10, 11, 12, 13]], dtype=np.int32)
    t = odt.build_tree(lp, ids, root_tok=0, B=4)
    assert list(t["rank"][1:5]) == [1, 2, 3, 4]


# ---------------------------------------------------------------------------
# Mask
# ---------------------------------------------------------------------------

def test_mask_is_ancestor_closure():
    lp, ids = _table(12, 8, 4, ties=True)
    B = 70
    tree = odt.build_tree(lp, ids, root_tok=0, B=B)
    m = tree["mask"]
    assert m.shape == (B + 1, (B + 1 + 31) // 32)
    n = tree["n_nodes"]
    for i in range(B + 1):
        bits = {j for j in range(B + 1) if (int(m[i, j // 32]) >> (j % 32)) & 1}
        if i > n:
            assert bits == set()
            continue
        chain, j = set(), i
        while j >= 0:
            chain.add(j)
            j = int(tree["parent"][j]) if j > 0 else -1
        assert bits == chain
        assert len(bits) == tree["depth"][i] + 1


# ---------------------------------------------------------------------------
# Verifier walk
# ---------------------------------------------------------------------------

def test_walk_on_chain_is_linear_acceptance():
    """A K=1 tree is the single DFlash trajectory; the walk must equal linear
    acceptance: accept the longest matching prefix, bonus = target at the stop."""
    D = 10
    rng = np.random.default_rng(13)
    lp = np.full((D, 1), -0.5, dtype=np.float32)
    ids = rng.integers(0, 50, size=(D, 1)).astype(np.int32)
    tree = odt.build_tree(lp, ids, root_tok=3, B=D)
    drafts = [int(ids[d, 0]) for d in range(D)]
    for trial in range(50):
        stop = int(rng.integers(0, D + 1))
        # target token at depth d (the node after d accepted drafts)
        target_by_depth = [drafts[d] if d < stop else (drafts[d] + 1) % 50 if d < D
                           else int(rng.integers(0, 50)) for d in range(D + 1)]
        target = np.array([target_by_depth[tree["depth"][i]] for i in range(D + 1)])
        a, nodes, bonus = odt.accept_walk(tree["tok"], tree["parent"], tree["n_nodes"],
                                          target, D)
        linear = 0
        while linear < D and drafts[linear] == target_by_depth[linear]:
            linear += 1
        assert a == linear == stop
        assert bonus == target_by_depth[linear]
        assert 1 <= a + 1 <= D + 1
        assert list(nodes[:a]) == list(range(1, a + 1)) and np.all(nodes[a:] == -1)


def test_walk_switches_branches_and_bounds():
    lp, ids = _table(14, 6, 4)
    tree = odt.build_tree(lp, ids, root_tok=0, B=40)
    n = tree["n_nodes"]
    tok, par, dep = tree["tok"], tree["parent"], tree["depth"]
    # pick the deepest node and make the target follow its path exactly
    leaf = int(np.argmax(dep[:n + 1]))
    path, j = [], leaf
    while j > 0:
        path.append(j)
        j = int(par[j])
    path = path[::-1]
    target = np.full(n + 1, 999_999, dtype=np.int64)
    node = 0
    for c in path:
        target[node] = tok[c]
        node = c
    target[leaf] = 123
    a, nodes, bonus = odt.accept_walk(tok, par, n, target, 6)
    assert a == dep[leaf] and list(nodes[:a]) == path and bonus == 123
    # nothing matches: only the bonus token is committed
    a, nodes, bonus = odt.accept_walk(tok, par, n, np.full(n + 1, -5), 6)
    assert a == 0 and bonus == -5 and np.all(nodes == -1)


def test_exact_tie_pop_order_by_creation():
    """q = (1/2, 1/2) at every depth makes all candidates of one depth tie
    exactly.  Following the rule (pop max score, ties to the earlier-created
    candidate; each pop creates its sibling before its child), by hand:
      pop (1)        creates (2)#1, (1,1)#2
      pop (2)        creates (2,1)#3                 [rank K reached: no sibling]
      pop (1,1)      creates (1,2)#4, (1,1,1)#5
      pop (2,1)      creates (2,2)#6, (2,1,1)#7
      pop (1,2)      creates (1,2,1)#8
      pop (2,2)      creates (2,2,1)#9
      then depth 3 in creation order: (1,1,1) (2,1,1) (1,2,1) (2,2,1)."""
    lp = np.full((3, 2), np.float32(np.log(0.5)), dtype=np.float32)
    ids = np.array([[10, 11], [20, 21], [30, 31]], dtype=np.int32)
    t = odt.build_tree(lp, ids, root_tok=0, B=10)
    got = _node_tuples(t)
    assert got == [(1,), (2,), (1, 1), (2, 1), (1, 2), (2, 2),
                   (1, 1, 1), (2, 1, 1), (1, 2, 1), (2, 2, 1)]


@pytest.mark.parametrize("V,D,B,seed", [(12, 4, 6, 0), (9, 3, 9, 1), (20, 5, 16, 2)])
def test_lemma1_top_b_lists_suffice(V, D, B, seed):
    # Lemma 1 (DDTree page, 3.4.4): the best tree of budget B only uses tokens of
    # rank <= B at each depth, so the tree over the full sorted vocabulary (K = V)
    # and the tree over the top-min(B, V) lists are the same tree.
    rng = np.random.default_rng(seed)
    raw = rng.normal(size=(D, V)) * 1.7
    lp_full = raw - np.log(np.exp(raw).sum(axis=1, keepdims=True))
    order = np.argsort(-lp_full, axis=1, kind="stable")
    lp_sorted = np.take_along_axis(lp_full, order, axis=1).astype(np.float32)
    ids_sorted = order.astype(np.int32)
    full = odt.build_tree(lp_sorted, ids_sorted, 3, B)
    k = min(B, V)
    cut = odt.build_tree(lp_sorted[:, :k], ids_sorted[:, :k], 3, B)
    for key in ("n_nodes", "tok", "parent", "depth", "rank"):
        assert np.array_equal(np.asarray(full[key]), np.asarray(cut[key])), key
    assert np.array_equal(full["mask"], cut["mask"])
    # no node of the full-vocabulary tree uses a rank above B
    assert int(np.max(full["rank"])) <= B
