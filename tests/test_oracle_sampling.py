"""Pins for the sampling / chain oracle: SplitMix64 against its published first
outputs, Gumbel-max frequencies against softmax(l / T) (chi-square), the
low-temperature and T = 0 limits with the tie rule, and the chain tree against
the DDTree oracle's mask and walk (a chain walk is linear acceptance)."""
import numpy as np
import scipy.stats

from oracle import ddtree as odt
from oracle import sampling as osm


def test_splitmix64_published_outputs():
    # the first three outputs of SplitMix64 seeded with 0
    assert osm.splitmix64(0, 1) == 0xE220A8397B1DCDAF
    assert osm.splitmix64(0, 2) == 0x6E789E6AA1B965F4
    assert osm.splitmix64(0, 3) == 0x06C45D188009454F
    ks = np.arange(1, 50, dtype=np.uint64)
    vec = osm.splitmix64_np(12345, ks)
    assert [int(x) for x in vec] == [osm.splitmix64(12345, int(k)) for k in ks]


def test_uniforms_open_interval_and_moments():
    u = osm.uniforms(7, 3, 200000)
    assert u.dtype == np.float32 and u.min() > 0 and u.max() < 1
    # every value is an odd multiple of 2^-24, exactly representable
    assert np.all(np.mod(u.astype(np.float64) * 2.0 ** 24, 2.0) == 1.0)
    # the extreme codes stay inside (0, 1) with a finite Gumbel value
    ends = np.array([(0 + 0.5) * 2.0 ** -23, (2 ** 23 - 1 + 0.5) * 2.0 ** -23], dtype=np.float32)
    assert ends[1] < 1 and np.all(np.isfinite(osm.gumbel(ends)))
    assert abs(float(u.mean()) - 0.5) < 3e-3
    assert abs(float(u.var()) - 1 / 12) < 2e-3


def test_gumbel_max_draws_follow_softmax():
    logits = np.array([1.0, 0.2, -0.5, 2.0, 0.0], dtype=np.float32)
    T = 1.0
    n = 20000
    draws = osm.sample_rows(np.tile(logits, (n, 1)), T, seed=99)
    counts = np.bincount(draws, minlength=5)
    p = np.exp(logits.astype(np.float64) / T)
    p /= p.sum()
    chi2, pval = scipy.stats.chisquare(counts, p * n)
    assert pval > 1e-4, (counts, p * n)
    # at T = 0.5 the distribution sharpens as softmax(2 l)
    draws = osm.sample_rows(np.tile(logits, (n, 1)), 0.5, seed=5)
    counts = np.bincount(draws, minlength=5)
    p2 = np.exp(logits.astype(np.float64) / 0.5)
    p2 /= p2.sum()
    assert scipy.stats.chisquare(counts, p2 * n)[1] > 1e-4


def test_gumbel_top2_is_a_draw_without_replacement():
    # P(first = a, second = b) = p_a * p_b / (1 - p_a) over the 6 ordered pairs
    logits = np.array([0.7, -0.3, 0.1], dtype=np.float32)
    n = 12000
    pairs = np.zeros((3, 3), dtype=np.int64)
    for r in range(n):
        ids, _ = osm.gumbel_topk(logits, 1.0, 17, r, 2)
        pairs[ids[0], ids[1]] += 1
    p = np.exp(logits.astype(np.float64))
    p /= p.sum()
    obs, exp = [], []
    for a in range(3):
        for b in range(3):
            if a != b:
                obs.append(pairs[a, b])
                exp.append(n * p[a] * p[b] / (1 - p[a]))
    assert np.trace(pairs) == 0
    assert scipy.stats.chisquare(obs, exp)[1] > 1e-4
    # entry 0 is the single-token sample, and the log-probabilities are exact
    ids, lq = osm.gumbel_topk(logits, 1.0, 17, 5, 3)
    assert ids[0] == osm.sample_rows(logits[None], 1.0, 17, row_offset=5)[0]
    assert np.allclose(lq, np.log(p[ids]), atol=1e-12)


def test_limits_and_ties():
    rng = np.random.default_rng(0)
    logits = rng.normal(size=(6, 50)).astype(np.float32) * 5
    assert np.array_equal(osm.sample_rows(logits, 1e-4, seed=1), np.argmax(logits, axis=1))
    tied = np.zeros((2, 8), dtype=np.float32)
    tied[:, 3] = tied[:, 6] = 1.0
    assert list(osm.sample_rows(tied, 0.0, seed=0)) == [3, 3]


def test_chain_tree_mask_and_walk():
    tokens = [11, 12, 13, 14]
    t = osm.chain_tree(9, tokens, B=6)
    assert t["n_nodes"] == 4
    assert np.array_equal(t["mask"], odt.tree_mask(t["parent"], 4, 6))
    assert list(t["rank"][:6]) == [0, 1, 1, 1, 1, -1]
    # a budget below D keeps the first B positions
    short = osm.chain_tree(9, tokens, B=2)
    assert short["n_nodes"] == 2 and list(short["tok"]) == [9, 11, 12]
    assert np.array_equal(short["mask"], odt.tree_mask(short["parent"], 2, 2))
    # the walk on a chain accepts the longest matching prefix (linear acceptance)
    for k in range(5):
        target = np.full(7, -1, dtype=np.int32)
        for d in range(k):
            target[d] = tokens[d]          # the target's choice at node d matches the child
        target[k] = 777                    # then it picks something else
        acc_len, acc, bonus = odt.accept_walk(t["tok"], t["parent"], 4, target, 4)
        assert acc_len == k and bonus == (777 if k < 4 else target[4])
