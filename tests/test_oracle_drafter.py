"""Pins for the drafter oracle: closed forms, independent formulations,
invariants and special cases that a dropped term, a wrong sign, a wrong index
or a transposed operand would break."""
import math

import numpy as np
import pytest
import scipy.special

from oracle import drafter as od


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def test_rms_norm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(0)
    x = rng.normal(size=(5, 64)) * 3.0 + 1.0
    y = od.rms_norm(x, np.ones(64), 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, atol=1e-14)
    assert np.allclose(od.rms_norm(7.5 * x, np.ones(64), 0.0), y, atol=1e-14)
    g = rng.uniform(0.5, 1.5, size=64)
    assert np.allclose(od.rms_norm(x, g, 0.0), y * g, atol=1e-14)
    # eps enters under the square root: a zero row stays zero, tiny rows shrink
    assert np.all(od.rms_norm(np.zeros((1, 8)), np.ones(8), 1e-6) == 0.0)
    small = np.full((1, 4), 1e-3)
    assert np.allclose(od.rms_norm(small, np.ones(4), 1e-6),
                       1e-3 / math.sqrt(1e-6 + 1e-6), rtol=1e-12)


# ---------------------------------------------------------------------------
# Rotary embedding
# ---------------------------------------------------------------------------

def _rope_complex(x, pos, theta):
    """Independent formulation: pair (a_i, b_i) as the complex number a + ib and
    multiply by exp(i * pos * theta^(-2i/hd))."""
    hd = x.shape[-1]
    half = hd // 2
    z = x[..., :half] + 1j * x[..., half:]
    freqs = np.array([theta ** (-2.0 * i / hd) for i in range(half)])
    rot = np.exp(1j * np.asarray(pos, dtype=np.float64)[:, None, None] * freqs[None, None, :])
    w = z * rot
    return np.concatenate([w.real, w.imag], axis=-1)


def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(6, 3, 16))
    pos = np.array([0, 1, 5, 100, 4097, 8191])
    for theta in (1.0e4, 1.0e6):
        assert np.allclose(od.apply_rope(x, pos, theta), _rope_complex(x, pos, theta),
                           atol=1e-12)


def test_rope_identity_at_zero_norm_and_quarter_turn():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(1, 2, 8))
    assert np.allclose(od.apply_rope(x, [0], 1e6), x, atol=0)
    y = od.apply_rope(np.repeat(x, 3, 0), [3, 70, 9000], 1e6)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), atol=1e-12)
    # head_dim 2: one pair, frequency 1; angle pi/2 maps (1, 0) to (0, 1)
    e = np.array([[[1.0, 0.0]]])
    assert np.allclose(od.apply_rope(e, [math.pi / 2], 1e6), [[[0.0, 1.0]]], atol=1e-15)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(3)
    q = rng.normal(size=(1, 1, 32))
    k = rng.normal(size=(1, 1, 32))
    s1 = np.sum(od.apply_rope(q, [10], 1e6) * od.apply_rope(k, [3], 1e6))
    s2 = np.sum(od.apply_rope(q, [1010], 1e6) * od.apply_rope(k, [1003], 1e6))
    s3 = np.sum(od.apply_rope(q, [11], 1e6) * od.apply_rope(k, [3], 1e6))
    assert s1 == pytest.approx(s2, abs=1e-10)
    assert abs(s1 - s3) > 1e-6


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def _attention_streaming(q, k, v):
    """Independent formulation: one key at a time with a running maximum and a
    running normaliser (log-sum-exp rescaling)."""
    out = np.zeros((q.shape[0], v.shape[1]))
    scale = 1.0 / math.sqrt(q.shape[1])
    for i in range(q.shape[0]):
        m, l, acc = -np.inf, 0.0, np.zeros(v.shape[1])
        for j in range(k.shape[0]):
            s = float(np.dot(q[i], k[j])) * scale
            m_new = max(m, s)
            c = math.exp(m - m_new) if m > -np.inf else 0.0
            p = math.exp(s - m_new)
            l = l * c + p
            acc = acc * c + p * v[j]
            m = m_new
        out[i] = acc / l
    return out


def test_attention_matches_streaming_formulation():
    rng = np.random.default_rng(4)
    q = rng.normal(size=(7, 16)) * 2.0
    k = rng.normal(size=(40, 16)) * 2.0
    v = rng.normal(size=(40, 16))
    assert np.allclose(od.attention(q, k, v), _attention_streaming(q, k, v), atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(5)
    q = rng.normal(size=(3, 8))
    v = rng.normal(size=(5, 8))
    # one key: output is that value
    assert np.allclose(od.attention(q, rng.normal(size=(1, 8)), v[:1]), np.repeat(v[:1], 3, 0))
    # identical keys: uniform weights, output is the mean value
    k = np.repeat(rng.normal(size=(1, 8)), 5, 0)
    assert np.allclose(od.attention(q, k, v), np.repeat(v.mean(0, keepdims=True), 3, 0))
    # a key far better aligned than the rest dominates
    k = rng.normal(size=(5, 8)) * 0.01
    k[2] = q[0] * 100.0
    assert np.allclose(od.attention(q[:1], k, v)[0], v[2], atol=1e-9)
    # permuting (key, value) pairs together changes nothing
    k = rng.normal(size=(5, 8))
    perm = rng.permutation(5)
    assert np.allclose(od.attention(q, k, v), od.attention(q, k[perm], v[perm]), atol=1e-14)


def test_silu_against_tanh_form():
    x = np.linspace(-30, 30, 601)
    sig = 0.5 * (1.0 + np.tanh(0.5 * x))
    assert np.allclose(od.silu(x), x * sig, atol=1e-12)
    assert od.silu(np.array([0.0]))[0] == 0.0


# ---------------------------------------------------------------------------
# Fusion and injection
# ---------------------------------------------------------------------------

def test_fusion_concatenation_order():
    # W_proj that copies layer 2's block out of [h_l1; h_l2; h_l3]
    rng = np.random.default_rng(6)
    d, nf = 4, 3
    feats = rng.normal(size=(5, nf * d))
    w = np.zeros((d, nf * d))
    w[:, d:2 * d] = np.eye(d)
    assert np.allclose(od.fuse_features(feats, w), feats[:, d:2 * d], atol=0)
    # a non-square W: entry [t, j] = sum_k W[j, k] feats[t, k]
    w = rng.normal(size=(3, nf * d))
    f = od.fuse_features(feats, w)
    assert f.shape == (5, 3)
    assert f[4, 2] == pytest.approx(float(sum(w[2, k] * feats[4, k] for k in range(nf * d))))


def test_inject_identity_projection_and_positions():
    rng = np.random.default_rng(7)
    n_kv, hd = 2, 8
    f = rng.normal(size=(3, n_kv * hd))
    eye = np.eye(n_kv * hd)
    K, V = od.inject_kv(f, eye, 2 * eye, [0, 0, 0], n_kv, hd, 1e6)
    assert K.shape == (n_kv, 3, hd)
    assert np.allclose(K, f.reshape(3, n_kv, hd).transpose(1, 0, 2))
    assert np.allclose(V, 2 * f.reshape(3, n_kv, hd).transpose(1, 0, 2))
    # keys carry RoPE at their own position; values do not
    K2, V2 = od.inject_kv(f, eye, eye, [5, 6, 7], n_kv, hd, 1e6)
    assert np.allclose(V2, f.reshape(3, n_kv, hd).transpose(1, 0, 2))
    want = _rope_complex(f.reshape(3, n_kv, hd), [5, 6, 7], 1e6).transpose(1, 0, 2)
    assert np.allclose(K2, want, atol=1e-12)


# ---------------------------------------------------------------------------
# The block pass
# ---------------------------------------------------------------------------

def _tiny(seed=0, n_layers=1, d=32, n_q=4, n_kv=2, hd=8, ff=24, V=50):
    rng = np.random.default_rng(seed)
    dims = dict(n_layers=n_layers, d=d, n_q=n_q, n_kv=n_kv, head_dim=hd, vocab=V,
                mask_id=V - 1, rope_theta=1e6, rms_eps=1e-6)

    def m(r, c):
        return rng.normal(size=(r, c)) / math.sqrt(c)

    w = {"embed": rng.normal(size=(V, d)), "lm_head": m(V, d),
         "final_norm": rng.uniform(0.5, 1.5, size=d)}
    for k in ("attn_norm", "mlp_norm"):
        w[k] = [rng.uniform(0.5, 1.5, size=d) for _ in range(n_layers)]
    w["wq"] = [m(n_q * hd, d) for _ in range(n_layers)]
    w["wk"] = [m(n_kv * hd, d) for _ in range(n_layers)]
    w["wv"] = [m(n_kv * hd, d) for _ in range(n_layers)]
    w["wo"] = [m(d, n_q * hd) for _ in range(n_layers)]
    w["w_gate"] = [m(ff, d) for _ in range(n_layers)]
    w["w_up"] = [m(ff, d) for _ in range(n_layers)]
    w["w_down"] = [m(d, ff) for _ in range(n_layers)]
    T = 12
    ck = [rng.normal(size=(n_kv, T + 4, hd)) for _ in range(n_layers)]
    cv = [rng.normal(size=(n_kv, T + 4, hd)) for _ in range(n_layers)]
    return dims, w, ck, cv, T


def test_block_with_silent_sublayers_is_norm_plus_head():
    dims, w, ck, cv, T = _tiny()
    w["wo"] = [np.zeros_like(a) for a in w["wo"]]
    w["w_down"] = [np.zeros_like(a) for a in w["w_down"]]
    L = 6
    logits = od.drafter_block(w, dims, ck, cv, T, anchor=3, L=L)
    h = w["embed"][dims["mask_id"]]
    h = h / np.sqrt(np.mean(h * h) + dims["rms_eps"]) * w["final_norm"]
    want = w["lm_head"] @ h
    assert logits.shape == (L - 1, dims["vocab"])
    assert np.allclose(logits, np.repeat(want[None], L - 1, 0), atol=1e-12)


def test_block_rows_differ_and_depend_on_anchor():
    dims, w, ck, cv, T = _tiny(n_layers=2)
    a = od.drafter_block(w, dims, ck, cv, T, anchor=3, L=6)
    b = od.drafter_block(w, dims, ck, cv, T, anchor=4, L=6)
    # the mask rows share an input; only the rotary positions separate them
    for i in range(1, 5):
        assert np.max(np.abs(a[i] - a[0])) > 1e-6
    # every mask row sees the anchor (bidirectional block)
    assert np.all(np.max(np.abs(a - b), axis=1) > 1e-9)


def test_block_ignores_cache_past_ctx_len_and_slot_order():
    dims, w, ck, cv, T = _tiny(n_layers=2)
    base = od.drafter_block(w, dims, ck, cv, T, anchor=3, L=5)
    ck2 = [c.copy() for c in ck]
    cv2 = [c.copy() for c in cv]
    for c in ck2 + cv2:
        c[:, T:] = 1e3          # garbage past the context
    assert np.allclose(od.drafter_block(w, dims, ck2, cv2, T, 3, 5), base, atol=1e-12)
    perm = np.random.default_rng(9).permutation(T)
    ck3 = [c.copy() for c in ck]
    cv3 = [c.copy() for c in cv]
    for c3, c in zip(ck3 + cv3, ck + cv):
        c3[:, :T] = c[:, perm]
    assert np.allclose(od.drafter_block(w, dims, ck3, cv3, T, 3, 5), base, atol=1e-12)
    # shortening the context changes the result
    assert np.max(np.abs(od.drafter_block(w, dims, ck, cv, T - 1, 3, 5) - base)) > 1e-9


def test_block_gqa_group_mapping():
    """Swap the two KV heads (cache and W_k/W_v rows) together with the two
    query-head groups (W_q rows, W_o columns): the output is unchanged only
    if query head h reads KV head h // (n_q / n_kv)."""
    dims, w, ck, cv, T = _tiny(n_layers=1, n_q=4, n_kv=2, hd=8)
    base = od.drafter_block(w, dims, ck, cv, T, anchor=3, L=5)
    hd = 8
    w2 = {k: (list(v) if isinstance(v, list) else v) for k, v in w.items()}
    qperm = np.concatenate([np.arange(2 * hd, 4 * hd), np.arange(0, 2 * hd)])
    kvperm = np.concatenate([np.arange(hd, 2 * hd), np.arange(0, hd)])
    w2["wq"] = [w["wq"][0][qperm]]
    w2["wo"] = [w["wo"][0][:, qperm]]
    w2["wk"] = [w["wk"][0][kvperm]]
    w2["wv"] = [w["wv"][0][kvperm]]
    ck2 = [ck[0][::-1].copy()]
    cv2 = [cv[0][::-1].copy()]
    assert np.allclose(od.drafter_block(w2, dims, ck2, cv2, T, 3, 5), base, atol=1e-12)
    # a mapping h % n_kv would not survive the same swap
    w3 = dict(w2)
    w3["wq"] = [w["wq"][0][np.concatenate([np.arange(hd, 2 * hd), np.arange(0, hd),
                                           np.arange(3 * hd, 4 * hd), np.arange(2 * hd, 3 * hd)])]]
    w3["wo"] = [w["wo"][0][:, np.concatenate([np.arange(hd, 2 * hd), np.arange(0, hd),
                                              np.arange(3 * hd, 4 * hd), np.arange(2 * hd, 3 * hd)])]]
    assert np.max(np.abs(od.drafter_block(w3, dims, ck2, cv2, T, 3, 5) - base)) > 1e-9


def test_anchor_isolation_variant():
    # one layer: mask rows read the anchor's layer-1 key/value, identical in both
    # variants, so the logits agree; two layers: they differ
    dims, w, ck, cv, T = _tiny(n_layers=1)
    a = od.drafter_block(w, dims, ck, cv, T, 3, 6, anchor_sees_block=True)
    b = od.drafter_block(w, dims, ck, cv, T, 3, 6, anchor_sees_block=False)
    assert np.allclose(a, b, atol=1e-12)
    dims, w, ck, cv, T = _tiny(n_layers=2)
    a = od.drafter_block(w, dims, ck, cv, T, 3, 6, anchor_sees_block=True)
    b = od.drafter_block(w, dims, ck, cv, T, 3, 6, anchor_sees_block=False)
    assert np.max(np.abs(a - b)) > 1e-9


def test_empty_context_is_block_only_attention():
    dims, w, ck, cv, T = _tiny()
    a = od.drafter_block(w, dims, ck, cv, 0, 3, 4)
    ck2 = [np.zeros((2, 0, 8))]
    cv2 = [np.zeros((2, 0, 8))]
    assert np.allclose(od.drafter_block(w, dims, ck2, cv2, 0, 3, 4), a, atol=0)


# ---------------------------------------------------------------------------
# log-softmax and top-K
# ---------------------------------------------------------------------------

def test_log_softmax_normalised_and_matches_scipy():
    rng = np.random.default_rng(10)
    x = rng.normal(size=(4, 1000)) * 5
    lp, lse = od.log_softmax(x)
    assert np.allclose(np.exp(lp).sum(1), 1.0, atol=1e-12)
    assert np.allclose(lp, scipy.special.log_softmax(x, axis=1), atol=1e-12)
    assert np.allclose(lse, scipy.special.logsumexp(x, axis=1), atol=1e-12)
    lp2, _ = od.log_softmax(x + 123.0)
    assert np.allclose(lp2, lp, atol=1e-11)


def test_topk_matches_full_sort_with_ties():
    rng = np.random.default_rng(11)
    x = np.round(rng.normal(size=(20, 300)) * 2) / 2      # many exact ties
    ids, vals = od.topk(x, 8)
    for r in range(20):
        order = sorted(range(300), key=lambda v: (-x[r, v], v))[:8]
        assert list(ids[r]) == order
        assert np.array_equal(vals[r], x[r, order])
    ids1, lp1, lse1 = od.logits_topk(x, 8)
    assert np.array_equal(ids1, ids)
    assert np.allclose(lp1, vals - scipy.special.logsumexp(x, axis=1)[:, None], atol=1e-12)


def test_context_copy_of_block_leaves_output_unchanged():
    """If the context holds an exact copy of every block key/value (keys rotated at
    the block's own positions ctx_len + j), each block entry's softmax weight is
    split evenly between the two copies and the output equals the run with no
    context at all.  Relative rotary positions make the absolute offset drop out.
    This pins both the block positions (ctx_len + j) and the use of block keys."""
    dims, w, _, _, _ = _tiny(n_layers=1, n_q=4, n_kv=2, hd=8)
    L = 4
    base = od.drafter_block(w, dims, [np.zeros((2, 0, 8))], [np.zeros((2, 0, 8))], 0, 3, L)
    x = np.stack([w["embed"][3]] + [w["embed"][dims["mask_id"]]] * (L - 1))
    h = od.rms_norm(x, w["attn_norm"][0], dims["rms_eps"])
    kraw = (h @ w["wk"][0].T).reshape(L, 2, 8)
    v = (h @ w["wv"][0].T).reshape(L, 2, 8)
    for copies in (1, 2):
        T = copies * L
        # the copies carry the rotary positions the block rows get in this run
        k = od.apply_rope(kraw, T + np.arange(L), 1e6).transpose(1, 0, 2)
        ck = np.concatenate([k] * copies, axis=1)
        cv = np.concatenate([v.transpose(1, 0, 2)] * copies, axis=1)
        out = od.drafter_block(w, dims, [ck], [cv], T, 3, L)
        assert np.allclose(out, base, atol=1e-10)


def test_block_and_context_keys_both_matter():
    dims, w, ck, cv, T = _tiny(n_layers=1)
    base0 = od.drafter_block(w, dims, ck, cv, 0, 3, 5)
    w2 = dict(w)
    w2["wk"] = [3.0 * w["wk"][0]]
    assert np.max(np.abs(od.drafter_block(w2, dims, ck, cv, 0, 3, 5) - base0)) > 1e-9
    base = od.drafter_block(w, dims, ck, cv, T, 3, 5)
    assert np.max(np.abs(od.drafter_block(w, dims, [3.0 * ck[0]], cv, T, 3, 5) - base)) > 1e-9


def test_swiglu_gate_sign_identity():
    """silu(-g) = silu(g) - g, so flipping W_gate moves the residual by exactly
    W_down (g * u).  Pins the SwiGLU form (a plain product g * u, or a missing
    gate nonlinearity, would move it by 2 W_down (g * u) or 0)."""
    dims, w, ck, cv, T = _tiny(n_layers=1)
    w["wo"] = [np.zeros_like(w["wo"][0])]
    _, xa = od.drafter_block(w, dims, ck, cv, T, 3, 5, return_residual=True)
    w2 = dict(w)
    w2["w_gate"] = [-w["w_gate"][0]]
    _, xb = od.drafter_block(w2, dims, ck, cv, T, 3, 5, return_residual=True)
    x0 = np.stack([w["embed"][3]] + [w["embed"][dims["mask_id"]]] * 4)
    h = od.rms_norm(x0, w["mlp_norm"][0], dims["rms_eps"])
    g, u = h @ w["w_gate"][0].T, h @ w["w_up"][0].T
    assert np.allclose(xa - xb, (g * u) @ w["w_down"][0].T, atol=1e-12)
    # and with the attention silent the residual is the embedding plus the MLP
    assert np.allclose(xa + xb - 2 * x0,
                       (2 * od.silu(g) * u - g * u) @ w["w_down"][0].T, atol=1e-12)
