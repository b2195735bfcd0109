"""Pins of the double-precision oracle against facts it does not itself define:
library routines (scipy softmax, numpy cumsum/searchsorted/argmax), closed
forms, the identity of the exactness theorem, and special cases the pages
state.  Each would fail under a plausible slip in the oracle (a swapped p/q,
a dropped temperature, a scalar subtracted instead of the draft row, an
off-by-one in the CDF, a tie broken the wrong way)."""
import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

from speculative_decoding_verification_52_gb300 import inputs as gen


def rand_logits(rng, V, scale=1.0):
    return scale * rng.standard_normal(V)


# --- softmax at temperature ("Speculative decoding and EAGLE", "Make it") ----

@pytest.mark.parametrize("V,T", [(2, 1.0), (8, 0.7), (1000, 1.3), (32000, 0.25)])
def test_softmax_matches_scipy(orc, V, T):
    rng = np.random.default_rng(V)
    z = rand_logits(rng, V, 3.0)
    p = orc.softmax(z, T)
    ref = sp_softmax(z / T)
    np.testing.assert_allclose(p, ref, rtol=1e-12, atol=1e-300)


def test_softmax_two_way_closed_form(orc):
    for z0, z1, T in [(0.3, -1.2, 1.0), (2.0, 2.5, 0.7), (-4.0, 1.0, 2.0)]:
        p = orc.softmax(np.array([z0, z1]), T)
        assert p[0] == pytest.approx(1.0 / (1.0 + np.exp((z1 - z0) / T)), rel=1e-14)


def test_softmax_uniform_and_shift(orc):
    p = orc.softmax(np.full(17, 3.25), 0.5)
    np.testing.assert_allclose(p, 1.0 / 17, rtol=1e-14)
    rng = np.random.default_rng(3)
    z = rand_logits(rng, 50)
    np.testing.assert_allclose(orc.softmax(z, 0.9), orc.softmax(z + 123.0, 0.9), rtol=1e-12)


def test_softmax_invalid_rows(orc):
    assert orc.softmax(np.array([0.0, np.nan, 1.0]), 1.0) is None
    assert orc.softmax(np.array([0.0, np.inf, 1.0]), 1.0) is None
    assert orc.softmax(np.array([-np.inf, -np.inf]), 1.0) is None
    p = orc.softmax(np.array([0.0, -np.inf, 0.0]), 1.0)
    assert p.tolist() == [0.5, 0.0, 0.5]


# --- residual and the exactness identity ("Speculative Decoding: from idea to
# SOTA", section 3) -------------------------------------------------------------

@pytest.mark.parametrize("V,seed", [(4, 0), (64, 1), (5000, 2)])
def test_exactness_identity_per_entry(orc, V, seed):
    """q*min(1,p/q) + (1-beta)*w/R == p for every entry; R == 1 - beta."""
    rng = np.random.default_rng(seed)
    p = sp_softmax(rand_logits(rng, V))
    q = sp_softmax(rand_logits(rng, V))
    w, R = orc.residual(p, q)
    beta = np.minimum(p, q).sum()
    assert R == pytest.approx(1.0 - beta, abs=1e-15)
    assert R == pytest.approx(np.abs(p - q).sum() / 2, abs=1e-15)
    accept_part = q * np.minimum(1.0, p / q)
    np.testing.assert_allclose(accept_part + (1.0 - beta) * w / R, p, rtol=0, atol=1e-15)


def test_residual_uses_whole_draft_row(orc):
    """With a one-hot draft at x the residual is p with x removed, renormalised
    (a scalar q(x) subtracted from every entry would not give this)."""
    p = np.array([0.1, 0.25, 0.4, 0.25])
    q = np.array([0.0, 0.0, 1.0, 0.0])
    w, R = orc.residual(p, q)
    assert R == pytest.approx(0.6, abs=1e-15)
    np.testing.assert_allclose(w / R, [0.1 / 0.6, 0.25 / 0.6, 0.0, 0.25 / 0.6], atol=1e-15)


def test_residual_sign(orc):
    p = np.array([0.7, 0.2, 0.1])
    q = np.array([0.2, 0.5, 0.3])
    w, R = orc.residual(p, q)
    assert w.tolist() == pytest.approx([0.5, 0.0, 0.0], abs=1e-16)
    assert R == pytest.approx(0.5, abs=1e-16)


# --- inverse CDF -----------------------------------------------------------------

def test_icdf_matches_searchsorted(orc):
    rng = np.random.default_rng(11)
    for V in (1, 3, 16, 1000):
        w = rng.random(V)
        w[rng.random(V) < 0.4] = 0.0
        if w.sum() == 0:
            w[-1] = 0.5
        R = w.sum()
        C = np.cumsum(w)
        for u in list(rng.random(200)) + [0.0]:
            v, gap = orc.icdf(w, R, u)
            ref = int(np.searchsorted(C, u * R, side="right"))
            assert v == ref
            assert w[v] > 0.0
            lo = C[v - 1] if v > 0 else 0.0
            assert gap == pytest.approx(min(u * R - lo, C[v] - u * R) / R, abs=1e-15)


def test_icdf_fallback_and_empty(orc):
    w = np.array([0.0, 0.3, 0.0])
    v, _ = orc.icdf(w, 0.3, 0.999999)
    assert v == 1
    v, _ = orc.icdf(np.zeros(4), 0.0, 0.5)
    assert v == -1
    # rounding leaves no crossing: fall back to the largest positive entry
    v, _ = orc.icdf(np.array([0.25, 0.25, 0.0]), 0.6, 0.99)
    assert v == 1


# --- accept test -------------------------------------------------------------------

def test_accept_rule(orc):
    # "Speculative decoding and EAGLE", "The exactness rule": r < p/q
    assert orc.accept(0.3, 0.5, 0.59) and not orc.accept(0.3, 0.5, 0.61)
    assert not orc.accept(0.3, 0.5, 0.6)            # strict
    assert orc.accept(0.9, 0.1, 0.999999)           # p >= q: always accepted
    # "Speculative decoding: draft, verify, repeat", step 1: zero draft probability accepted
    assert orc.accept(0.0, 0.0, 0.5) and orc.accept(0.2, 0.0, 0.99)
    # p/q, not q/p
    assert not orc.accept(0.1, 0.4, 0.3) and orc.accept(0.4, 0.1, 0.3)


# --- argmax ---------------------------------------------------------------------------

def test_argmax_first_index(orc):
    rng = np.random.default_rng(5)
    for _ in range(50):
        z = rng.integers(-3, 3, size=40).astype(np.float64)
        assert orc.argmax(z) == int(np.argmax(z))
    assert orc.argmax(np.array([1.0, np.nan])) == -1
    assert orc.argmax(np.array([-np.inf, -np.inf])) == 0
    assert orc.argmax(np.array([0.0, np.inf, np.inf])) == 1


# --- whole-step special cases the pages state -----------------------------------------

def _chain_inputs(target_rows, draft_rows, tokens, uniforms):
    t = np.asarray(target_rows, np.float32)[None]
    d = np.asarray(draft_rows, np.float32)[None]
    return t, d, np.asarray(tokens, np.int32)[None], np.asarray(uniforms, np.float32)[None]


def test_perfect_draft_gives_k_plus_one_tokens(orc):
    """"Speculative decoding and EAGLE", section "The concept": a perfect draft
    yields K+1 tokens per target pass; "Speculative decoding: draft, verify,
    repeat", step 3: five acceptances + one bonus = six tokens."""
    rng = np.random.default_rng(0)
    K, V = 5, 50
    z = rng.standard_normal((K + 1, V)).astype(np.float32)
    tok = rng.integers(0, V, size=K)
    uni = rng.random((K + 1, 2)).astype(np.float32)
    t, d, x, u = _chain_inputs(z, z[:K], tok, uni)
    r = orc.verify_sample(t, "f32", d, "f32", False, x, u, 1.0)
    assert r["num_accepted"][0] == K
    assert (r["out_tokens"][0, :K] == tok).all()
    p = sp_softmax(z[K].astype(np.float64))
    assert r["out_tokens"][0, K] == int(np.searchsorted(np.cumsum(p), uni[K, 1] * p.sum(), side="right"))


def test_wrong_first_draft_gives_one_token(orc):
    """A draft the target rules out at position 1 yields exactly one token,
    drawn from the residual ("Speculative decoding and EAGLE", "The concept")."""
    V, K = 6, 3
    z = np.zeros((K + 1, V), np.float32)
    z[0, 2] = -np.inf                       # p_0(2) = 0
    q = np.zeros((K, V), np.float32)
    q[:, 2] = 1.0                           # the draft proposes token 2 with certainty
    for u1 in (0.05, 0.5, 0.95):
        t, d, x, u = _chain_inputs(z, q, [2, 2, 2], [[0.0, u1]] * (K + 1))
        r = orc.verify_sample(t, "f32", d, "f32", True, x, u, 1.0)
        assert r["num_accepted"][0] == 0
        assert r["out_tokens"][0, 1:].tolist() == [-1] * K
        # residual = p_0 (token 2 removed) = uniform over the other 5 tokens
        expect = [0, 1, 3, 4, 5][int(u1 * 5)]
        assert r["out_tokens"][0, 0] == expect


def test_identical_draft_always_accepts(orc):
    rng = np.random.default_rng(1)
    K, V, B = 4, 30, 200
    z = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    tok = rng.integers(0, V, size=(B, K)).astype(np.int32)
    uni = rng.random((B, K + 1, 2)).astype(np.float32)
    r = orc.verify_sample(z, "f32", z[:, :K], "f32", False, tok, uni, 0.8)
    assert (r["num_accepted"] == K).all()
    assert np.allclose(r["ratio"], 1.0, atol=1e-12)


def test_temperature_zero_is_greedy(orc):
    rng = np.random.default_rng(2)
    K, V, B = 4, 40, 64
    z = rng.integers(-4, 4, size=(B, K + 1, V)).astype(np.float32)   # many ties
    g = np.argmax(z, axis=-1)
    tok = g[:, :K].copy()
    flip = rng.random((B, K)) < 0.3
    tok[flip] = (tok[flip] + 1) % V
    out, n = orc.verify_greedy(z, "f32", tok)
    r = orc.verify_sample(z, "f32", z[:, :K], "f32", False, tok, np.zeros((B, K + 1, 2), np.float32), 0.0)
    assert (r["num_accepted"] == n).all() and (r["out_tokens"] == out).all()
    for b in range(B):
        m = 0
        while m < K and tok[b, m] == g[b, m]:
            m += 1
        assert n[b] == m
        assert out[b, :m].tolist() == tok[b, :m].tolist()
        assert out[b, m] == g[b, m]
        assert (out[b, m + 1:] == -1).all()


def test_invalid_sequences(orc):
    K, V = 2, 8
    z = np.zeros((3, K + 1, V), np.float32)
    tok = np.zeros((3, K), np.int32)
    tok[1, 1] = V                              # out of range
    z[2, 0, 3] = np.nan                        # NaN in a row that is read
    uni = np.full((3, K + 1, 2), 0.5, np.float32)
    r = orc.verify_sample(z, "f32", z[:, :K], "f32", False, tok, uni, 1.0)
    assert r["num_accepted"].tolist() == [K, -1, -1]
    assert (r["out_tokens"][1:] == -1).all()
    out, n = orc.verify_greedy(z, "f32", tok)
    assert n.tolist()[1:] == [-1, -1]


# --- tree --------------------------------------------------------------------------

def _brute_tree(rows, parents, tokens):
    """Independent restatement: a node is on an accepted path iff every edge on
    its root path matches the argmax of the edge's upper end."""
    N = len(parents)
    g = [int(np.argmax(r)) for r in rows]
    best, bd = 0, 0
    for i in range(N):
        path, node, ok = [], i, True
        while node != 0:
            if tokens[node] != g[parents[node]]:
                ok = False
            path.append(node)
            node = parents[node]
        if ok and len(path) > bd:
            best, bd = i, len(path)
    path, node = [], best
    while node != 0:
        path.append(node)
        node = parents[node]
    path = path[::-1]
    return bd, [tokens[j] for j in path] + [g[best]], path


def test_tree_matches_brute_force(orc):
    rng = np.random.default_rng(7)
    for trial in range(300):
        br = [int(x) for x in rng.integers(1, 4, size=rng.integers(1, 4))]
        parents = gen.bfs_tree(br, max_nodes=16)
        N = len(parents)
        depth = int(gen.tree_depths(parents).max())
        V = 5
        rows = rng.integers(-2, 3, size=(N, V)).astype(np.float32)
        g = np.argmax(rows, axis=-1)
        tok = np.where(rng.random(N) < 0.6, g[np.maximum(parents, 0)], rng.integers(0, V, size=N)).astype(np.int32)
        tok[0] = -1
        out, n, path = orc.verify_tree_greedy(rows[None], "f32", parents, tok[None], depth)
        bd, btok, bpath = _brute_tree(rows, parents, tok)
        assert n[0] == bd
        assert out[0, :bd + 1].tolist() == btok
        assert (out[0, bd + 1:] == -1).all()
        assert path[0, :bd].tolist() == bpath


def test_chain_tree_equals_chain_greedy(orc):
    rng = np.random.default_rng(8)
    B, K, V = 40, 4, 20
    parents = gen.bfs_tree([1] * K)
    z = rng.integers(-3, 3, size=(B, K + 1, V)).astype(np.float32)
    g = np.argmax(z, axis=-1)
    tok = np.where(rng.random((B, K)) < 0.7, g[:, :K], rng.integers(0, V, size=(B, K))).astype(np.int32)
    out_c, n_c = orc.verify_greedy(z, "f32", tok)
    node_tok = np.concatenate([np.full((B, 1), -1, np.int32), tok], axis=1)
    out_t, n_t, _ = orc.verify_tree_greedy(z, "f32", parents, node_tok, K)
    assert (n_c == n_t).all() and (out_c == out_t).all()


def test_tree_bad_topology(orc):
    z = np.zeros((2, 3, 4), np.float32)
    for parents in ([0, 0, 1], [-1, 1, 0], [-1, 0, 5]):
        out, n, path = orc.verify_tree_greedy(z, "f32", np.array(parents, np.int32),
                                              np.zeros((2, 3), np.int32), 2)
        assert (n == -1).all() and (out == -1).all()
    out, n, _ = orc.verify_tree_greedy(z, "f32", np.array([-1, 0, 1], np.int32),
                                       np.zeros((2, 3), np.int32), 1)   # depth 2 > max_depth 1
    assert (n == -1).all()
