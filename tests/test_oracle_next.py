"""Pins of the oracle's tree-attention mask and KV commit (the steps before
and after verification): the pages' worked example and exercise, closed forms
for chains and stars, and invariants of ancestor sets and of an append."""
import json
import os

import numpy as np
import pytest

from speculative_decoding_verification_52_gb300 import inputs as gen

CASES = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "next_cases.json")))


def bits(mask_row, N):
    return [j for j in range(N) if (int(mask_row[j // 32]) >> (j % 32)) & 1]


def test_tree_mask_page_example(orc):
    c = CASES["tree_mask_example"]
    m, st = orc.tree_mask(np.array(c["parents"]))
    assert st.tolist() == [0]
    N = len(c["parents"])
    assert [bits(m[0, i], N) for i in range(N)] == c["attends_to"]


@pytest.mark.parametrize("N", [1, 5, 32, 33, 100])
def test_tree_mask_chain_is_causal(orc, N):
    m, st = orc.tree_mask(np.arange(-1, N - 1))
    assert st[0] == 0
    for i in range(N):
        assert bits(m[0, i], N) == list(range(i + 1))


def test_tree_mask_star(orc):
    N = 40
    m, _ = orc.tree_mask(np.array([-1] + [0] * (N - 1)))
    assert bits(m[0, 0], N) == [0]
    for i in range(1, N):
        assert bits(m[0, i], N) == [0, i]


def test_tree_mask_random_trees_invariants(orc):
    rng = np.random.default_rng(5)
    for _ in range(30):
        N = int(rng.integers(1, 200))
        par = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, N)])
        m, st = orc.tree_mask(par)
        assert st[0] == 0
        depth = gen.tree_depths(par)
        for i in range(N):
            row = bits(m[0, i], N)
            assert len(row) == depth[i] + 1 and row[-1] == i and row[0] == 0
            for j in row:   # ancestor sets are closed: j's ancestors are i's
                assert set(bits(m[0, j], N)) <= set(row)


def test_tree_mask_batch_and_invalid(orc):
    good = [-1, 0, 0, 1]
    par = np.array([good, [0, 0, 0, 1], [-1, 0, 3, 1], [-1, -1, 0, 1], good])
    m, st = orc.tree_mask(par)
    assert st.tolist() == [0, -1, -1, -1, 0]
    assert not m[1:4].any()
    assert (m[0] == m[4]).all()


def test_kv_commit_rollback_exercise(orc):
    c = CASES["kv_rollback_exercise"]
    L, K = c["prefix_len"], c["drafts"]
    Lmax, E = 32, 3
    rng = np.random.default_rng(0)
    prefix = rng.integers(0, 255, size=(L, E), dtype=np.uint8)
    cache = np.zeros((1, Lmax, E), np.uint8)
    cache[0, :L] = prefix
    scratch = rng.integers(0, 255, size=(1, K, E), dtype=np.uint8)   # the 5 drafts' entries
    accepted = c["rejected_at_position"] - 1                         # drafts before the rejected one
    out, newl = orc.kv_commit(cache, [L], scratch, None, [accepted])
    assert newl.tolist() == [c["expected_len"]]
    assert (out[0, :L] == prefix).all()
    assert (out[0, L:newl[0]] == scratch[0, :2]).all()
    assert not out[0, newl[0]:].any()


def test_kv_commit_paths_and_errors(orc):
    rng = np.random.default_rng(1)
    B, Lmax, N, W = 4, 16, 7, 4
    cache = rng.integers(0, 255, size=(B, Lmax, 2, 3), dtype=np.uint8)
    scratch = rng.integers(0, 255, size=(B, N, 2, 3), dtype=np.uint8)
    lengths = np.array([3, 0, 15, 5])
    path = np.array([[1, 3, 6, -1], [0, 1, 2, 3], [2, -1, -1, -1], [5, 9, -1, -1]])
    count = np.array([3, 4, 2, 2])
    out, newl = orc.kv_commit(cache, lengths, scratch, path, count)
    assert newl.tolist() == [6, 4, -1, -1]          # seq 2 overflows, seq 3 names slot 9 >= N
    assert (out[0, 3:6] == scratch[0, [1, 3, 6]]).all()
    assert (out[1, 0:4] == scratch[1, :4]).all()
    assert (out[2] == cache[2]).all() and (out[3] == cache[3]).all()
    assert (out[0, :3] == cache[0, :3]).all() and (out[0, 6:] == cache[0, 6:]).all()
    # identity path equals no path; a negative count appends nothing
    o1, n1 = orc.kv_commit(cache, lengths, scratch, np.tile(np.arange(W), (B, 1)), [2, 2, 1, -1])
    o2, n2 = orc.kv_commit(cache, lengths, scratch, None, [2, 2, 1, -1])
    assert (o1 == o2).all() and (n1 == n2).all() and n2[3] == lengths[3]


# --- acceptance statistics ------------------------------------------------------

def _stats_batch(rng, B, K, V, scale=2.0, sigma=0.7):
    z = scale * rng.standard_normal((B, K + 1, V))
    y = z[:, :K] + sigma * rng.standard_normal((B, K, V))
    return z.astype(np.float32), y.astype(np.float32)


def test_row_stats_match_scipy(orc):
    from scipy.special import rel_entr, softmax
    rng = np.random.default_rng(9)
    z, y = _stats_batch(rng, 3, 4, 500)
    T = 0.8
    a, k, tv = orc.row_stats(z, "f32", y, "f32", False, T)
    P = softmax(z[:, :4].astype(np.float64) / T, axis=-1)
    Q = softmax(y.astype(np.float64) / T, axis=-1)
    np.testing.assert_allclose(a, np.minimum(P, Q).sum(-1), rtol=1e-12)
    np.testing.assert_allclose(k, rel_entr(Q, P).sum(-1), rtol=1e-10)
    np.testing.assert_allclose(tv, 0.5 * np.abs(P - Q).sum(-1), rtol=1e-12)


def test_row_stats_identities(orc):
    rng = np.random.default_rng(10)
    for sigma in (0.01, 0.3, 1.0, 3.0):
        z, y = _stats_batch(rng, 2, 3, 1000, sigma=sigma)
        a, k, tv = orc.row_stats(z, "f32", y, "f32", False, 1.0)
        np.testing.assert_allclose(tv, 1.0 - a, atol=1e-12)     # TV = 1 - sum min(p, q)
        assert (tv <= np.sqrt(k / 2.0) + 1e-12).all()           # Pinsker
        assert (k >= 0).all() and ((0 <= a) & (a <= 1)).all()
    z, _ = _stats_batch(rng, 2, 3, 300)
    a, k, tv = orc.row_stats(z, "f32", z[:, :3], "f32", False, 0.7)   # q = p
    np.testing.assert_allclose(a, 1.0, atol=1e-12)
    np.testing.assert_allclose(k, 0.0, atol=1e-12)


def test_row_stats_two_point_closed_form(orc):
    for pa, qa in [(0.3, 0.6), (0.9, 0.1), (0.5, 0.5)]:
        z = np.log(np.array([[[pa, 1 - pa], [0.5, 0.5]]]))
        y = np.array([[[qa, 1 - qa]]], np.float32)
        a, k, tv = orc.row_stats(z.astype(np.float32), "f32", y, "f32", True, 1.0)
        assert a[0, 0] == pytest.approx(min(pa, qa) + min(1 - pa, 1 - qa), abs=1e-7)
        assert k[0, 0] == pytest.approx(qa * np.log(qa / pa) + (1 - qa) * np.log((1 - qa) / (1 - pa)), abs=1e-6)


def test_alpha_is_the_acceptance_probability_of_the_law(orc):
    """alpha_0 is the probability that position 0 is accepted, by the
    brute-force law of one verification step (every draft, every branch)."""
    from scipy.special import softmax
    from test_oracle_law import exact_law
    rng = np.random.default_rng(11)
    for V in (3, 5, 8):
        z, y = _stats_batch(rng, 1, 2, V, scale=1.0, sigma=0.8)
        a, _, _ = orc.row_stats(z, "f32", y, "f32", False, 1.0)
        law = exact_law(softmax(z[0].astype(np.float64), axis=-1), softmax(y[0].astype(np.float64), axis=-1))
        p_acc0 = sum(pr for (n, _), pr in law.items() if n >= 1)
        assert a[0, 0] == pytest.approx(p_acc0, abs=1e-12)


def test_row_stats_invalid_rows(orc):
    rng = np.random.default_rng(12)
    z, y = _stats_batch(rng, 2, 2, 50)
    z[0, 1, 3] = np.nan
    y[1, 0, 7] = np.inf
    a, k, tv = orc.row_stats(z, "f32", y, "f32", False, 1.0)
    assert np.isnan(a[0, 1]) and np.isnan(k[1, 0]) and np.isnan(tv[1, 0])
    assert np.isfinite(a[0, 0]) and np.isfinite(a[1, 1])


# --- top-k tree drafting ------------------------------------------------------------

def _np_topk(row, k):
    """Reference order: decreasing logit, smaller index first on ties (numpy lexsort)."""
    order = np.lexsort((np.arange(len(row)), -row.astype(np.float64)))
    return order[:k]


def test_tree_draft_page_example(orc):
    """The pages' example tree: root with candidates a, b; c, d under a; e, f
    under b.  Each node's children are the top-2 of its draft row."""
    c = CASES["tree_mask_example"]
    par = np.array(c["parents"], np.int32)
    V = 6
    rows = np.full((1, 7, V), -5.0, np.float32)
    rows[0, 0, [4, 1]] = [3.0, 2.0]        # root: a = token 4, b = token 1
    rows[0, 1, [0, 5]] = [1.0, 0.5]        # under a: c = 0, d = 5
    rows[0, 2, [2, 3]] = [0.25, 0.25]      # under b: a tie, the smaller index first: e = 2, f = 3
    tok, lq, rc = orc.tree_draft(rows, "f32", par, 1.0)
    assert rc == 0
    assert tok[0].tolist() == [-1, 4, 1, 0, 5, 2, 3]
    from scipy.special import log_softmax
    ls = log_softmax(rows[0].astype(np.float64), axis=-1)
    assert lq[0, 0] == 0.0
    for i in range(1, 7):
        assert lq[0, i] == pytest.approx(ls[par[i], tok[0, i]], abs=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tree_draft_matches_numpy_topk(orc, dtype):
    rng = np.random.default_rng(21)
    par = gen.bfs_tree([4, 3, 2, 1], 64)
    B, N, V, T = 3, len(par), 500, 0.7
    z = rng.standard_normal((B, N, V))
    z = np.round(z * 4) / 4                   # many exact ties
    raw = gen._store(z, dtype) if dtype == "bf16" else z.astype(np.float32)
    tok, lq, rc = orc.tree_draft(raw, dtype, par, T)
    zz = gen.as_f64(raw, dtype)
    from scipy.special import log_softmax
    for b in range(B):
        for p in range(N):
            kids = [i for i in range(N) if par[i] == p]
            if not kids:
                continue
            want = _np_topk(zz[b, p], len(kids))
            assert tok[b, kids].tolist() == want.tolist()
            np.testing.assert_allclose(lq[b, kids], log_softmax(zz[b, p] / T)[want], atol=1e-12)


def test_tree_draft_flat_rows_take_the_smallest_indices(orc):
    """A row of equal logits: every token ties, so the children take tokens
    0, 1, 2, ... in node order, each with log q = -ln V (uniform)."""
    par = gen.bfs_tree([5, 3], None)
    B, N, V = 2, len(par), 300
    z = np.full((B, N, V), 1.25, np.float32)
    tok, lq, _ = orc.tree_draft(z, "f32", par, 0.9)
    for p in range(N):
        kids = [i for i in range(N) if par[i] == p]
        if kids:
            assert tok[:, kids].tolist() == [list(range(len(kids)))] * B
            np.testing.assert_allclose(lq[:, kids], -np.log(V), atol=1e-12)


def test_tree_draft_chain_is_greedy_and_perfect_draft_is_accepted(orc):
    """A chain tree drafts the argmax at every step; with the target equal to
    the draft, greedy tree verification accepts the whole tree depth along the
    first children."""
    rng = np.random.default_rng(22)
    V = 300
    chain = np.arange(-1, 5, dtype=np.int32)
    z = rng.standard_normal((2, 6, V)).astype(np.float32)
    tok, _, _ = orc.tree_draft(z, "f32", chain, 1.0)
    for b in range(2):
        assert tok[b, 1:].tolist() == [int(np.argmax(z[b, t])) for t in range(5)]
    par = gen.bfs_tree([3, 3, 2], None)
    N = len(par)
    z = rng.standard_normal((4, N, V)).astype(np.float32)
    tok, _, _ = orc.tree_draft(z, "f32", par, 1.0)
    depth = gen.tree_depths(par)
    out, n, path = orc.verify_tree_greedy(z, "f32", par, tok, int(depth.max()))
    assert (n == depth.max()).all()
    first_child = {p: min(i for i in range(N) if par[i] == p) for p in set(par[1:].tolist())}
    for b in range(4):
        node = 0
        for d in range(int(depth.max())):
            node = first_child[node]
            assert path[b, d] == node


def test_tree_draft_invalid_rows_and_topology(orc):
    par = np.array([-1, 0, 0, 1, 1], np.int32)
    z = np.zeros((2, 5, 8), np.float32)
    z[0, 1, 3] = np.nan                       # node 1's row: its children get -1
    z[1, 0, :] = -np.inf                      # root row with no finite entry
    tok, lq, rc = orc.tree_draft(z, "f32", par, 1.0)
    assert rc == 0
    assert tok[0, 3] == -1 and tok[0, 4] == -1 and np.isnan(lq[0, 3])
    assert tok[0, 1] == 0 and tok[0, 2] == 1   # all-equal row: indices in order
    assert tok[1, 1] == -1 and tok[1, 2] == -1
    tok, lq, rc = orc.tree_draft(z, "f32", np.array([-1, 0, 2, 1, 1], np.int32), 1.0)
    assert rc == 1 and (tok == -1).all() and np.isnan(lq).all()
    tok, lq, rc = orc.tree_draft(z, "f32", par, 1.0, max_children=1)   # the root has 2 children
    assert rc == 1 and (tok == -1).all() and np.isnan(lq).all()
    tiny = np.zeros((1, 4, 2), np.float32)   # 3 children, V = 2: the third gets -1
    tok, lq, _ = orc.tree_draft(tiny, "f32", np.array([-1, 0, 0, 0], np.int32), 1.0)
    assert tok[0].tolist() == [-1, 0, 1, -1] and np.isnan(lq[0, 3])
