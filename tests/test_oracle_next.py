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
