"""Distribution-level pins of the oracle's sampler.

* The exact output law of one verification step is enumerated by brute force
  (every draft sequence, every accept/reject branch) for tiny vocabularies;
  the enumeration is itself checked against the exactness theorem of
  "Speculative Decoding: from idea to SOTA", section 3 (the first emitted token
  is distributed as p), and the oracle's sampled outputs over many trials are
  chi-square tested against it.
* The expected number of tokens per target pass is tested against the closed
  form (1 - a^(K+1)) / (1 - a) of "Speculative decoding and EAGLE", section
  "Expected speedup", on inputs with a controlled per-position acceptance a.
* The emitted token is chi-square tested against direct sampling from p, as the
  exercises of "Speculative decoding: draft, verify, repeat" prescribe.
"""
from collections import defaultdict

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax
from scipy.stats import chi2_contingency, chisquare

from speculative_decoding_verification_52_gb300 import inputs as gen

P_MIN = 1e-3


def closed_form_tokens(alpha, K):
    return (1.0 - alpha ** (K + 1)) / (1.0 - alpha) if alpha != 1.0 else K + 1.0


def exact_law(P, Q):
    """Brute-force law of (num_accepted, emitted tokens) for target rows P
    [K+1, V] and draft rows Q [K, V] (probabilities)."""
    K = Q.shape[0]
    V = P.shape[1]
    law = defaultdict(float)

    def rec(t, prefix, prob):
        if t == K:
            for v in range(V):
                law[(K, prefix + (v,))] += prob * P[K][v]
            return
        r = np.maximum(P[t] - Q[t], 0.0)
        Rs = r.sum()
        for x in range(V):
            if Q[t][x] == 0.0:
                continue
            a = min(1.0, P[t][x] / Q[t][x])
            rec(t + 1, prefix + (x,), prob * Q[t][x] * a)
            rej = prob * Q[t][x] * (1.0 - a)
            if rej > 0.0:
                for v in range(V):
                    if r[v] > 0.0:
                        law[(t, prefix + (v,))] += rej * r[v] / Rs

    rec(0, (), 1.0)
    return law


def run_trials(orc, z, y, T, M, seed):
    """M independent trials of one step with target logits z [K+1,V] and draft
    logits y [K,V]: draft tokens drawn from softmax(y/T) per trial."""
    rng = np.random.default_rng(seed)
    K, V = y.shape
    Q = sp_softmax(y.astype(np.float64) / T, axis=-1)
    tok = np.stack([rng.choice(V, size=M, p=Q[t]) for t in range(K)], axis=1).astype(np.int32)
    uni = rng.random((M, K + 1, 2), dtype=np.float32)
    tgt = np.broadcast_to(z.astype(np.float32), (M, K + 1, V))
    dft = np.broadcast_to(y.astype(np.float32), (M, K, V))
    return orc.verify_sample(tgt, "f32", dft, "f32", False, tok, uni, T)


@pytest.mark.parametrize("V,K,T", [(4, 2, 1.0), (3, 3, 0.8), (8, 2, 1.0), (8, 3, 1.3)])
def test_enumeration_obeys_theorem(V, K, T):
    rng = np.random.default_rng(100 + V * 10 + K)
    z = rng.standard_normal((K + 1, V))
    y = z[:K] + 0.6 * rng.standard_normal((K, V))
    P = sp_softmax(z / T, axis=-1)
    Q = sp_softmax(y / T, axis=-1)
    law = exact_law(P, Q)
    assert sum(law.values()) == pytest.approx(1.0, abs=1e-12)
    # slot j, conditional on reaching it, is distributed as p_j (rows do not
    # depend on the prefix here, so every slot obeys the theorem)
    for j in range(K + 1):
        reach = sum(pr for (n, _), pr in law.items() if n >= j)
        marg = np.zeros(V)
        for (n, toks), pr in law.items():
            if n >= j:
                marg[toks[j]] += pr
        np.testing.assert_allclose(marg / reach, P[j], atol=1e-12)


def _merge_bins(obs, exp, min_exp=5.0):
    order = np.argsort(exp)
    obs, exp = obs[order], exp[order]
    small = np.cumsum(exp) < min_exp * 4
    o, e = list(obs[~small]), list(exp[~small])
    if small.any():
        o.append(obs[small].sum())
        e.append(exp[small].sum())
    return np.array(o), np.array(e)


@pytest.mark.parametrize("V,K,T,seed", [(4, 2, 1.0, 1), (8, 3, 1.0, 2), (5, 3, 0.7, 3)])
def test_oracle_matches_exact_law(orc, V, K, T, seed):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((K + 1, V)).astype(np.float32)
    y = (z[:K] + 0.5 * rng.standard_normal((K, V))).astype(np.float32)
    M = 200_000
    r = run_trials(orc, z, y, T, M, seed + 1000)
    P = sp_softmax(z.astype(np.float64) / T, axis=-1)
    Q = sp_softmax(y.astype(np.float64) / T, axis=-1)
    law = exact_law(P, Q)
    keys = list(law.keys())
    index = {k: i for i, k in enumerate(keys)}
    counts = np.zeros(len(keys))
    n = r["num_accepted"]
    out = r["out_tokens"]
    for m in range(M):
        counts[index[(int(n[m]), tuple(int(v) for v in out[m, :n[m] + 1]))]] += 1
    expected = np.array([law[k] for k in keys]) * M
    o, e = _merge_bins(counts, expected)
    stat, pval = chisquare(o, e * o.sum() / e.sum())
    assert pval > P_MIN, (stat, pval)


def test_tiny_workload_first_token_is_p(orc):
    """The tiny exactness workload (V=8, K=4, fp32, T=1, 200k trials): the
    first emitted token follows p_0 and the accept count follows the law."""
    b = gen.config_tiny()
    r = orc.verify_sample(b.target, "f32", b.draft, "f32", False, b.draft_tokens, b.uniforms, b.T)
    P = sp_softmax(b.target[0].astype(np.float64) / b.T, axis=-1)
    Q = sp_softmax(b.draft[0].astype(np.float64) / b.T, axis=-1)
    counts = np.bincount(r["out_tokens"][:, 0], minlength=b.V)
    _, pval = chisquare(counts, P[0] * b.B)
    assert pval > P_MIN
    law = exact_law(P, Q)
    n_law = np.zeros(b.K + 1)
    for (n, _), pr in law.items():
        n_law[n] += pr
    _, pval = chisquare(np.bincount(r["num_accepted"], minlength=b.K + 1), n_law * b.B)
    assert pval > P_MIN


def test_tiny_workload_kl_and_tv_against_plain_sampling(orc):
    """The pages' own acceptance checks ("Speculative decoding and EAGLE",
    "Make it": the empirical KL of speculative sampling against plain target
    sampling below 0.01; exercise 1: the TV distance between the two output
    distributions): the first emitted token over 200k trials against p_0 and
    against 200k direct draws from p_0.  With 8 tokens the sampling noise is
    KL ~ 7 / (2 n) ~ 2e-5 and TV ~ 0.004."""
    b = gen.config_tiny()
    r = orc.verify_sample(b.target, "f32", b.draft, "f32", False, b.draft_tokens, b.uniforms, b.T)
    P0 = sp_softmax(b.target[0, 0].astype(np.float64))
    emp = np.bincount(r["out_tokens"][:, 0], minlength=b.V) / b.B
    direct = np.bincount(np.random.default_rng(13).choice(b.V, size=b.B, p=P0), minlength=b.V) / b.B
    kl = float(np.sum(np.where(emp > 0, emp * np.log(np.where(emp > 0, emp, 1.0) / P0), 0.0)))
    assert kl < 0.01
    assert 0.5 * np.abs(emp - P0).sum() < 0.01
    assert 0.5 * np.abs(emp - direct).sum() < 0.015


def test_two_sample_against_direct_sampling(orc):
    b = gen.config_tiny(trials=50_000, seed=7)
    r = orc.verify_sample(b.target, "f32", b.draft, "f32", False, b.draft_tokens, b.uniforms, b.T)
    P0 = sp_softmax(b.target[0, 0].astype(np.float64))
    direct = np.random.default_rng(9).choice(b.V, size=b.B, p=P0)
    table = np.stack([np.bincount(r["out_tokens"][:, 0], minlength=b.V),
                      np.bincount(direct, minlength=b.V)])
    _, pval, _, _ = chi2_contingency(table)
    assert pval > P_MIN


@pytest.mark.parametrize("alpha,K", [(0.8, 4), (0.75, 5), (0.5, 4), (0.7, 4), (0.9, 4), (0.85, 8)])
def test_expected_tokens_closed_form(orc, alpha, K):
    """Per-position acceptance exactly alpha: p_t(0) = alpha and a one-hot
    draft on token 0, so each test accepts with probability min(1, alpha)."""
    V, M = 6, 200_000
    p = np.full(V, (1.0 - alpha) / (V - 1))
    p[0] = alpha
    z = np.broadcast_to(np.log(p), (M, K + 1, V)).astype(np.float32)
    q = np.zeros((M, K, V), np.float32)
    q[:, :, 0] = 1.0
    tok = np.zeros((M, K), np.int32)
    uni = np.random.default_rng(int(alpha * 1000) + K).random((M, K + 1, 2), dtype=np.float32)
    r = orc.verify_sample(z, "f32", q, "f32", True, tok, uni, 1.0)
    toks = r["num_accepted"] + 1.0
    se = toks.std() / np.sqrt(M)
    assert abs(toks.mean() - closed_form_tokens(alpha, K)) < 4.5 * se
    # bonus / residual tokens follow the right rows
    rej = r["num_accepted"] < K
    assert (r["out_tokens"][rej, r["num_accepted"][rej]] != 0).all()   # residual excludes token 0


def test_closed_form_against_pages():
    # "Speculative decoding and EAGLE", section "Expected speedup": a=0.8, K=4 -> 3.36
    assert round(closed_form_tokens(0.8, 4), 2) == 3.36
    # "Speculative decoding: draft, verify, repeat", section "What determines
    # the speed": a=0.75, N=5 -> about 3x fewer large-model calls
    assert 2.9 < closed_form_tokens(0.75, 5) < 3.4
    # "Speculative Decoding: from idea to SOTA", section 4: the geometric sum
    for a in (0.5, 0.7, 0.9):
        for K in range(1, 9):
            assert closed_form_tokens(a, K) == pytest.approx(sum(a ** j for j in range(K + 1)), rel=1e-12)
