"""CUDA path vs the double-precision oracle on the same seeded inputs, through
the C ABI.  Greedy and tree modes are bit-exact; sampling mode is bit-exact
except after decisions within 1e-6 of flipping (counted); the replacement
distribution the device builds is within 1e-6 absolute of the oracle's."""
import numpy as np
import pytest
import torch
from scipy.special import softmax as sp_softmax
from scipy.stats import chisquare

import golden_cases as gc
import gpu_util as gu
import speculative_decoding_verification_52_gb300 as sv
from speculative_decoding_verification_52_gb300 import inputs as gen

pytestmark = pytest.mark.gpu
CASES = gc.load()


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    sv.lib()


# --- hand-derived cases ------------------------------------------------------------

@pytest.mark.parametrize("case", CASES["sample_cases"], ids=lambda c: c["name"])
def test_golden_sample(case):
    target, draft, tokens, uni = gc.sample_case(case)
    out, n = sv.spec_verify_sample(gu.f32(target), gu.f32(draft), gu.i32(tokens), gu.f32(uni), 1.0,
                                   draft_kind="probs")
    assert out.cpu().numpy()[0].tolist() == case["out_tokens"]
    assert int(n.cpu()[0]) == case["num_accepted"]


@pytest.mark.parametrize("case", CASES["greedy_cases"], ids=lambda c: c["name"])
def test_golden_greedy(case):
    target, tokens = gc.greedy_case(case)
    for dt in ("f32", "bf16"):
        t = gen.f32_to_bf16_bits(target) if dt == "bf16" else target
        out, n = sv.spec_verify_greedy(gu.dev_tensor(t, dt), gu.i32(tokens))
        assert out.cpu().numpy()[0].tolist() == case["out_tokens"]
        assert int(n.cpu()[0]) == case["num_accepted"]


@pytest.mark.parametrize("case", CASES["tree_cases"], ids=lambda c: c["name"])
def test_golden_tree(case):
    rows, parents, tokens, max_depth = gc.tree_case(case)
    out, n, path = sv.spec_verify_tree_greedy(gu.f32(rows), gu.i32(parents), gu.i32(tokens), max_depth)
    assert out.cpu().numpy()[0].tolist() == case["out_tokens"]
    assert int(n.cpu()[0]) == case["num_accepted"]
    assert path.cpu().numpy()[0].tolist() == case["out_path"]


# --- greedy ----------------------------------------------------------------------

def test_greedy_zipf_fp32(orc):
    """B=64, V=32000, K=4 fp32, temperature 0 (greedy run)."""
    b = gen.config_zipf(T=0.0)
    ro, rn = orc.verify_greedy(b.target, "f32", b.draft_tokens)
    out, n = sv.spec_verify_greedy(gu.f32(b.target), gu.i32(b.draft_tokens))
    assert (n.cpu().numpy() == rn).all() and (out.cpu().numpy() == ro).all()
    assert rn.mean() > 0.5            # the greedy draft is often right
    out2, n2 = gu.gpu_sample(b, T=0.0)   # temperature 0 through the sampling entry
    assert (n2 == rn).all() and (out2 == ro).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V,K,B", [(8, 4, 33), (1000, 0, 5), (4096, 5, 40), (1001, 3, 17), (16387, 2, 9),
                                   (100000, 31, 3), (3, 1, 50)])
def test_greedy_ties_and_shapes(orc, dtype, V, K, B):
    rng = np.random.default_rng(V * 31 + K)
    z = rng.integers(-3, 3, size=(B, K + 1, V)).astype(np.float32)      # heavy ties
    raw = gen.f32_to_bf16_bits(z) if dtype == "bf16" else z
    g = np.argmax(z, axis=-1)
    tok = np.where(rng.random((B, K)) < 0.8, g[:, :K], rng.integers(0, V, size=(B, K))).astype(np.int32)
    ro, rn = orc.verify_greedy(raw, dtype, tok)
    out, n = sv.spec_verify_greedy(gu.dev_tensor(raw, dtype), gu.i32(tok))
    assert (n.cpu().numpy() == rn).all() and (out.cpu().numpy() == ro).all()


def test_greedy_invalid_rows(orc):
    rng = np.random.default_rng(3)
    B, K, V = 12, 3, 2048
    z = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    g = np.argmax(z, axis=-1)
    tok = g[:, :K].copy().astype(np.int32)
    z[1, 0, 5] = np.nan            # row read -> invalid
    z[2, 3, 7] = np.nan            # bonus row read (all accepted) -> invalid
    tok[3, 0] = (tok[3, 0] + 1) % V
    z[3, 2, 9] = np.nan            # after the stop: not read -> fine
    tok[4, 1] = V                  # out of range -> invalid
    tok[5, 2] = -1
    z[6, 1, :] = -np.inf           # argmax of an all -inf row is index 0
    z[7, 0, 11] = np.inf
    ro, rn = orc.verify_greedy(z, "f32", tok)
    out, n = sv.spec_verify_greedy(gu.f32(z), gu.i32(tok))
    assert (n.cpu().numpy() == rn).all() and (out.cpu().numpy() == ro).all()
    assert rn[1] == -1 and rn[2] == -1 and rn[3] == 0 and rn[4] == -1 and rn[5] == -1


# --- sampling ----------------------------------------------------------------------

def test_sample_tiny_exactness(orc):
    """V=8, K=4 fp32, T=1, 200k trials: bit-exact against the oracle outside
    flagged decisions; the first emitted token follows p_0 (chi-square)."""
    b = gen.config_tiny()
    ref = gu.oracle_sample(orc, b)
    out, n = gu.gpu_sample(b)
    flagged = gu.compare_sample(out, n, ref)
    assert flagged < 50
    P0 = sp_softmax(b.target[0, 0].astype(np.float64))
    _, pval = chisquare(np.bincount(out[:, 0], minlength=b.V), P0 * b.B)
    assert pval > 1e-3
    # the pages' checks: empirical KL against the target below 0.01, and a small
    # TV distance between speculative and plain target sampling
    emp = np.bincount(out[:, 0], minlength=b.V) / b.B
    direct = np.bincount(np.random.default_rng(13).choice(b.V, size=b.B, p=P0), minlength=b.V) / b.B
    kl = float(np.sum(np.where(emp > 0, emp * np.log(np.where(emp > 0, emp, 1.0) / P0), 0.0)))
    assert kl < 0.01
    assert 0.5 * np.abs(emp - P0).sum() < 0.01
    assert 0.5 * np.abs(emp - direct).sum() < 0.015


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_sample_zipf_fp32(orc, T):
    b = gen.config_zipf(T=T)
    ref = gu.oracle_sample(orc, b, T)
    out, n = gu.gpu_sample(b, T)
    gu.compare_sample(out, n, ref)
    assert (n >= 0).all()


def test_sample_headline_full(orc):
    """B=256, V=128256, K=5 bf16, T=0.7 -- the benchmark workload, every sequence."""
    b = gen.config_headline()
    ref = gu.oracle_sample(orc, b)
    out, n = gu.gpu_sample(b)
    st = {}
    gu.compare_sample(out, n, ref, st)
    # at V = 128256 a token's residual mass is ~1e-5 of the total, so about one
    # draw in eight lands within 1e-6 of a CDF boundary (the oracle flags 31 of
    # these 256 sequences, all at the draw, none at an accept test); nearly all
    # still agree
    print("headline flagged:", st)
    assert st["flagged"] <= 0.15 * b.B
    assert int((ref["near_accept"] >= 0).sum()) == 0
    assert st["flagged_mismatch"] <= 2
    acc = (n.astype(np.float64)).mean() / b.K
    assert 0.4 < acc < 0.95


@pytest.mark.parametrize("B,K", [(1, 4), (1, 8), (8, 4), (8, 8), (64, 4), (64, 8)])
def test_sample_controlled(orc, B, K):
    b = gen.config_controlled(B, K)
    ref = gu.oracle_sample(orc, b)
    out, n = gu.gpu_sample(b)
    gu.compare_sample(out, n, ref)


def test_sample_controlled_b512_k8_sampled(orc):
    """The largest sweep case, B=512, K=8, V=151936 (2.8 GB of logits), in one
    call; every fourth sequence against the oracle (the generator seeds each
    sequence on its own, so a subset reproduces the same rows)."""
    b = gen.config_controlled(512, 8)
    out, n = gu.gpu_sample(b)
    sel = list(range(0, 512, 4))
    sub = gen.config_controlled(512, 8, seqs=sel)
    ref = gu.oracle_sample(orc, sub)
    assert (sub.target == b.target[sel]).all()
    gu.compare_sample(out[sel], n[sel], ref)
    assert (n >= 0).all()


def test_sample_controlled_b512_expected_tokens(orc):
    """B=512, K=4, V=151936: parity, and the device's mean tokens per step over
    many uniform draws matches each sequence's exact conditional expectation
    sum_j prod_{t<j} min(1, p_t(x_t)/q_t(x_t)) (the closed form of "Expected
    speedup" holds per sequence with per-position acceptances)."""
    b = gen.config_controlled(512, 4)
    ref = gu.oracle_sample(orc, b)
    out, n = gu.gpu_sample(b)
    gu.compare_sample(out, n, ref)
    # per-position acceptance min(1, p_t(x_t)/q_t(x_t)) at every position (oracle softmax)
    acc = np.empty((b.B, b.K))
    for i in range(b.B):
        for t in range(b.K):
            x = b.draft_tokens[i, t]
            p = orc.softmax(gen.as_f64(b.target[i, t], b.dtype), b.T)
            q = orc.softmax(gen.as_f64(b.draft[i, t], b.dtype), b.T)
            acc[i, t] = min(1.0, p[x] / q[x])
    cond = np.ones(b.B)
    prod = np.ones(b.B)
    for t in range(b.K):
        prod = prod * acc[:, t]
        cond += prod
    rng = np.random.default_rng(77)
    tgt = gu.dev_tensor(b.target, b.dtype)
    dft = gu.dev_tensor(b.draft, b.dtype)
    tok = gu.i32(b.draft_tokens)
    R = 64
    tot = np.zeros(b.B)
    for _ in range(R):
        uni = gu.f32(rng.random((b.B, b.K + 1, 2), dtype=np.float32))
        _, nn = sv.spec_verify_sample(tgt, dft, tok, uni, b.T)
        tot += nn.cpu().numpy() + 1.0
    mean = tot / R
    # per-sequence variance of (n+1) <= (K+1)^2/4; average over B sequences
    se = np.sqrt(((b.K + 1) ** 2 / 4.0) / R / b.B)
    assert abs(mean.mean() - cond.mean()) < 5 * se


def test_sample_draft_probs(orc):
    rng = np.random.default_rng(5)
    B, K, V, T = 32, 5, 5000, 0.9
    z = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    q = sp_softmax(z[:, :K].astype(np.float64) / T + 0.5 * rng.standard_normal((B, K, V)), axis=-1)
    q = q.astype(np.float32)
    q[0, 0, :] = 0.0
    q[0, 0, 3] = 1.0               # one-hot draft
    tok = np.array([[np.searchsorted(np.cumsum(q[b, t].astype(np.float64)), rng.random() * q[b, t].sum())
                     for t in range(K)] for b in range(B)], np.int32).clip(0, V - 1)
    tok[0, 0] = 3
    uni = rng.random((B, K + 1, 2), dtype=np.float32)
    batch = gen.ChainBatch(B, K, V, T, "f32", z, q, True, tok, uni)
    ref = gu.oracle_sample(orc, batch)
    out, n = gu.gpu_sample(batch)
    gu.compare_sample(out, n, ref)


@pytest.mark.parametrize("dt,ddt,V", [("f32", "f32", 1001), ("bf16", "bf16", 1003), ("bf16", "f32", 4096),
                                      ("f32", "bf16", 2000), ("bf16", "bf16", 8)])
def test_sample_ragged_and_mixed(orc, dt, ddt, V):
    rng = np.random.default_rng(V)
    B, K, T = 24, 3, 1.1
    z = rng.standard_normal((B, K + 1, V))
    y = z[:, :K] + 0.5 * rng.standard_normal((B, K, V))
    tgt = gen.f32_to_bf16_bits(z) if dt == "bf16" else z.astype(np.float32)
    dft = gen.f32_to_bf16_bits(y) if ddt == "bf16" else y.astype(np.float32)
    yq = gen.as_f64(dft, ddt)
    g = -np.log(-np.log(rng.random((B, K, V))))
    tok = np.argmax(yq / T + g, axis=-1).astype(np.int32)
    uni = rng.random((B, K + 1, 2), dtype=np.float32)
    ref = orc.verify_sample(tgt, dt, dft, ddt, False, tok, uni, T)
    out, n = sv.spec_verify_sample(gu.dev_tensor(tgt, dt), gu.dev_tensor(dft, ddt), gu.i32(tok), gu.f32(uni), T)
    gu.compare_sample(out.cpu().numpy(), n.cpu().numpy(), ref)


def test_sample_k0_is_bonus_only(orc):
    rng = np.random.default_rng(9)
    B, V = 40, 3000
    z = rng.standard_normal((B, 1, V)).astype(np.float32)
    uni = rng.random((B, 1, 2), dtype=np.float32)
    batch = gen.ChainBatch(B, 0, V, 1.0, "f32", z, np.zeros((B, 0, V), np.float32), False,
                           np.zeros((B, 0), np.int32), uni)
    ref = gu.oracle_sample(orc, batch)
    out, n = gu.gpu_sample(batch)
    gu.compare_sample(out, n, ref)
    assert (n == 0).all()


def test_sample_invalid_rows(orc):
    rng = np.random.default_rng(4)
    B, K, V, T = 10, 3, 4096, 1.0
    z = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    y = z[:, :K].copy()
    tok = np.argmax(y, axis=-1).astype(np.int32)
    uni = np.full((B, K + 1, 2), 0.5, np.float32)
    z[1, 0, 3] = np.nan
    y[2, 1, 4] = np.nan
    z[3, 3, :] = -np.inf           # bonus row without finite entry
    z[4, 2, 1] = np.inf
    tok[5, 0] = V
    z[6, 0, :] = -np.inf
    batch = gen.ChainBatch(B, K, V, T, "f32", z, y, False, tok, uni)
    ref = gu.oracle_sample(orc, batch)
    out, n = gu.gpu_sample(batch)
    assert (n == ref["num_accepted"]).all() and (out == ref["out_tokens"]).all()
    assert (ref["num_accepted"][[1, 2, 3, 4, 5, 6]] == -1).all()
    assert (ref["num_accepted"][[0, 7, 8, 9]] == K).all()


@pytest.mark.parametrize("cfg", ["zipf", "headline"])
def test_debug_residual_rows(orc, cfg):
    if cfg == "zipf":
        b = gen.config_zipf(T=1.0, B=4)
    else:
        b = gen.config_headline(seqs=[0, 1, 2])
    tgt = gu.dev_tensor(b.target, b.dtype)
    dft = gu.dev_tensor(b.draft, b.dtype)
    tok = gu.i32(b.draft_tokens)
    uni = gu.f32(b.uniforms)
    for (bb, t) in [(0, 0), (1, 2), (b.B - 1, b.K)]:
        row, mass, _, _ = sv.spec_debug_residual(tgt, dft, tok, uni, b.T, bb, t)
        rrow, rmass = orc.residual_row(b.target, b.dtype, b.draft, b.dtype, False, b.T, bb, t)
        row = row.cpu().numpy().astype(np.float64)
        assert np.abs(row - rrow).max() < 1e-6
        assert abs(float(mass.cpu()[0]) - rmass) < 1e-6 * max(1.0, rmass)
        assert abs(row.sum() - 1.0) < 1e-4


# --- tree --------------------------------------------------------------------------

def test_tree_full_workload(orc):
    """B=128, N=64, V=128256 bf16, BFS tree [4,3,2,1] truncated to 64 nodes."""
    t = gen.config_tree()
    ro, rn, rp = orc.verify_tree_greedy(t.target, t.dtype, t.parents, t.node_tokens, t.max_depth)
    out, n, path = sv.spec_verify_tree_greedy(gu.dev_tensor(t.target, t.dtype), gu.i32(t.parents),
                                              gu.i32(t.node_tokens), t.max_depth)
    assert (n.cpu().numpy() == rn).all()
    assert (out.cpu().numpy() == ro).all()
    assert (path.cpu().numpy() == rp).all()
    assert rn.mean() > 1.0


def test_tree_random_small(orc):
    rng = np.random.default_rng(21)
    for trial in range(40):
        br = [int(x) for x in rng.integers(1, 4, size=rng.integers(1, 5))]
        parents = gen.bfs_tree(br, max_nodes=int(rng.integers(2, 40)))
        N = len(parents)
        depth = int(gen.tree_depths(parents).max())
        B, V = 7, int(rng.choice([5, 64, 1000, 1003]))
        rows = rng.integers(-2, 3, size=(B, N, V)).astype(np.float32)
        g = np.argmax(rows, axis=-1)
        tok = np.where(rng.random((B, N)) < 0.7, g[:, np.maximum(parents, 0)],
                       rng.integers(-1, V + 1, size=(B, N))).astype(np.int32)
        ro, rn, rp = orc.verify_tree_greedy(rows, "f32", parents, tok, depth)
        out, n, path = sv.spec_verify_tree_greedy(gu.f32(rows), gu.i32(parents), gu.i32(tok), depth)
        assert (n.cpu().numpy() == rn).all() and (out.cpu().numpy() == ro).all()
        assert (path.cpu().numpy() == rp).all()


def test_tree_bad_topology_and_nan(orc):
    rows = np.zeros((3, 4, 16), np.float32)
    rows[2, 0, 5] = np.nan
    tok = np.zeros((3, 4), np.int32)
    for parents, md in (([-1, 0, 5, 1], 2), ([0, 0, 1, 2], 3), ([-1, 0, 1, 2], 2)):
        ro, rn, _ = orc.verify_tree_greedy(rows, "f32", np.array(parents, np.int32), tok, md)
        out, n, _ = sv.spec_verify_tree_greedy(gu.f32(rows), gu.i32(parents), gu.i32(tok), md)
        assert (n.cpu().numpy() == rn).all() and (out.cpu().numpy() == ro).all()
        assert (rn == -1).all()
    ro, rn, _ = orc.verify_tree_greedy(rows, "f32", np.array([-1, 0, 1, 2], np.int32), tok, 3)
    out, n, _ = sv.spec_verify_tree_greedy(gu.f32(rows), gu.i32([-1, 0, 1, 2]), gu.i32(tok), 3)
    assert (n.cpu().numpy() == rn).all() and (out.cpu().numpy() == ro).all()
    assert rn.tolist() == [3, 3, -1]


@pytest.mark.parametrize("dt,V", [("bf16", 32768), ("f32", 4000)])
def test_greedy_controlled_agreement(orc, dt, V):
    """Greedy rule on drafts that copy the target argmax w.p. 0.8: long accepted
    prefixes, so rows well past position 0 are needed (and rows after the first
    mismatch are not)."""
    b = gen.config_greedy(B=96, V=V, K=7, dtype=dt)
    ro, rn = orc.verify_greedy(b.target, b.dtype, b.draft_tokens)
    out, n = sv.spec_verify_greedy(gu.dev_tensor(b.target, b.dtype), gu.i32(b.draft_tokens))
    np.testing.assert_array_equal(n.cpu().numpy(), rn)
    np.testing.assert_array_equal(out.cpu().numpy(), ro)
    assert rn.mean() > 2


def _tree_case(rng, parents, B, V, dtype, match=0.7):
    N = len(parents)
    z = rng.standard_normal((B, N, V))
    rows = gen.f32_to_bf16_bits(z) if dtype == "bf16" else z.astype(np.float32)
    g = np.argmax(gen.as_f64(rows, dtype), axis=-1)
    tok = np.where(rng.random((B, N)) < match, g[:, np.maximum(parents, 0)],
                   rng.integers(0, V, size=(B, N))).astype(np.int32)
    return rows, tok


def _tree_check(orc, rows, dtype, parents, tok, depth):
    ro, rn, rp = orc.verify_tree_greedy(rows, dtype, parents, tok, depth)
    out, n, path = sv.spec_verify_tree_greedy(gu.dev_tensor(rows, dtype), gu.i32(parents), gu.i32(tok), depth)
    np.testing.assert_array_equal(n.cpu().numpy(), rn)
    np.testing.assert_array_equal(out.cpu().numpy(), ro)
    np.testing.assert_array_equal(path.cpu().numpy(), rp)
    return rn


@pytest.mark.parametrize("shape", ["chain48", "wide1024", "deep_bushy"])
def test_tree_pruned_shapes(orc, shape):
    """Dependency chains much deeper than the headline tree, and node counts up
    to the 1024-node limit (every node bit in use)."""
    rng = np.random.default_rng({"chain48": 1, "wide1024": 2, "deep_bushy": 3}[shape])
    if shape == "chain48":
        parents = gen.bfs_tree([1] * 47)            # 48 nodes in one chain
        rows, tok = _tree_case(rng, parents, 6, 4096, "bf16", match=0.97)
    elif shape == "wide1024":
        parents = gen.bfs_tree([32, 31], max_nodes=1024)
        rows, tok = _tree_case(rng, parents, 3, 2048, "bf16", match=0.9)
    else:
        parents = gen.bfs_tree([3, 2, 2, 2, 2, 2, 2], max_nodes=300)
        rows, tok = _tree_case(rng, parents, 5, 1000, "f32", match=0.8)
    depth = int(gen.tree_depths(parents).max())
    rn = _tree_check(orc, rows, "bf16" if shape != "deep_bushy" else "f32", parents, tok, depth)
    assert rn.max() >= 2


@pytest.mark.parametrize("B", [600, 2000])
def test_tree_many_sequences(orc, B):
    """More sequences than CTAs (several per finisher), and beyond the pruned
    kernel's per-finisher limit (the full-sweep path)."""
    rng = np.random.default_rng(B)
    parents = gen.bfs_tree([3, 2, 2], max_nodes=20)
    rows, tok = _tree_case(rng, parents, B, 256, "bf16")
    _tree_check(orc, rows, "bf16", parents, tok, int(gen.tree_depths(parents).max()))


def test_tree_nan_outside_accepted_nodes_is_ignored(orc):
    """Only accepted nodes' rows are read: a NaN in a rejected node's row does
    not invalidate the sequence; one in an accepted node's row does."""
    rng = np.random.default_rng(7)
    parents = gen.bfs_tree([2, 2])                  # 7 nodes: 0 | 1 2 | 3 4 5 6
    rows, tok = _tree_case(rng, parents, 4, 512, "f32", match=1.0)
    tok[:, 2] = (tok[:, 1] + 1) % 512                # node 2 (and 5, 6) rejected
    rows[0, 2, 17] = np.nan                          # rejected: ignored
    rows[1, 5, 3] = np.nan                           # rejected descendant: ignored
    rows[2, 3, 9] = np.nan                           # accepted leaf: invalid
    rn = _tree_check(orc, rows, "f32", parents, tok, 2)
    assert rn[0] >= 0 and rn[1] >= 0 and rn[2] == -1


def test_calls_finish_without_hitting_wait_bounds():
    """Every wait in the kernels is bounded (1 s); a call that silently ran into
    a bound would still be correct but slow.  The headline-sized call must take
    milliseconds, repeatedly."""
    import time
    b = gen.config_headline(seqs=list(range(64)))
    tgt, dft = gu.dev_tensor(b.target, b.dtype), gu.dev_tensor(b.draft, b.dtype)
    tok, uni = gu.i32(b.draft_tokens), gu.f32(b.uniforms)
    sv.spec_verify_sample(tgt, dft, tok, uni, b.T)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    t = gen.config_tree(seqs=list(range(16)), V=32768)
    ttgt, tpar, ttok = gu.dev_tensor(t.target, t.dtype), gu.i32(t.parents), gu.i32(t.node_tokens)
    sv.spec_verify_tree_greedy(ttgt, tpar, ttok, t.max_depth)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(5):
        _, n = sv.spec_verify_sample(tgt, dft, tok, uni, b.T)
        sv.spec_verify_greedy(tgt, tok)
        _, tn, _ = sv.spec_verify_tree_greedy(ttgt, tpar, ttok, t.max_depth)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 0.5
    assert (n.cpu().numpy() >= 0).all() and (tn.cpu().numpy() >= 0).all()


def test_non_default_stream(orc):
    b = gen.config_zipf(T=1.0, B=16, V=8192)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        tgt, dft = gu.f32(b.target), gu.f32(b.draft)
        out, n = sv.spec_verify_sample(tgt, dft, gu.i32(b.draft_tokens), gu.f32(b.uniforms), b.T)
    s.synchronize()
    ref = gu.oracle_sample(orc, b)
    gu.compare_sample(out.cpu().numpy(), n.cpu().numpy(), ref)


@pytest.mark.parametrize("K,V,probs", [(31, 4096, False), (20, 1003, False), (31, 2048, True)])
def test_sample_long_drafts(orc, K, V, probs):
    """Long drafts (up to the K = 31 limit: 63 rows per sequence, two per lane
    of the accept scan) with a near-perfect draft, so that deep positions and
    the bonus draw are reached; logits (fused path, and the scalar path for an
    odd V) and draft probabilities."""
    rng = np.random.default_rng(K * 7 + V)
    B, T = 12, 1.0
    z = rng.standard_normal((B, K + 1, V))
    y = z[:, :K] + 0.05 * rng.standard_normal((B, K, V))
    tgt = gen.f32_to_bf16_bits(z)
    if probs:
        dft = sp_softmax(gen.as_f64(gen.f32_to_bf16_bits(y), "bf16") / T, axis=-1).astype(np.float32)
        yq = np.log(np.maximum(dft.astype(np.float64), 1e-300))
    else:
        dft = gen.f32_to_bf16_bits(y)
        yq = gen.as_f64(dft, "bf16") / T
    g = -np.log(-np.log(rng.random((B, K, V))))
    tok = np.argmax(yq + g, axis=-1).astype(np.int32)
    uni = rng.random((B, K + 1, 2), dtype=np.float32)
    batch = gen.ChainBatch(B, K, V, T, "bf16", tgt, dft, probs, tok, uni)
    ref = gu.oracle_sample(orc, batch)
    out, n = gu.gpu_sample(batch)
    gu.compare_sample(out, n, ref)
    assert ref["num_accepted"].max() >= K // 2     # deep positions were reached
