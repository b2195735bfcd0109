"""Tree attention masks and KV commit-on-accept on the GPU against the oracle,
bit for bit, through the C ABI."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import speculative_decoding_verification_52_gb300 as sv
from speculative_decoding_verification_52_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


def _mask_gpu(par):
    m, st = sv.spec_tree_mask(gu.i32(par))
    return m.cpu().numpy().view(np.uint32), st.cpu().numpy()


def test_tree_mask_page_example_and_static_trees(orc):
    for par in ([-1, 0, 0, 1, 1, 2, 2], gen.bfs_tree([4, 3, 2, 1], 64), gen.bfs_tree([32, 31], 1024),
                np.arange(-1, 1023), [-1]):
        par = np.asarray(par, np.int32)
        m, st = _mask_gpu(par)
        rm, rst = orc.tree_mask(par)
        np.testing.assert_array_equal(st, rst)
        np.testing.assert_array_equal(m, rm)


@pytest.mark.parametrize("N", [2, 31, 32, 33, 70, 100, 257, 500, 600])
def test_tree_mask_random_per_sequence_trees(orc, N):
    rng = np.random.default_rng(N)
    B = 37
    par = np.empty((B, N), np.int32)
    par[:, 0] = -1
    for i in range(1, N):
        par[:, i] = rng.integers(0, i, size=B)
    par[3, 5 % N] = 7 % N if N > 1 else -1       # may break the rule (parent >= child)
    par[9, 0] = 0                                 # breaks it (the root has a parent)
    m, st = _mask_gpu(par)
    rm, rst = orc.tree_mask(par)
    np.testing.assert_array_equal(st, rst)
    np.testing.assert_array_equal(m, rm)
    assert rst[9] == -1


@pytest.mark.parametrize("E,vec", [(64, True), (4096, True), (20000, True), (6, False), (1000, False)])
def test_kv_commit_matches_oracle(orc, E, vec):
    rng = np.random.default_rng(E)
    B, Lmax, N, W = 24, 40, 9, 6
    cache = rng.integers(0, 256, size=(B, Lmax, E), dtype=np.uint8)
    scratch = rng.integers(0, 256, size=(B, N, E), dtype=np.uint8)
    lengths = rng.integers(0, Lmax - 3, size=B).astype(np.int32)
    lengths[0] = Lmax - 2                          # overflows with count 3
    count = rng.integers(-1, W + 1, size=B).astype(np.int32)
    count[0] = 3
    path = rng.integers(0, N, size=(B, W)).astype(np.int32)
    path[1, 0] = N                                 # a slot outside the scratch buffer
    count[1] = max(count[1], 1)
    for use_path in (True, False):
        pth = path if use_path else None
        cnt = count if use_path else np.minimum(count, N)
        ref_cache, ref_len = orc.kv_commit(cache, lengths, scratch, pth, cnt)
        c = torch.from_numpy(cache.copy()).to(gu.DEV)
        newl = sv.spec_kv_commit(c, gu.i32(lengths), torch.from_numpy(scratch).to(gu.DEV), gu.i32(cnt),
                                 path=gu.i32(pth) if use_path else None)
        np.testing.assert_array_equal(newl.cpu().numpy(), ref_len)
        np.testing.assert_array_equal(c.cpu().numpy(), ref_cache)


def test_commit_after_tree_verification(orc):
    """The accepted path of a tree verification drives the commit: the cache
    gains exactly the accepted nodes' entries, in path order."""
    t = gen.config_tree(seqs=list(range(8)), V=4096)
    _, n, path = sv.spec_verify_tree_greedy(gu.dev_tensor(t.target, t.dtype), gu.i32(t.parents),
                                            gu.i32(t.node_tokens), t.max_depth)
    _, rn, rpath = orc.verify_tree_greedy(t.target, t.dtype, t.parents, t.node_tokens, t.max_depth)
    np.testing.assert_array_equal(path.cpu().numpy(), rpath)
    rng = np.random.default_rng(3)
    B, Lmax, E = t.B, 32, 256
    cache = rng.integers(0, 256, size=(B, Lmax, E), dtype=np.uint8)
    scratch = rng.integers(0, 256, size=(B, t.N, E), dtype=np.uint8)
    lengths = np.full(B, 10, np.int32)
    ref_cache, ref_len = orc.kv_commit(cache, lengths, scratch, rpath, rn)
    c = torch.from_numpy(cache.copy()).to(gu.DEV)
    newl = sv.spec_kv_commit(c, gu.i32(lengths), torch.from_numpy(scratch).to(gu.DEV), n, path=path)
    np.testing.assert_array_equal(newl.cpu().numpy(), ref_len)
    np.testing.assert_array_equal(c.cpu().numpy(), ref_cache)
    assert (ref_len - lengths == rn).all()


# --- acceptance statistics --------------------------------------------------------
# Tolerances (fp32 path against the double oracle): every summed term carries the
# ex2 approximation's relative error (a few 1e-7) and the normalisers one more
# such factor each, so alpha and TV (sums of terms <= 1 that total <= 1) are
# within 2e-6; KL combines O(10)-sized log-domain terms whose fp32 rounding is
# ~1e-6 each, so it is checked to 1e-5 absolute plus 1e-5 relative.
ALPHA_TOL, KL_ABS, KL_REL = 2e-6, 1e-5, 1e-5


def _softmax_probs(draft, dtype, T):
    y = gen.as_f64(draft, dtype) / T
    y -= y.max(-1, keepdims=True)
    e = np.exp(y)
    return (e / e.sum(-1, keepdims=True)).astype(np.float32)


def _stats_pair(orc, target, tdt, draft, ddt, T, probs=False):
    g = sv.spec_row_stats(gu.dev_tensor(target, tdt), gu.dev_tensor(draft, ddt), T,
                          draft_kind="probs" if probs else "logits")
    g = [x.cpu().numpy().astype(np.float64) for x in g]
    r = orc.row_stats(target, tdt, draft, ddt, probs, T)
    for name, gv, rv in zip(("alpha", "kl", "tv"), g, r):
        np.testing.assert_array_equal(np.isnan(gv), np.isnan(rv), err_msg=f"{name}: invalid rows differ")
        ok = ~np.isnan(rv)
        if name == "kl":
            np.testing.assert_allclose(gv[ok], rv[ok], rtol=KL_REL, atol=KL_ABS, err_msg=name)
        else:
            np.testing.assert_allclose(gv[ok], rv[ok], rtol=0, atol=ALPHA_TOL, err_msg=name)
    return g, r


@pytest.mark.parametrize("V,dtype", [(128256, "bf16"), (32000, "f32"), (1000, "bf16"), (999, "bf16"),
                                     (37, "f32"), (77777, "bf16"), (8, "f32"), (40000, "f32"),
                                     (65544, "bf16")])
def test_row_stats_match_oracle(orc, V, dtype):
    """The streaming kernel (aligned rows of more than 64 KB per pair; 65544
    bf16 ends in an 8-element chunk) and the cluster kernel (shorter rows: a
    cluster of one; odd V: element loads, clusters of 8, 4 and 1)."""
    b = gen.gaussian_chain(6, V, 5, sigma=0.445, T=0.7, dtype=dtype, seed=52_310 + V)
    _stats_pair(orc, b.target, dtype, b.draft, dtype, 0.7)


def test_row_stats_zipf_and_mixed_dtypes(orc):
    b = gen.config_zipf(seqs=range(6))
    _stats_pair(orc, b.target, "f32", b.draft, "f32", 1.0)
    h = gen.config_headline(seqs=range(3), V=4096)
    d32 = gen.as_f64(h.draft, "bf16").astype(np.float32)
    _stats_pair(orc, h.target, "bf16", d32, "f32", 0.7)
    t32 = gen.as_f64(h.target, "bf16").astype(np.float32)
    _stats_pair(orc, t32, "f32", h.draft, "bf16", 0.7)


@pytest.mark.parametrize("tdt", ["bf16", "f32"])
def test_row_stats_draft_probabilities(orc, tdt):
    h = gen.config_headline(seqs=range(4), V=32000, K=4)
    target = h.target if tdt == "bf16" else gen.as_f64(h.target, "bf16").astype(np.float32)
    q = _softmax_probs(h.draft, "bf16", 0.7)
    q[1, 2, :] = 0.0
    q[1, 2, 17] = 1.0                      # one-hot draft: alpha = p(17), KL = -log p(17)
    q[2, 0, ::3] = 0.0                     # zeros skipped by the KL sum
    g, r = _stats_pair(orc, target, tdt, q, "f32", 0.7, probs=True)
    assert g[0][1, 2] < 1e-3


def test_row_stats_identical_and_controlled(orc):
    """Bit-identical draft rows give alpha = 1, KL = 0, TV = 0 (V = 151936)."""
    b = gen.config_controlled(4, 4, seqs=range(4))
    g, _ = _stats_pair(orc, b.target, "bf16", b.draft, "bf16", 1.0)
    cp = b.meta["copied"]
    assert cp.any() and (~cp).any()
    np.testing.assert_allclose(g[0][cp], 1.0, atol=ALPHA_TOL)
    assert (g[1][cp] == 0.0).all()


@pytest.mark.parametrize("V", [4096, 40000])
def test_row_stats_invalid_rows(orc, V):
    """V=4096 through the cluster kernel (one CTA per pair), V=40000 through
    the streaming kernel, with the NaN in the row's last chunk."""
    b = gen.gaussian_chain(4, V, 3, sigma=0.5, T=1.0, dtype="f32", seed=52_390)
    t, d = b.target.copy(), b.draft.copy()
    t[0, 1, V - 100] = np.nan
    d[1, 0, 5] = np.inf
    t[2, 2, :] = -np.inf
    t[3, 0, :] = -np.inf
    t[3, 0, 9] = 0.5                       # one finite entry: valid (p is one-hot)
    g, r = _stats_pair(orc, t, "f32", d, "f32", 1.0)
    assert np.isnan(g[0][0, 1]) and np.isnan(g[0][1, 0]) and np.isnan(g[0][2, 2])
    assert np.isfinite(g[0]).sum() == 12 - 3
    q = _softmax_probs(b.draft, "f32", 1.0)
    q[0, 0, 3] = -1e-3
    q[1, 1, 8] = np.nan
    g, _ = _stats_pair(orc, b.target, "f32", q, "f32", 1.0, probs=True)
    assert np.isnan(g[0][0, 0]) and np.isnan(g[0][1, 1]) and np.isfinite(g[0]).sum() == 10


def test_row_stats_full_headline_batch(orc):
    """B=256, V=128256, K=5 bf16, T=0.7 in the benchmark's launch configuration;
    every position against the oracle, and the mean alpha of the workload."""
    b = gen.config_headline()
    g, r = _stats_pair(orc, b.target, "bf16", b.draft, "bf16", 0.7)
    assert abs(r[0].mean() - 0.75) < 0.01


def test_row_stats_empty():
    t = torch.zeros((3, 1, 64), dtype=torch.bfloat16, device=gu.DEV)
    d = torch.zeros((3, 0, 64), dtype=torch.bfloat16, device=gu.DEV)
    a, k, tv = sv.spec_row_stats(t, d, 1.0)
    assert a.shape == (3, 0)


# --- top-k tree drafting ------------------------------------------------------------
# Tokens are compared bit for bit (the selection compares logits exactly).  log q
# = ln2 (z c - fl(M c) - log2 S) in fp32: log2 S (|.| <= ~20) and the final
# difference carry ~1 ulp of ~20 each, ~4e-6 in all, so 2e-5 absolute.
LOGQ_ATOL = 2e-5


def _draft_pair(orc, draft, dtype, parents, T, max_children):
    tok, lq = sv.spec_tree_draft(gu.dev_tensor(draft, dtype), gu.i32(parents), T, max_children)
    tok, lq = tok.cpu().numpy(), lq.cpu().numpy().astype(np.float64)
    rt, rl, _ = orc.tree_draft(draft, dtype, parents, T, max_children)
    np.testing.assert_array_equal(tok, rt)
    np.testing.assert_array_equal(np.isnan(lq), np.isnan(rl))
    ok = ~np.isnan(rl)
    np.testing.assert_allclose(lq[ok], rl[ok], rtol=1e-6, atol=LOGQ_ATOL)
    return tok, lq


@pytest.mark.parametrize("dtype,V,branching,N,mc", [
    ("bf16", 128256, (4, 3, 2, 1), 64, 4),
    ("f32", 32000, (3, 3, 2), None, 3),
    ("bf16", 999, (4, 3, 2, 1), 64, 4),      # rows not 16-byte aligned: element loads
    ("f32", 37, (1, 1, 1, 1, 1), None, 1),   # a chain: the argmax at every step
    ("bf16", 4096, (16, 2), None, 16),
    ("f32", 5000, (2, 2, 2, 2, 2, 2), None, 8),
])
def test_tree_draft_matches_oracle(orc, dtype, V, branching, N, mc):
    par, draft = gen.config_tree_draft(B=5, V=V, branching=branching, N=N, dtype=dtype, seed=52_910 + V)
    _draft_pair(orc, draft, dtype, par, 0.8, mc)


def test_tree_draft_ties_and_small_vocab(orc):
    rng = np.random.default_rng(7)
    par = gen.bfs_tree([5, 2], None)
    z = (np.round(rng.standard_normal((6, len(par), 700)) * 2) / 2).astype(np.float32)   # many exact ties
    _draft_pair(orc, z, "f32", par, 1.0, 5)
    _draft_pair(orc, gen._store(z.astype(np.float64), "bf16"), "bf16", par, 1.3, 8)
    tiny = rng.standard_normal((3, 4, 2)).astype(np.float32)          # 3 children, V = 2
    _draft_pair(orc, tiny, "f32", np.array([-1, 0, 0, 0], np.int32), 1.0, 3)


def test_tree_draft_invalid_rows_and_topology(orc):
    par = gen.bfs_tree([3, 2], None)
    rng = np.random.default_rng(8)
    z = rng.standard_normal((4, len(par), 256)).astype(np.float32)
    z[0, 1, 7] = np.nan
    z[1, 0, :] = -np.inf
    z[2, 2, 5] = np.inf
    _draft_pair(orc, z, "f32", par, 1.0, 3)
    bad = par.copy()
    bad[4] = 6                                           # a parent after its child
    tok, lq = _draft_pair(orc, z, "f32", bad, 1.0, 3)
    assert (tok == -1).all()
    tok, _ = _draft_pair(orc, z, "f32", par, 1.0, 2)     # the root has 3 children > 2
    assert (tok == -1).all()


def test_tree_draft_full_workload_sampled(orc):
    """B=128, N=64, V=128256 bf16 in the benchmark's launch configuration; every
    8th sequence against the oracle."""
    par, draft = gen.config_tree_draft()
    tok, lq = sv.spec_tree_draft(gu.dev_tensor(draft, "bf16"), gu.i32(par), 0.7, 4)
    tok, lq = tok.cpu().numpy(), lq.cpu().numpy().astype(np.float64)
    sel = np.arange(0, 128, 8)
    rt, rl, _ = orc.tree_draft(np.ascontiguousarray(draft[sel]), "bf16", par, 0.7, 4)
    np.testing.assert_array_equal(tok[sel], rt)
    np.testing.assert_allclose(lq[sel], rl, rtol=1e-6, atol=LOGQ_ATOL)


def test_draft_mask_verify_pipeline(orc):
    """Draft a tree, build its attention mask, verify it: a target equal to the
    draft accepts the whole depth along the first children; a target whose
    root row prefers the root's second token accepts through the second child."""
    par, draft = gen.config_tree_draft(B=6, V=8192, seed=52_920)
    d = gu.dev_tensor(draft, "bf16")
    ptr = gu.i32(par)
    tok, _ = sv.spec_tree_draft(d, ptr, 1.0, 4)
    masks, st = sv.spec_tree_mask(ptr)
    rm, _ = orc.tree_mask(par)
    np.testing.assert_array_equal(masks.cpu().numpy().view(np.uint32)[0], rm[0])
    depth = gen.tree_depths(par)
    out, n, path = sv.spec_verify_tree_greedy(d, ptr, tok, int(depth.max()))
    assert (n.cpu().numpy() == depth.max()).all()
    first = {p: min(i for i in range(len(par)) if par[i] == p) for p in set(par[1:].tolist())}
    node = 0
    for dd in range(int(depth.max())):
        node = first[node]
        assert (path.cpu().numpy()[:, dd] == node).all()
    # a target whose root row ranks the root's second child's token first
    t = draft.copy()
    tnp = tok.cpu().numpy()
    for b in range(6):
        row = gen.as_f64(t[b, 0], "bf16")
        row[tnp[b, 2]] = row.max() + 1.0
        t[b, 0] = gen._store(row, "bf16")
    out, n, path = sv.spec_verify_tree_greedy(gu.dev_tensor(t, "bf16"), ptr, tok, int(depth.max()))
    ro, rn, rp = orc.verify_tree_greedy(t, "bf16", par, tnp, int(depth.max()))
    np.testing.assert_array_equal(path.cpu().numpy(), rp)
    assert (rp[:, 0] == 2).all()


def test_tree_draft_large_tree_multi_chunk(orc):
    """A 700-node tree (the kernel scans the parent array in chunks of 256 to
    find a node's children): random parents, at most 8 children per node."""
    rng = np.random.default_rng(70)
    N = 700
    par = np.empty(N, np.int32)
    par[0] = -1
    kids = np.zeros(N, np.int64)
    for i in range(1, N):
        while True:
            p = int(rng.integers(0, i))
            if kids[p] < 8:
                break
        par[i] = p
        kids[p] += 1
    z = rng.standard_normal((3, N, 512)).astype(np.float32)
    _draft_pair(orc, z, "f32", par, 0.9, 8)
    _draft_pair(orc, gen._store(z.astype(np.float64), "bf16"), "bf16", par, 0.9, 8)
