"""The seeded generators: bf16 rounding, per-sequence reproducibility, and the
structure each workload asks for."""
import numpy as np
import torch

from speculative_decoding_verification_52_gb300 import inputs as gen


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100_000) * 10.0 ** rng.integers(-3, 4, 100_000),
                        [0.0, -0.0, 1.0, -2.5, 65504.0, 1e-30]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (gen.f32_to_bf16_bits(x) == ref).all()
    back = gen.bf16_bits_to_f64(ref)
    assert (back == torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()).all()


def test_subset_reproduces_full_batch():
    full = gen.config_headline(B=6, V=1024, seqs=None)
    part = gen.config_headline(B=6, V=1024, seqs=[4, 1])
    for i, b in enumerate([4, 1]):
        assert (part.target[i] == full.target[b]).all()
        assert (part.draft[i] == full.draft[b]).all()
        assert (part.draft_tokens[i] == full.draft_tokens[b]).all()
        assert (part.uniforms[i] == full.uniforms[b]).all()


def test_uniforms_in_unit_interval():
    b = gen.config_zipf(B=8, V=512)
    assert b.uniforms.dtype == np.float32
    assert (b.uniforms >= 0).all() and (b.uniforms < 1).all()


def test_headline_acceptance_near_target(orc):
    b = gen.config_headline(seqs=[0, 1])
    acc = []
    for i in range(b.B):
        for t in range(b.K):
            p = orc.softmax(gen.as_f64(b.target[i, t], b.dtype), b.T)
            q = orc.softmax(gen.as_f64(b.draft[i, t], b.dtype), b.T)
            acc.append(np.minimum(p, q).sum())
    assert abs(np.mean(acc) - 0.75) < 0.01


def test_controlled_copies_are_bit_identical():
    b = gen.config_controlled(B=8, K=4, V=2048)
    c = b.meta["copied"]
    for i in range(b.B):
        for t in range(b.K):
            same = (b.draft[i, t] == b.target[i, t]).all()
            assert same == c[i, t]
    assert 0.5 < c.mean() < 1.0


def test_tree_topology_and_tokens():
    parents = gen.bfs_tree([4, 3, 2, 1], 64)
    assert len(parents) == 64 and parents[0] == -1
    assert all(0 <= parents[i] < i for i in range(1, 64))
    assert gen.tree_depths(parents).max() == 4
    # 1 + 4 + 12 + 24 + 24 = 65 nodes, truncated: the last depth-4 leaf goes
    assert len(gen.bfs_tree([4, 3, 2, 1])) == 65
    t = gen.config_tree(B=4, V=4096)
    rows = gen.as_f64(t.target, t.dtype)
    match = [t.node_tokens[b, j] == np.argmax(rows[b, t.parents[j]]) for b in range(4) for j in range(1, 64)]
    assert 0.55 < np.mean(match) < 0.85


def test_greedy_copy_flags_predict_the_oracle(orc):
    """The greedy workload's copy draws fix how many drafts the greedy rule
    accepts (leading copied positions), which the benchmark uses to count the
    rows the rule needs."""
    b = gen.config_greedy(B=24, V=2048, K=6)
    out, n = orc.verify_greedy(b.target, b.dtype, b.draft_tokens)
    f = b.meta["copied"]
    lead = np.where(f.all(axis=1), f.shape[1], np.argmin(f, axis=1))
    np.testing.assert_array_equal(n, lead)
    assert 0 < n.mean() < b.K


def test_tree_copy_flags_predict_the_oracle(orc):
    """Tree workload: a node is accepted iff every node on its root path copied
    its parent's argmax; the oracle's chosen depth is the deepest such node."""
    t = gen.config_tree(seqs=list(range(12)), V=1024)
    _, n, path = orc.verify_tree_greedy(t.target, t.dtype, t.parents, t.node_tokens, t.max_depth)
    acc = np.zeros((t.B, t.N), dtype=bool)
    acc[:, 0] = True
    for j in range(1, t.N):
        acc[:, j] = acc[:, t.parents[j]] & t.copied[:, j]
    depth = gen.tree_depths(t.parents)
    np.testing.assert_array_equal(n, [depth[acc[i]].max() for i in range(t.B)])
    for i in range(t.B):
        assert all(acc[i, p] for p in path[i] if p >= 0)
