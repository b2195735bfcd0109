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


@pytest.mark.parametrize("E,vec", [(64, True), (4096, True), (6, False), (1000, False)])
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
