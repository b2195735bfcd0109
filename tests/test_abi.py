"""The C-ABI library on the host (no GPU needed): it builds, loads, exports
every function include/spec_verify.h declares, sizes workspaces, and rejects
bad arguments before touching the device."""
import ctypes

import pytest

from speculative_decoding_verification_52_gb300 import binding as B
from speculative_decoding_verification_52_gb300 import build as build_mod


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return B.lib()


def test_exports_every_declared_symbol(L):
    names = B.declared_functions()
    assert {"spec_verify_sample", "spec_verify_greedy", "spec_verify_tree_greedy",
            "spec_workspace_bytes", "spec_debug_residual"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/spec_verify.h but not exported"


def test_workspace_sizes(L):
    # control block (32 B) + per-sequence counters and readiness flags (one
    # 32-byte block each), per-sequence info (32 B), residual block sums
    # (ceil(V/256) floats per sequence), and one 16-byte partial per sweep
    # unit (rows x at most ceil(V/2048) slices)
    def al(x, a):
        return (x + a - 1) // a * a
    B_, K_, V_ = 256, 5, 128256
    zero = al(32 + 32 * B_, 32)   # 8 flag words per sequence
    bsum = al(zero + 32 * B_, 16)
    part = al(bsum + 4 * B_ * (-(-V_ // 256)), 16)
    fused = al(part + B_ * (2 * K_ + 1) * 63 * 16, 256)
    assert L.spec_workspace_bytes(B_, K_, V_) == fused   # larger than the greedy chain's pruned layout here
    fused1 = al(al(al(al(32 + 32, 32) + 32, 16) + 4, 16) + 16, 256)
    # the greedy chain's pruned layout: control block + counters + FIFO + done flags, then partials
    assert L.spec_workspace_bytes(1, 0, 8) == max(fused1, al(al(256 + 4, 256) + 64, 256))
    # tree: max(full sweep partials, pruned-kernel layout with at most ceil(V/4096) slices)
    nodes, smax = 128 * 64, -(-128256 // 4096)
    fifo = al(128 + 4 * nodes, 128)
    pruned = al(al(fifo + 4 * 128 * 63 * smax + 4 * 128, 256) + nodes * smax * 8 * 8, 256)
    assert L.spec_tree_workspace_bytes(128, 64, 128256) == max(128 * 64 * 63 * 8, pruned)
    for bad in [(-1, 4, 10), (1, -1, 10), (1, 32, 10), (1, 4, 0)]:
        assert L.spec_workspace_bytes(*bad) == 0
    assert L.spec_tree_workspace_bytes(1, 0, 10) == 0
    assert L.spec_tree_workspace_bytes(1, 1025, 10) == 0


def _sample(L, **kw):
    a = dict(target=1 << 20, tdt=1, draft=1 << 21, ddt=1, kind=0, tokens=1 << 22, uni=1 << 23, T=0.7,
             B=2, K=3, V=64, out=1 << 24, nacc=1 << 25, ws=1 << 26, wsb=1 << 20)
    a.update(kw)
    P = ctypes.c_void_p
    return L.spec_verify_sample(P(a["target"]), a["tdt"], P(a["draft"]), a["ddt"], a["kind"], P(a["tokens"]),
                                P(a["uni"]), a["T"], a["B"], a["K"], a["V"], P(a["out"]), P(a["nacc"]),
                                P(a["ws"]), a["wsb"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(K=32), B.SPEC_ERR_INVALID_ARG),
    (dict(K=-1), B.SPEC_ERR_INVALID_ARG),
    (dict(V=0), B.SPEC_ERR_INVALID_ARG),
    (dict(B=-3), B.SPEC_ERR_INVALID_ARG),
    (dict(T=float("nan")), B.SPEC_ERR_INVALID_ARG),
    (dict(T=-1.0), B.SPEC_ERR_INVALID_ARG),
    (dict(T=float("inf")), B.SPEC_ERR_INVALID_ARG),
    (dict(tdt=7), B.SPEC_ERR_INVALID_ARG),
    (dict(kind=1, ddt=1), B.SPEC_ERR_INVALID_ARG),   # probabilities must be f32
    (dict(target=0), B.SPEC_ERR_INVALID_ARG),
    (dict(tokens=0), B.SPEC_ERR_INVALID_ARG),
    (dict(uni=0), B.SPEC_ERR_INVALID_ARG),
    (dict(ws=0), B.SPEC_ERR_WORKSPACE),
    (dict(wsb=8), B.SPEC_ERR_WORKSPACE),
    (dict(ws=(1 << 26) + 4), B.SPEC_ERR_WORKSPACE),   # misaligned
    (dict(T=1e-6), B.SPEC_ERR_UNSUPPORTED),
])
def test_sample_rejects_bad_arguments(L, kw, status):
    assert _sample(L, **kw) == status
    assert B.last_error()


def test_empty_batch_is_a_no_op(L):
    assert _sample(L, B=0, target=0, out=0, nacc=0, ws=0) == B.SPEC_OK
    P = ctypes.c_void_p
    assert L.spec_verify_greedy(None, 0, None, 0, 4, 100, None, None, None, 0, None) == B.SPEC_OK
    assert L.spec_verify_tree_greedy(None, 0, None, None, 0, 3, 100, 2, None, None, None, None, 0, None) == B.SPEC_OK


def test_greedy_and_tree_reject_bad_arguments(L):
    P = ctypes.c_void_p
    assert L.spec_verify_greedy(P(16), 0, P(32), 1, 40, 10, P(48), P(64), P(256), 1 << 20, None) == B.SPEC_ERR_INVALID_ARG
    assert L.spec_verify_greedy(P(16), 0, P(32), 1, 4, 10, P(48), P(64), P(256), 4, None) == B.SPEC_ERR_WORKSPACE
    tree = L.spec_verify_tree_greedy
    assert tree(P(16), 0, P(32), P(48), 1, 2000, 10, 3, P(64), P(80), None, P(256), 1 << 20, None) == B.SPEC_ERR_INVALID_ARG
    assert tree(P(16), 0, P(32), P(48), 1, 8, 10, 8, P(64), P(80), None, P(256), 1 << 20, None) == B.SPEC_ERR_INVALID_ARG
    assert tree(P(16), 0, None, P(48), 1, 8, 10, 3, P(64), P(80), None, P(256), 1 << 20, None) == B.SPEC_ERR_INVALID_ARG


def test_debug_residual_rejects_bad_position(L):
    P = ctypes.c_void_p
    f = L.spec_debug_residual
    args = [P(16), 0, P(32), 0, 0, P(48), P(64), 1.0, 2, 3, 10]
    assert f(*args, 2, 0, P(80), P(96), P(112), P(128), P(256), 1 << 20, None) == B.SPEC_ERR_INVALID_ARG
    assert f(*args, 0, 4, P(80), P(96), P(112), P(128), P(256), 1 << 20, None) == B.SPEC_ERR_INVALID_ARG


def test_status_strings(L):
    assert B.status_string(0) == "SPEC_OK"
    assert B.status_string(4) == "SPEC_ERR_WORKSPACE"
    assert B.status_string(99) == "SPEC_ERR_UNKNOWN"


def test_tree_mask_and_kv_commit_reject_bad_arguments(L):
    P = ctypes.c_void_p
    assert L.spec_tree_mask(P(16), 2, 0, P(32), P(48), None) == B.SPEC_ERR_INVALID_ARG
    assert L.spec_tree_mask(P(16), 2, 1025, P(32), P(48), None) == B.SPEC_ERR_INVALID_ARG
    assert L.spec_tree_mask(None, 2, 8, P(32), P(48), None) == B.SPEC_ERR_INVALID_ARG
    assert L.spec_tree_mask(None, 0, 8, None, None, None) == B.SPEC_OK
    kv = L.spec_kv_commit
    assert kv(P(16), P(32), P(48), None, P(64), 2, 8, 0, 0, 64, P(80), None) == B.SPEC_ERR_INVALID_ARG
    assert kv(P(16), P(32), P(48), P(96), P(64), 2, 8, 4, 0, 64, P(80), None) == B.SPEC_ERR_INVALID_ARG
    assert kv(P(16), P(32), P(48), None, P(64), 2, 8, 4, 0, 0, P(80), None) == B.SPEC_ERR_INVALID_ARG
    assert kv(P(16), None, P(48), None, P(64), 2, 8, 4, 0, 64, P(80), None) == B.SPEC_ERR_INVALID_ARG
    assert kv(None, None, None, None, None, 0, 8, 4, 0, 64, None, None) == B.SPEC_OK


def test_row_stats_rejects_bad_arguments(L):
    P, F = ctypes.c_void_p, ctypes.c_float
    rs = L.spec_row_stats
    ok = dict(t=P(16), td=B.SPEC_BF16, d=P(32), dd=B.SPEC_BF16, kind=B.SPEC_DRAFT_LOGITS, T=F(0.7), Bn=2, K=3,
              V=64, a=P(48), k=P(64), v=P(80))

    def call(**kw):
        a = {**ok, **kw}
        return rs(a["t"], a["td"], a["d"], a["dd"], a["kind"], a["T"], a["Bn"], a["K"], a["V"], a["a"], a["k"],
                  a["v"], None)

    assert call(T=F(0.0)) == B.SPEC_ERR_INVALID_ARG
    assert call(T=F(float("nan"))) == B.SPEC_ERR_INVALID_ARG
    assert call(T=F(1e-5)) == B.SPEC_ERR_UNSUPPORTED
    assert call(K=-1) == B.SPEC_ERR_INVALID_ARG
    assert call(K=B.SPEC_MAX_K + 1) == B.SPEC_ERR_INVALID_ARG
    assert call(V=0) == B.SPEC_ERR_INVALID_ARG
    assert call(td=7) == B.SPEC_ERR_INVALID_ARG
    assert call(kind=B.SPEC_DRAFT_PROBS) == B.SPEC_ERR_INVALID_ARG       # probabilities must be f32
    assert call(kind=5) == B.SPEC_ERR_INVALID_ARG
    assert call(a=None) == B.SPEC_ERR_INVALID_ARG
    assert call(d=None) == B.SPEC_ERR_INVALID_ARG
    assert call(V=1_000_000) == B.SPEC_ERR_UNSUPPORTED       # slice pair beyond the limit
    assert call(Bn=0, t=None, d=None, a=None) == B.SPEC_OK
    assert call(K=0, t=None, d=None, a=None) == B.SPEC_OK


def test_tree_draft_rejects_bad_arguments(L):
    P, F = ctypes.c_void_p, ctypes.c_float
    td = L.spec_tree_draft
    assert td(P(16), B.SPEC_BF16, P(32), 2, 0, 64, 4, F(1.0), P(48), P(64), None) == B.SPEC_ERR_INVALID_ARG
    assert td(P(16), B.SPEC_BF16, P(32), 2, 1025, 64, 4, F(1.0), P(48), P(64), None) == B.SPEC_ERR_INVALID_ARG
    assert td(P(16), B.SPEC_BF16, P(32), 2, 8, 0, 4, F(1.0), P(48), P(64), None) == B.SPEC_ERR_INVALID_ARG
    assert td(P(16), B.SPEC_BF16, P(32), 2, 8, 64, 0, F(1.0), P(48), P(64), None) == B.SPEC_ERR_INVALID_ARG
    assert td(P(16), B.SPEC_BF16, P(32), 2, 8, 64, 17, F(1.0), P(48), P(64), None) == B.SPEC_ERR_INVALID_ARG
    assert td(P(16), B.SPEC_BF16, P(32), 2, 8, 64, 4, F(0.0), P(48), P(64), None) == B.SPEC_ERR_INVALID_ARG
    assert td(P(16), B.SPEC_BF16, P(32), 2, 8, 64, 4, F(1e-6), P(48), P(64), None) == B.SPEC_ERR_UNSUPPORTED
    assert td(P(16), 9, P(32), 2, 8, 64, 4, F(1.0), P(48), P(64), None) == B.SPEC_ERR_INVALID_ARG
    assert td(P(16), B.SPEC_BF16, None, 2, 8, 64, 4, F(1.0), P(48), P(64), None) == B.SPEC_ERR_INVALID_ARG
    assert td(None, B.SPEC_BF16, None, 0, 8, 64, 4, F(1.0), None, None, None) == B.SPEC_OK


def test_debug_stall_rejects_bad_arguments(L):
    P, F = ctypes.c_void_p, ctypes.c_float
    ds = L.spec_debug_stall

    def call(stall_b=0, timeout_us=2000, T=0.7, Bn=4):
        return ds(P(16), B.SPEC_BF16, P(32), B.SPEC_BF16, B.SPEC_DRAFT_LOGITS, P(48), P(64), F(T), Bn, 3, 64,
                  stall_b, timeout_us, P(80), P(96), P(112), 1 << 20, None)

    assert call(stall_b=-1) == B.SPEC_ERR_INVALID_ARG
    assert call(stall_b=4) == B.SPEC_ERR_INVALID_ARG          # outside the batch
    assert call(timeout_us=10) == B.SPEC_ERR_INVALID_ARG      # below 100 us
    assert call(timeout_us=2_000_000) == B.SPEC_ERR_INVALID_ARG
    assert call(T=0.0) == B.SPEC_ERR_INVALID_ARG              # the hook needs the sampling rule
