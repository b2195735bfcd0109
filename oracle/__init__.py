"""Double-precision CPU oracle for batched speculative-decoding verification.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the product package.  The
arithmetic lives in ``spec_oracle.c`` (plain C, double precision, scalar loops
in vocabulary order); this module only compiles it with gcc and marshals numpy
arrays through ctypes.  It shares no code with the CUDA library.

Pins (tests that tie the oracle to something other than itself) are in
``tests/test_oracle_pins.py``, ``tests/test_oracle_law.py`` and
``tests/test_golden.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
NEAR_TOL = 1e-6


def build(force: bool = False) -> str:
    """Compile spec_oracle.c into liboracle.so (strict IEEE double: no fast-math,
    no FMA contraction, so x86 and Arm hosts evaluate the same expressions)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            L.orc_softmax.argtypes = [P, I, D, P]
            L.orc_softmax.restype = I
            L.orc_residual.argtypes = [P, P, I, P]
            L.orc_residual.restype = D
            L.orc_icdf.argtypes = [P, I, D, D, P]
            L.orc_icdf.restype = I
            L.orc_accept.argtypes = [D, D, D]
            L.orc_accept.restype = I
            L.orc_argmax.argtypes = [P, I]
            L.orc_argmax.restype = I
            L.orc_verify_greedy.argtypes = [P, I, P, I, I, I, P, P]
            L.orc_verify_greedy.restype = I
            L.orc_verify_sample.argtypes = [P, I, P, I, I, P, P, D, I, I, I, P, P, P, P, D, P]
            L.orc_verify_sample.restype = I
            L.orc_residual_row.argtypes = [P, I, P, I, I, D, I, I, I, I, P, P]
            L.orc_residual_row.restype = I
            L.orc_verify_tree_greedy.argtypes = [P, I, P, P, I, I, I, I, P, P, P]
            L.orc_tree_mask.argtypes = [P, I, I, P, P]
            L.orc_tree_mask.restype = None
            L.orc_kv_commit.argtypes = [P, P, P, P, P, I, I, I, I, ctypes.c_size_t, P]
            L.orc_kv_commit.restype = None
            L.orc_row_stats.argtypes = [P, I, P, I, I, D, I, I, I, P, P, P]
            L.orc_row_stats.restype = I
            L.orc_verify_tree_greedy.restype = I
            L.orc_tree_draft.argtypes = [P, I, P, I, I, I, D, I, P, P]
            L.orc_tree_draft.restype = I
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dt(dtype) -> int:
    return BF16 if dtype in ("bf16", BF16) else F32


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# ---- primitives (double in, double out) ------------------------------------

def softmax(z, T: float):
    """Temperature softmax of one row; None if the row is invalid."""
    z = _c(z, np.float64)
    p = np.empty_like(z)
    rc = lib().orc_softmax(_ptr(z), z.size, float(T), _ptr(p))
    return None if rc else p


def residual(p, q):
    """(w, R): w = max(0, p - q) elementwise, R = sum w."""
    p = _c(p, np.float64)
    q = _c(q, np.float64)
    w = np.empty_like(p)
    R = lib().orc_residual(_ptr(p), _ptr(q), p.size, _ptr(w))
    return w, R


def icdf(w, R: float, u: float):
    """(v, gap): inverse-CDF draw in vocabulary order."""
    w = _c(w, np.float64)
    gap = np.zeros(1)
    v = lib().orc_icdf(_ptr(w), w.size, float(R), float(u), _ptr(gap))
    return v, float(gap[0])


def accept(a: float, c: float, u: float) -> bool:
    return bool(lib().orc_accept(float(a), float(c), float(u)))


def argmax(z) -> int:
    z = _c(z, np.float64)
    return lib().orc_argmax(_ptr(z), z.size)


# ---- batched verification ---------------------------------------------------

def _raw(x, dtype):
    return _c(x, np.uint16) if _dt(dtype) == BF16 else _c(x, np.float32)


def verify_greedy(target, dtype, draft_tokens):
    """Greedy chain verification.  target [B,K+1,V]; returns (out_tokens, num_accepted)."""
    t = _raw(target, dtype)
    B, W, V = t.shape
    K = W - 1
    tok = _c(draft_tokens, np.int32).reshape(B, K)
    out = np.empty((B, W), np.int32)
    n = np.empty(B, np.int32)
    rc = lib().orc_verify_greedy(_ptr(t), _dt(dtype), _ptr(tok), B, K, V, _ptr(out), _ptr(n))
    if rc:
        raise MemoryError("oracle allocation failed")
    return out, n


def verify_sample(target, target_dtype, draft, draft_dtype, draft_is_probs, draft_tokens,
                  uniforms, T: float, tol: float = NEAR_TOL):
    """Sampling-mode chain verification.

    Returns dict(out_tokens [B,K+1], num_accepted [B], near_accept [B] (first
    position whose accept test was within ``tol`` of flipping, else -1),
    near_cdf [B] (replacement draw within ``tol`` of a CDF boundary),
    ratio [B,K] (p/q at evaluated positions, NaN elsewhere))."""
    t = _raw(target, target_dtype)
    B, W, V = t.shape
    K = W - 1
    if draft_is_probs:
        d = _c(draft, np.float32)
        ddt = F32
    else:
        d = _raw(draft, draft_dtype)
        ddt = _dt(draft_dtype)
    if K > 0:
        d = d.reshape(B, K, V)
    tok = _c(draft_tokens, np.int32).reshape(B, K)
    uni = _c(uniforms, np.float32).reshape(B, W, 2)
    out = np.empty((B, W), np.int32)
    n = np.empty(B, np.int32)
    na = np.empty(B, np.int32)
    nc = np.empty(B, np.int32)
    ratio = np.empty((B, max(K, 1)), np.float64)
    rc = lib().orc_verify_sample(_ptr(t), _dt(target_dtype), _ptr(d), ddt, int(bool(draft_is_probs)),
                                 _ptr(tok), _ptr(uni), float(T), B, K, V, _ptr(out), _ptr(n),
                                 _ptr(na), _ptr(nc), float(tol), _ptr(ratio))
    if rc:
        raise MemoryError("oracle allocation failed")
    return dict(out_tokens=out, num_accepted=n, near_accept=na, near_cdf=nc,
                ratio=ratio[:, :K])


def residual_row(target, target_dtype, draft, draft_dtype, draft_is_probs, T, b, t):
    """(w/R as float64 [V], R) for sequence b at position t (t == K: the bonus row p_K)."""
    tg = _raw(target, target_dtype)
    B, W, V = tg.shape
    K = W - 1
    if draft_is_probs:
        d = _c(draft, np.float32)
        ddt = F32
    else:
        d = _raw(draft, draft_dtype)
        ddt = _dt(draft_dtype)
    row = np.empty(V, np.float64)
    mass = np.zeros(1)
    rc = lib().orc_residual_row(_ptr(tg), _dt(target_dtype), _ptr(d), ddt, int(bool(draft_is_probs)),
                                float(T), K, V, int(b), int(t), _ptr(row), _ptr(mass))
    if rc:
        return None, None
    return row, float(mass[0])


def verify_tree_greedy(target, dtype, parents, node_tokens, max_depth: int):
    """Greedy tree verification.  target [B,N,V]; returns (out_tokens, num_accepted, out_path)."""
    t = _raw(target, dtype)
    B, N, V = t.shape
    par = _c(parents, np.int32)
    tok = _c(node_tokens, np.int32).reshape(B, N)
    W = max_depth + 1
    out = np.empty((B, W), np.int32)
    n = np.empty(B, np.int32)
    path = np.empty((B, W), np.int32)
    rc = lib().orc_verify_tree_greedy(_ptr(t), _dt(dtype), _ptr(par), _ptr(tok), B, N, V, int(max_depth),
                                      _ptr(out), _ptr(n), _ptr(path))
    if rc:
        raise MemoryError("oracle allocation failed")
    return out, n, path


def tree_mask(parents):
    """Ancestor masks of per-sequence trees.  parents [B, N] (or [N] for one
    tree); returns (masks [B, N, ceil(N/32)] uint32, status [B] int32)."""
    par = np.atleast_2d(_c(parents, np.int32))
    B, N = par.shape
    NW = (N + 31) // 32
    out = np.empty((B, N, NW), np.uint32)
    st = np.empty(B, np.int32)
    lib().orc_tree_mask(_ptr(par), B, N, _ptr(out), _ptr(st))
    return out, st


def kv_commit(cache, lengths, scratch, path, count):
    """Append the selected scratch entries to the cache (a copy is returned).
    cache [B, Lmax, ...], scratch [B, N, ...] (same trailing shape and dtype),
    lengths [B], path [B, W] or None, count [B].  Returns (cache, new_lengths)."""
    cache = np.array(cache, copy=True, order="C")
    scratch = np.ascontiguousarray(scratch)
    B, Lmax = cache.shape[:2]
    N = scratch.shape[1]
    E = cache[0, 0].nbytes if Lmax else scratch[0, 0].nbytes
    ln = _c(lengths, np.int32)
    cnt = _c(count, np.int32)
    pth = None if path is None else _c(path, np.int32)
    W = 0 if pth is None else pth.shape[1]
    newl = np.empty(B, np.int32)
    lib().orc_kv_commit(_ptr(cache), _ptr(ln), _ptr(scratch), None if pth is None else _ptr(pth), _ptr(cnt),
                        B, Lmax, N, W, E, _ptr(newl))
    return cache, newl


def row_stats(target, target_dtype, draft, draft_dtype, draft_is_probs, T: float):
    """Per drafted position: (alpha = sum min(p, q), KL(q || p), TV), each [B, K]."""
    t = _raw(target, target_dtype)
    B, W, V = t.shape
    K = W - 1
    d = _raw(draft, "f32" if draft_is_probs else draft_dtype)
    out = [np.empty((B, K), np.float64) for _ in range(3)]
    rc = lib().orc_row_stats(_ptr(t), _dt(target_dtype), _ptr(d), _dt("f32" if draft_is_probs else draft_dtype),
                             1 if draft_is_probs else 0, float(T), B, K, V, *[_ptr(o) for o in out])
    if rc:
        raise MemoryError("oracle allocation failed")
    return tuple(out)


def tree_draft(draft, dtype, parents, T: float, max_children: int = 16):
    """Top-k tree drafting: (node_tokens [B, N] int32, node_logq [B, N] f64, rc);
    rc = 1 for a malformed topology or a node with more than max_children children."""
    d = _raw(draft, dtype)
    B, N, V = d.shape
    par = np.ascontiguousarray(parents, dtype=np.int32)
    tok = np.empty((B, N), np.int32)
    lq = np.empty((B, N), np.float64)
    rc = lib().orc_tree_draft(_ptr(d), _dt(dtype), _ptr(par), B, N, V, float(T), int(max_children), _ptr(tok),
                               _ptr(lq))
    if rc == 2:
        raise MemoryError("oracle allocation failed")
    return tok, lq, rc
