"""Thin Python binding of the C ABI in include/spec_verify.h.

Argument marshalling only: torch tensors are checked for device, dtype and
layout, outputs and the caller-side workspace are allocated with torch when
not supplied, and the C entry points of libspecverify.so are called with raw
pointers and the current CUDA stream.  Every step of the verification runs in
the library's CUDA kernels; there is no fallback of any kind -- if the library
is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecverify.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "spec_verify.h")

SPEC_OK, SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED, SPEC_ERR_CUDA, SPEC_ERR_WORKSPACE = range(5)
SPEC_F32, SPEC_BF16 = 0, 1
SPEC_DRAFT_LOGITS, SPEC_DRAFT_PROBS = 0, 1
SPEC_MAX_K = 31
SPEC_MAX_TREE_NODES = 1024

_lock = threading.Lock()
_lib = None


class SpecError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {status_string(status)}: {msg}")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libspecverify.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            L.spec_workspace_bytes.argtypes = [I, I, I]
            L.spec_workspace_bytes.restype = Z
            L.spec_tree_workspace_bytes.argtypes = [I, I, I]
            L.spec_tree_workspace_bytes.restype = Z
            L.spec_verify_sample.argtypes = [P, I, P, I, I, P, P, F, I, I, I, P, P, P, Z, P]
            L.spec_verify_sample.restype = I
            L.spec_verify_sample_noalloc.argtypes = [P, I, P, I, I, P, P, F, I, I, I, P, P, P]
            L.spec_verify_sample_noalloc.restype = I
            L.spec_verify_greedy.argtypes = [P, I, P, I, I, I, P, P, P, Z, P]
            L.spec_verify_greedy.restype = I
            L.spec_verify_tree_greedy.argtypes = [P, I, P, P, I, I, I, I, P, P, P, P, Z, P]
            L.spec_verify_tree_greedy.restype = I
            L.spec_debug_residual.argtypes = [P, I, P, I, I, P, P, F, I, I, I, I, I, P, P, P, P, P, Z, P]
            L.spec_debug_residual.restype = I
            L.spec_debug_stall.argtypes = [P, I, P, I, I, P, P, F, I, I, I, I, ctypes.c_uint, P, P, P, Z, P]
            L.spec_debug_stall.restype = I
            L.spec_tree_mask.argtypes = [P, I, I, P, P, P]
            L.spec_tree_mask.restype = I
            L.spec_kv_commit.argtypes = [P, P, P, P, P, I, I, I, I, Z, P, P]
            L.spec_kv_commit.restype = I
            L.spec_row_stats.argtypes = [P, I, P, I, I, F, I, I, I, P, P, P, P]
            L.spec_row_stats.restype = I
            L.spec_tree_draft.argtypes = [P, I, P, I, I, I, I, F, P, P, P]
            L.spec_tree_draft.restype = I
            L.spec_profile_begin.argtypes = [I]
            L.spec_profile_begin.restype = I
            L.spec_profile_end.argtypes = [P, P, P]
            L.spec_profile_end.restype = I
            L.spec_status_string.argtypes = [I]
            L.spec_status_string.restype = ctypes.c_char_p
            L.spec_last_error.argtypes = []
            L.spec_last_error.restype = ctypes.c_char_p
            _lib = L
    return _lib


def declared_functions() -> list[str]:
    """Names of the functions include/spec_verify.h declares."""
    with open(HEADER) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_]+)\s*\(", text)))


def status_string(status: int) -> str:
    return lib().spec_status_string(int(status)).decode()


def last_error() -> str:
    return lib().spec_last_error().decode()


def _check(fn: str, status: int):
    if status != SPEC_OK:
        raise SpecError(fn, status, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"unsupported dtype {t.dtype}: use torch.bfloat16 or torch.float32")


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def spec_workspace_bytes(B: int, K: int, V: int) -> int:
    return int(lib().spec_workspace_bytes(B, K, V))


def spec_tree_workspace_bytes(B: int, N: int, V: int) -> int:
    return int(lib().spec_tree_workspace_bytes(B, N, V))


def workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def _outputs(B, W, device, out_tokens, num_accepted):
    if out_tokens is None:
        out_tokens = torch.empty((B, W), dtype=torch.int32, device=device)
    if num_accepted is None:
        num_accepted = torch.empty((B,), dtype=torch.int32, device=device)
    _dev(out_tokens, "out_tokens")
    _dev(num_accepted, "num_accepted")
    return out_tokens, num_accepted


def spec_verify_sample(target_logits, draft, draft_tokens, uniforms, temperature, *,
                       draft_kind: str = "logits", out_tokens=None, num_accepted=None,
                       workspace_buf=None, stream=None):
    """Sampling-mode verification.  target_logits [B,K+1,V] (bf16/f32),
    draft [B,K,V] (logits: bf16/f32; probs: f32), draft_tokens [B,K] int32,
    uniforms [B,K+1,2] f32.  Returns (out_tokens [B,K+1], num_accepted [B])."""
    _dev(target_logits, "target_logits")
    B, W, V = target_logits.shape
    K = W - 1
    kind = SPEC_DRAFT_PROBS if draft_kind == "probs" else SPEC_DRAFT_LOGITS
    for t, n in ((draft, "draft"), (draft_tokens, "draft_tokens"), (uniforms, "uniforms")):
        if t is not None:
            _dev(t, n)
    ddt = _dtype_code(draft) if draft is not None else SPEC_F32
    out_tokens, num_accepted = _outputs(B, W, target_logits.device, out_tokens, num_accepted)
    if workspace_buf is None:
        workspace_buf = workspace(spec_workspace_bytes(B, K, V), target_logits.device)
    st = lib().spec_verify_sample(_ptr(target_logits), _dtype_code(target_logits), _ptr(draft), ddt, kind,
                                  _ptr(draft_tokens), _ptr(uniforms), float(temperature), B, K, V,
                                  _ptr(out_tokens), _ptr(num_accepted), _ptr(workspace_buf),
                                  workspace_buf.numel(), _stream(stream))
    _check("spec_verify_sample", st)
    return out_tokens, num_accepted


def spec_verify_sample_noalloc(target_logits, draft, draft_tokens, uniforms, temperature, *,
                               draft_kind: str = "logits", out_tokens=None, num_accepted=None, stream=None):
    """spec_verify_sample with the library's fixed scratch instead of a
    workspace.  Pass out_tokens / num_accepted to keep the call free of any
    allocation (otherwise they are allocated here)."""
    _dev(target_logits, "target_logits")
    B, W, V = target_logits.shape
    K = W - 1
    kind = SPEC_DRAFT_PROBS if draft_kind == "probs" else SPEC_DRAFT_LOGITS
    for t, n in ((draft, "draft"), (draft_tokens, "draft_tokens"), (uniforms, "uniforms")):
        if t is not None:
            _dev(t, n)
    ddt = _dtype_code(draft) if draft is not None else SPEC_F32
    out_tokens, num_accepted = _outputs(B, W, target_logits.device, out_tokens, num_accepted)
    st = lib().spec_verify_sample_noalloc(_ptr(target_logits), _dtype_code(target_logits), _ptr(draft), ddt, kind,
                                          _ptr(draft_tokens), _ptr(uniforms), float(temperature), B, K, V,
                                          _ptr(out_tokens), _ptr(num_accepted), _stream(stream))
    _check("spec_verify_sample_noalloc", st)
    return out_tokens, num_accepted


def spec_verify_greedy(target_logits, draft_tokens, *, out_tokens=None, num_accepted=None,
                       workspace_buf=None, stream=None):
    """Greedy verification.  Returns (out_tokens [B,K+1], num_accepted [B])."""
    _dev(target_logits, "target_logits")
    B, W, V = target_logits.shape
    K = W - 1
    if draft_tokens is not None:
        _dev(draft_tokens, "draft_tokens")
    out_tokens, num_accepted = _outputs(B, W, target_logits.device, out_tokens, num_accepted)
    if workspace_buf is None:
        workspace_buf = workspace(spec_workspace_bytes(B, K, V), target_logits.device)
    st = lib().spec_verify_greedy(_ptr(target_logits), _dtype_code(target_logits), _ptr(draft_tokens), B, K, V,
                                  _ptr(out_tokens), _ptr(num_accepted), _ptr(workspace_buf),
                                  workspace_buf.numel(), _stream(stream))
    _check("spec_verify_greedy", st)
    return out_tokens, num_accepted


def spec_verify_tree_greedy(target_logits, parents, node_tokens, max_depth: int, *, with_path: bool = True,
                            out_tokens=None, num_accepted=None, out_path=None, workspace_buf=None,
                            stream=None):
    """Greedy tree verification.  target_logits [B,N,V], parents [N] int32,
    node_tokens [B,N] int32.  Returns (out_tokens, num_accepted, out_path|None)."""
    _dev(target_logits, "target_logits")
    _dev(parents, "parents")
    _dev(node_tokens, "node_tokens")
    B, N, V = target_logits.shape
    W = max_depth + 1
    out_tokens, num_accepted = _outputs(B, W, target_logits.device, out_tokens, num_accepted)
    if with_path and out_path is None:
        out_path = torch.empty((B, W), dtype=torch.int32, device=target_logits.device)
    if workspace_buf is None:
        workspace_buf = workspace(spec_tree_workspace_bytes(B, N, V), target_logits.device)
    st = lib().spec_verify_tree_greedy(_ptr(target_logits), _dtype_code(target_logits), _ptr(parents),
                                       _ptr(node_tokens), B, N, V, int(max_depth), _ptr(out_tokens),
                                       _ptr(num_accepted), _ptr(out_path), _ptr(workspace_buf),
                                       workspace_buf.numel(), _stream(stream))
    _check("spec_verify_tree_greedy", st)
    return out_tokens, num_accepted, out_path


def spec_debug_residual(target_logits, draft, draft_tokens, uniforms, temperature, debug_b: int, debug_t: int,
                        *, draft_kind: str = "logits", stream=None):
    """The device's normalised replacement distribution at (debug_b, debug_t).
    Returns (row [V] f32, mass [1] f32, out_tokens, num_accepted)."""
    _dev(target_logits, "target_logits")
    B, W, V = target_logits.shape
    K = W - 1
    dev = target_logits.device
    row = torch.full((V,), float("nan"), dtype=torch.float32, device=dev)
    mass = torch.zeros((1,), dtype=torch.float32, device=dev)
    out_tokens, num_accepted = _outputs(B, W, dev, None, None)
    ws = workspace(spec_workspace_bytes(B, K, V), dev)
    kind = SPEC_DRAFT_PROBS if draft_kind == "probs" else SPEC_DRAFT_LOGITS
    ddt = _dtype_code(draft) if draft is not None else SPEC_F32
    st = lib().spec_debug_residual(_ptr(target_logits), _dtype_code(target_logits), _ptr(draft), ddt, kind,
                                   _ptr(draft_tokens), _ptr(uniforms), float(temperature), B, K, V, int(debug_b),
                                   int(debug_t), _ptr(row), _ptr(mass), _ptr(out_tokens), _ptr(num_accepted),
                                   _ptr(ws), ws.numel(), _stream(stream))
    _check("spec_debug_residual", st)
    return row, mass, out_tokens, num_accepted


def spec_debug_stall(target_logits, draft, draft_tokens, uniforms, temperature, stall_b: int, timeout_us: int, *,
                     stream=None):
    """Test hook: spec_verify_sample with short wait limits while one
    sequence's scan waits for a unit that never comes.  Returns
    (out_tokens, num_accepted); every sequence should read -2."""
    _dev(target_logits, "target_logits")
    B, W, V = target_logits.shape
    K = W - 1
    out_tokens, num_accepted = _outputs(B, W, target_logits.device, None, None)
    ws = workspace(spec_workspace_bytes(B, K, V), target_logits.device)
    st = lib().spec_debug_stall(_ptr(target_logits), _dtype_code(target_logits), _ptr(draft), _dtype_code(draft),
                                SPEC_DRAFT_LOGITS, _ptr(draft_tokens), _ptr(uniforms), float(temperature), B, K, V,
                                int(stall_b), int(timeout_us), _ptr(out_tokens), _ptr(num_accepted), _ptr(ws),
                                ws.numel(), _stream(stream))
    _check("spec_debug_stall", st)
    return out_tokens, num_accepted


def spec_tree_mask(parents, *, masks=None, status=None, stream=None):
    """Ancestor masks.  parents [B, N] (or [N]) int32 on the device.  Returns
    (masks [B, N, ceil(N/32)] int32 holding the uint32 bit words, status [B])."""
    _dev(parents, "parents")
    par = parents if parents.dim() == 2 else parents.unsqueeze(0)
    par = par.contiguous()
    B, N = par.shape
    NW = (N + 31) // 32
    if masks is None:
        masks = torch.empty((B, N, NW), dtype=torch.int32, device=par.device)
    if status is None:
        status = torch.empty((B,), dtype=torch.int32, device=par.device)
    st = lib().spec_tree_mask(_ptr(par), B, N, _ptr(masks), _ptr(status), _stream(stream))
    _check("spec_tree_mask", st)
    return masks, status


def spec_kv_commit(cache, lengths, scratch, count, *, path=None, new_lengths=None, stream=None):
    """Append the selected scratch entries to the cache in place.  cache
    [B, Lmax, ...], scratch [B, N, ...] (same trailing shape and dtype),
    lengths / count [B] int32, path [B, W] int32 or None.  Returns new_lengths."""
    for t, n in ((cache, "cache"), (lengths, "lengths"), (scratch, "scratch"), (count, "count")):
        _dev(t, n)
    B, Lmax = cache.shape[:2]
    N = scratch.shape[1]
    E = cache[0, 0].numel() * cache.element_size() if Lmax else scratch[0, 0].numel() * scratch.element_size()
    W = 0
    if path is not None:
        _dev(path, "path")
        W = path.shape[1]
    if new_lengths is None:
        new_lengths = torch.empty((B,), dtype=torch.int32, device=cache.device)
    st = lib().spec_kv_commit(_ptr(cache), _ptr(lengths), _ptr(scratch), _ptr(path), _ptr(count), B, Lmax, N, W, E,
                              _ptr(new_lengths), _stream(stream))
    _check("spec_kv_commit", st)
    return new_lengths


def spec_row_stats(target_logits, draft, temperature, *, draft_kind: str = "logits", alpha=None, kl=None,
                   tv=None, stream=None):
    """Per-position acceptance statistics.  target_logits [B,K+1,V] (bf16/f32),
    draft [B,K,V] (logits: bf16/f32; probs: f32).  Returns (alpha, kl, tv), each
    [B,K] f32: sum min(p,q), KL(q||p), TV(p,q)."""
    _dev(target_logits, "target_logits")
    _dev(draft, "draft")
    B, W, V = target_logits.shape
    K = W - 1
    kind = SPEC_DRAFT_PROBS if draft_kind == "probs" else SPEC_DRAFT_LOGITS
    outs = []
    for o, n in ((alpha, "alpha"), (kl, "kl"), (tv, "tv")):
        if o is None:
            o = torch.empty((B, K), dtype=torch.float32, device=target_logits.device)
        _dev(o, n)
        outs.append(o)
    st = lib().spec_row_stats(_ptr(target_logits), _dtype_code(target_logits), _ptr(draft), _dtype_code(draft), kind,
                              float(temperature), B, K, V, _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]),
                              _stream(stream))
    _check("spec_row_stats", st)
    return tuple(outs)


def spec_tree_draft(draft_logits, parents, temperature, max_children: int, *, node_tokens=None, node_logq=None,
                    stream=None):
    """Top-k tree drafting.  draft_logits [B,N,V] (bf16/f32), parents [N] int32.
    Returns (node_tokens [B,N] int32, node_logq [B,N] f32)."""
    _dev(draft_logits, "draft_logits")
    _dev(parents, "parents")
    B, N, V = draft_logits.shape
    if node_tokens is None:
        node_tokens = torch.empty((B, N), dtype=torch.int32, device=draft_logits.device)
    if node_logq is None:
        node_logq = torch.empty((B, N), dtype=torch.float32, device=draft_logits.device)
    _dev(node_tokens, "node_tokens")
    _dev(node_logq, "node_logq")
    st = lib().spec_tree_draft(_ptr(draft_logits), _dtype_code(draft_logits), _ptr(parents), B, N, V,
                               int(max_children), float(temperature), _ptr(node_tokens), _ptr(node_logq),
                               _stream(stream))
    _check("spec_tree_draft", st)
    return node_tokens, node_logq


def spec_profile_begin(max_calls: int):
    _check("spec_profile_begin", lib().spec_profile_begin(int(max_calls)))


def spec_profile_end():
    """(sweep_ms_total, finish_ms_total, calls) over the recorded calls."""
    a, b, n = ctypes.c_float(), ctypes.c_float(), ctypes.c_int()
    _check("spec_profile_end", lib().spec_profile_end(ctypes.byref(a), ctypes.byref(b), ctypes.byref(n)))
    return a.value, b.value, n.value
