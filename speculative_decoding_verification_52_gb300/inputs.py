"""Seeded synthetic inputs for batched draft-token verification.

This module only *generates* inputs: target logits, draft logits or
probabilities, draft tokens, uniforms and tree topologies.  It holds none of
the verification arithmetic (no softmax normaliser, no acceptance test, no
residual), so both the CUDA path and the double-precision oracle can be fed
from it without sharing any of the method's code.

Every generator draws from numpy's PCG64, seeded per sequence with
``SeedSequence([seed, b])``: sequence ``b`` of a batch is identical whether
the whole batch or only a subset of sequences is generated, which is what
lets a test or the CPU baseline regenerate a bounded sample of a large batch.

bf16 tensors are produced by rounding float32 to bfloat16 (round to nearest
even) here, once, and are handed out as raw ``uint16`` bit patterns; both
sides read exactly those bits.

Draft tokens are drawn with the Gumbel-max trick, ``argmax(y / T + G)`` with
``G = -log(-log U)``, which is an exact sample from ``softmax(y / T)`` of the
(rounded) draft logits ``y`` -- this plays the role of the draft model's
proposal step ("Speculative decoding and EAGLE", section "The concept", step
1) without computing any normaliser.

Workload shapes follow the pages' settings: vocabularies of 32k-152k entries,
draft lengths K = 4-8, batches 1-512 ("Speculative decoding and EAGLE",
section "Expected speedup"; "Speculative decoding: draft, verify, repeat",
section "What determines the speed").
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F32 = "f32"
BF16 = "bf16"

# Draft-noise scale for the B=256, V=128256, K=5, T=0.7 workload.  Chosen so
# that the mean per-position acceptance sum_v min(p, q) over all rows is 0.75;
# tests/golden/calibrate_sigma.py recomputes it with the oracle and
# tests/test_inputs.py checks the resulting acceptance on a sample.
SIGMA_B256_V128K = 0.445


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float values to bfloat16 (nearest, ties to even); return uint16 bits."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    b = f.view(np.uint32)
    # b + 0x7FFF + lsb stays below 2^32 for every finite or infinite value
    # (the largest, 0xFF800000, gains at most 0x8000)
    r = (b >> 16) & 1
    r += 0x7FFF
    r += b
    r >>= 16
    return r.astype(np.uint16)


def bf16_bits_to_f64(h: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float64 (exact)."""
    u = np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def as_f64(values: np.ndarray, dtype: str) -> np.ndarray:
    """The exact float64 value of a generated tensor (bf16 bits or float32)."""
    if dtype == BF16:
        return bf16_bits_to_f64(values)
    return np.asarray(values, dtype=np.float32).astype(np.float64)


def _store(x64: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == BF16:
        return f32_to_bf16_bits(x64)
    return np.asarray(x64, dtype=np.float32)


def _rng(seed: int, b: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(b)])))


def _gumbel_token(rng: np.random.Generator, y: np.ndarray, T: float) -> int:
    """One exact sample from softmax(y / T) by the Gumbel-max trick; T == 0 is argmax."""
    if T == 0.0:
        return int(np.argmax(y))
    u = rng.random(y.shape[-1])
    g = -np.log(-np.log(np.maximum(u, 1e-300)))
    return int(np.argmax(y / T + g))


@dataclass
class ChainBatch:
    """Inputs of one chain-verification call (shapes as the C ABI takes them)."""

    B: int
    K: int
    V: int
    T: float
    dtype: str                 # element type of target (and draft logits)
    target: np.ndarray         # [B, K+1, V]  uint16 bf16 bits or float32
    draft: np.ndarray          # [B, K, V]    same dtype as target (logits) or float32 probs
    draft_is_probs: bool
    draft_tokens: np.ndarray   # [B, K] int32
    uniforms: np.ndarray       # [B, K+1, 2] float32 in [0, 1)
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def draft_dtype(self) -> str:
        return F32 if self.draft_is_probs else self.dtype


@dataclass
class TreeBatch:
    """Inputs of one greedy tree-verification call."""

    B: int
    N: int
    V: int
    dtype: str
    target: np.ndarray         # [B, N, V] one logit row per tree node
    parents: np.ndarray        # [N] int32, parents[0] = -1, parents[i] < i
    node_tokens: np.ndarray    # [B, N] int32 (node 0's entry is ignored)
    max_depth: int
    name: str = ""
    copied: np.ndarray | None = None   # [B, N] bool: the generator set the token to the parent's argmax


def _uniforms(rng: np.random.Generator, K: int) -> np.ndarray:
    return rng.random((K + 1, 2), dtype=np.float32)


def gaussian_chain(B: int, V: int, K: int, sigma: float, T: float, dtype: str,
                   seed: int, seqs=None, scale: float = 1.0,
                   zipf_bias: float = 0.0, name: str = "") -> ChainBatch:
    """Target logits ~ scale*N(0,1) (+ optional Zipf-like bias -zipf_bias*log(rank)
    over a per-sequence random vocabulary permutation); draft logits = target +
    N(0, sigma^2); draft tokens sampled from softmax(draft/T)."""
    seqs = list(range(B)) if seqs is None else list(seqs)
    n = len(seqs)
    tgt = np.empty((n, K + 1, V), dtype=np.uint16 if dtype == BF16 else np.float32)
    dft = np.empty((n, K, V), dtype=tgt.dtype)
    tok = np.empty((n, K), dtype=np.int32)
    uni = np.empty((n, K + 1, 2), dtype=np.float32)
    for i, b in enumerate(seqs):
        rng = _rng(seed, b)
        z = scale * rng.standard_normal((K + 1, V))
        if zipf_bias:
            perm = rng.permutation(V)
            bias = np.empty(V)
            bias[perm] = -zipf_bias * np.log(np.arange(1, V + 1, dtype=np.float64))
            z = z + bias
        y = z[:K] + sigma * rng.standard_normal((K, V))
        tgt[i] = _store(z, dtype)
        dft[i] = _store(y, dtype)
        yq = as_f64(dft[i], dtype)
        for t in range(K):
            tok[i, t] = _gumbel_token(rng, yq[t], T)
        uni[i] = _uniforms(rng, K)
    return ChainBatch(n, K, V, T, dtype, tgt, dft, False, tok, uni, name=name,
                      meta=dict(sigma=sigma, seed=seed, seqs=seqs))


def gaussian_chain_batch(B: int, V: int, K: int, sigma: float, T: float, seed: int,
                         name: str = "") -> ChainBatch:
    """gaussian_chain's recipe (target ~ N(0,1), draft = target + N(0, sigma^2),
    draft tokens sampled from softmax(draft/T) by Gumbel-max), f32, drawn
    from one generator for the whole batch (vectorised; large measurement
    batches, where a subset need not reproduce the full batch's rows)."""
    rng = np.random.default_rng([int(seed), 7])
    z = rng.standard_normal((B, K + 1, V))
    y = z[:, :K] + sigma * rng.standard_normal((B, K, V))
    tgt = z.astype(np.float32)
    dft = y.astype(np.float32)
    g = -np.log(-np.log(np.maximum(rng.random((B, K, V)), 1e-300)))
    tok = np.argmax(dft.astype(np.float64) / T + g, axis=-1).astype(np.int32)
    uni = rng.random((B, K + 1, 2), dtype=np.float32)
    return ChainBatch(B, K, V, T, F32, tgt, dft, False, tok, uni, name=name,
                      meta=dict(sigma=sigma, seed=seed))


def controlled_chain_batch(B: int, K: int, V: int, copy_prob: float, T: float, seed: int,
                           name: str = "") -> ChainBatch:
    """config_controlled's recipe (target rows ~ N(0,1); each draft row a copy of
    its target row with probability copy_prob, else an independent N(0,1) row;
    tokens sampled from the draft), f32, drawn from one generator for the whole
    batch (vectorised)."""
    rng = np.random.default_rng([int(seed), 11])
    tgt = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    indep = rng.standard_normal((B, K, V)).astype(np.float32)
    copied = rng.random((B, K)) < copy_prob
    dft = np.where(copied[..., None], tgt[:, :K], indep)
    g = -np.log(-np.log(np.maximum(rng.random((B, K, V)), 1e-300)))
    tok = np.argmax(dft.astype(np.float64) / T + g, axis=-1).astype(np.int32)
    uni = rng.random((B, K + 1, 2), dtype=np.float32)
    return ChainBatch(B, K, V, T, F32, tgt, np.ascontiguousarray(dft), False, tok, uni, name=name,
                      meta=dict(copied=copied, copy_prob=copy_prob, seed=seed))


def config_tiny(trials: int = 200_000, seed: int = 52_100, V: int = 8, K: int = 4,
                T: float = 1.0, sigma: float = 0.5) -> ChainBatch:
    """Tiny exactness workload: one (target, draft) pair of fp32 logit sets
    (target ~ N(0,1), draft = target + N(0, 0.5^2)), replicated over
    ``trials`` independent trials; each trial draws its own draft tokens from
    softmax(draft/T) and its own uniforms."""
    rng = _rng(seed, 0)
    z = rng.standard_normal((K + 1, V))
    y = z[:K] + sigma * rng.standard_normal((K, V))
    zf = z.astype(np.float32)
    yf = y.astype(np.float32)
    tgt = np.broadcast_to(zf, (trials, K + 1, V)).copy()
    dft = np.broadcast_to(yf, (trials, K, V)).copy()
    # Gumbel-max over all trials at once (row-wise independent noise).
    g = -np.log(-np.log(np.maximum(rng.random((trials, K, V)), 1e-300)))
    if T == 0.0:
        tok = np.broadcast_to(np.argmax(yf.astype(np.float64), axis=-1), (trials, K)).astype(np.int32)
    else:
        tok = np.argmax(yf.astype(np.float64)[None] / T + g, axis=-1).astype(np.int32)
    uni = rng.random((trials, K + 1, 2), dtype=np.float32)
    return ChainBatch(trials, K, V, T, F32, tgt, dft, False, tok, uni, name="tiny",
                      meta=dict(seed=seed, sigma=sigma))


def config_zipf(T: float = 1.0, B: int = 64, V: int = 32000, K: int = 4,
                seed: int = 52_200, seqs=None) -> ChainBatch:
    """B=64, V=32000, K=4 fp32: target ~ N(0, 2^2) - 1.1*log(rank) over a random
    vocabulary permutation; draft = target + N(0, 0.7^2)."""
    return gaussian_chain(B, V, K, sigma=0.7, T=T, dtype=F32, seed=seed, seqs=seqs,
                          scale=2.0, zipf_bias=1.1, name=f"zipf_T{T:g}")


def config_headline(B: int = 256, V: int = 128256, K: int = 5, T: float = 0.7,
                    seed: int = 52_300, seqs=None) -> ChainBatch:
    """B=256, V=128256, K=5 bf16, T=0.7: target ~ N(0,1), draft = target +
    N(0, sigma^2) with sigma set for a mean acceptance of 0.75."""
    return gaussian_chain(B, V, K, sigma=SIGMA_B256_V128K, T=T, dtype=BF16, seed=seed,
                          seqs=seqs, name="headline")


def config_controlled(B: int, K: int, V: int = 151936, copy_prob: float = 0.8,
                      T: float = 1.0, seed: int = 52_400, seqs=None,
                      dtype: str = BF16) -> ChainBatch:
    """Controlled-acceptance sweep: target rows ~ N(0,1); at each position the
    draft row is a bit-identical copy of the target row with probability
    ``copy_prob``, else an independent N(0,1) row."""
    seqs = list(range(B)) if seqs is None else list(seqs)
    n = len(seqs)
    tgt = np.empty((n, K + 1, V), dtype=np.uint16 if dtype == BF16 else np.float32)
    dft = np.empty((n, K, V), dtype=tgt.dtype)
    tok = np.empty((n, K), dtype=np.int32)
    uni = np.empty((n, K + 1, 2), dtype=np.float32)
    copied = np.empty((n, K), dtype=bool)
    for i, b in enumerate(seqs):
        rng = _rng(seed + 1000 * K, b)
        tgt[i] = _store(rng.standard_normal((K + 1, V)), dtype)
        for t in range(K):
            c = bool(rng.random() < copy_prob)
            copied[i, t] = c
            dft[i, t] = tgt[i, t] if c else _store(rng.standard_normal(V), dtype)
            tok[i, t] = _gumbel_token(rng, as_f64(dft[i, t], dtype), T)
        uni[i] = _uniforms(rng, K)
    return ChainBatch(n, K, V, T, dtype, tgt, dft, False, tok, uni,
                      name=f"controlled_B{B}_K{K}",
                      meta=dict(copied=copied, copy_prob=copy_prob, seed=seed, seqs=seqs))


def config_greedy(B: int = 256, V: int = 128256, K: int = 5, match_prob: float = 0.8,
                  seed: int = 52_600, seqs=None, dtype: str = BF16) -> ChainBatch:
    """Greedy chain verification with controlled agreement: target rows ~ N(0,1);
    the draft token at position t is the argmax of target row t with
    probability ``match_prob``, else uniform in [0, V) (``meta["copied"]``
    records which).  No draft rows or uniforms: the greedy rule reads neither."""
    seqs = list(range(B)) if seqs is None else list(seqs)
    n = len(seqs)
    tgt = np.empty((n, K + 1, V), dtype=np.uint16 if dtype == BF16 else np.float32)
    tok = np.empty((n, K), dtype=np.int32)
    copied = np.zeros((n, K), dtype=bool)
    for i, b in enumerate(seqs):
        rng = _rng(seed, b)
        tgt[i] = _store(rng.standard_normal((K + 1, V)), dtype)
        for t in range(K):
            if rng.random() < match_prob:
                tok[i, t] = int(np.argmax(as_f64(tgt[i, t], dtype)))
                copied[i, t] = True
            else:
                tok[i, t] = int(rng.integers(0, V))
    return ChainBatch(n, K, V, 0.0, dtype, tgt, np.zeros((n, K, 0), dtype=tgt.dtype), False, tok,
                      np.zeros((n, K + 1, 2), dtype=np.float32), name=f"greedy_B{B}_K{K}",
                      meta=dict(copied=copied, match_prob=match_prob, seed=seed, seqs=seqs))


def config_tree_masks(B: int = 4096, N: int = 256, seed: int = 52_700, seqs=None) -> np.ndarray:
    """Per-sequence candidate trees (a dynamic tree per sequence, as a drafter
    that widens where it is unsure would build): node i's parent is uniform
    over the nodes before it.  Returns parents [B, N] int32, parents[:, 0] = -1."""
    seqs = list(range(B)) if seqs is None else list(seqs)
    par = np.empty((len(seqs), N), dtype=np.int32)
    for i, b in enumerate(seqs):
        rng = _rng(seed, b)
        par[i, 0] = -1
        if N > 1:
            par[i, 1:] = np.floor(rng.random(N - 1) * np.arange(1, N)).astype(np.int32)
    return par


@dataclass
class KvBatch:
    """Inputs of one KV commit: cache [B, Lmax, E] bytes, lengths [B],
    scratch [B, N, E] bytes, count [B] (entries to append, slots 0..count-1)."""

    B: int
    Lmax: int
    N: int
    E: int
    cache: np.ndarray
    lengths: np.ndarray
    scratch: np.ndarray
    count: np.ndarray


def config_kv_commit(B: int = 256, K: int = 5, E: int = 65536, Lmax: int = 64, alpha: float = 0.75,
                     seed: int = 52_800, seqs=None) -> KvBatch:
    """Chain drafts of length K with i.i.d. acceptance alpha: the number of
    accepted drafts is the run of successes before the first failure (capped
    at K).  Entries are E random bytes (e.g. 32 layers x 8 KV heads x 128 dims
    x bf16 = 64 KB per token); the scratch buffer holds K + 1 slots."""
    seqs = list(range(B)) if seqs is None else list(seqs)
    n = len(seqs)
    N = K + 1
    cache = np.empty((n, Lmax, E), dtype=np.uint8)
    scratch = np.empty((n, N, E), dtype=np.uint8)
    lengths = np.empty(n, dtype=np.int32)
    count = np.empty(n, dtype=np.int32)
    for i, b in enumerate(seqs):
        rng = _rng(seed, b)
        cache[i] = rng.integers(0, 256, size=(Lmax, E), dtype=np.uint8)
        scratch[i] = rng.integers(0, 256, size=(N, E), dtype=np.uint8)
        lengths[i] = int(rng.integers(0, Lmax - K))
        runs = rng.random(K) < alpha
        count[i] = K if runs.all() else int(np.argmin(runs))
    return KvBatch(n, Lmax, N, E, cache, lengths, scratch, count)


def config_tree_draft(B: int = 128, V: int = 128256, branching=(4, 3, 2, 1), N: int = 64,
                      seed: int = 52_900, seqs=None, dtype: str = BF16):
    """Top-k tree drafting: draft logit rows ~ N(0,1), one per node of the static
    BFS tree ``branching`` truncated to N nodes (row p: the draft's distribution
    for the children of node p).  Returns (parents [N], draft [B, N, V])."""
    seqs = list(range(B)) if seqs is None else list(seqs)
    par = bfs_tree(branching, N)
    draft = np.empty((len(seqs), len(par), V), dtype=np.uint16 if dtype == BF16 else np.float32)
    for i, b in enumerate(seqs):
        draft[i] = _store(_rng(seed, b).standard_normal((len(par), V)), dtype)
    return par, draft


def bfs_tree(branching, max_nodes=None) -> np.ndarray:
    """Parent array of a static tree in breadth-first order: the root, then
    ``branching[0]`` children of the root, then ``branching[1]`` children of
    each depth-1 node, and so on; optionally truncated to ``max_nodes`` nodes."""
    parents = [-1]
    level = [0]
    for br in branching:
        nxt = []
        for p in level:
            for _ in range(br):
                parents.append(p)
                nxt.append(len(parents) - 1)
        level = nxt
    if max_nodes is not None:
        parents = parents[:max_nodes]
    return np.asarray(parents, dtype=np.int32)


def tree_depths(parents: np.ndarray) -> np.ndarray:
    d = np.zeros(len(parents), dtype=np.int32)
    for i in range(1, len(parents)):
        d[i] = d[parents[i]] + 1
    return d


def config_tree(B: int = 128, V: int = 128256, branching=(4, 3, 2, 1), N: int = 64,
                match_prob: float = 0.7, seed: int = 52_500, seqs=None,
                dtype: str = BF16) -> TreeBatch:
    """Greedy tree verification: target logits ~ N(0,1) at every node of a
    static BFS tree with the given branching, truncated to N nodes; a node's
    token is its parent's argmax with probability ``match_prob``, else uniform
    in [0, V)."""
    parents = bfs_tree(branching, N)
    N = len(parents)
    depth = int(tree_depths(parents).max())
    seqs = list(range(B)) if seqs is None else list(seqs)
    n = len(seqs)
    tgt = np.empty((n, N, V), dtype=np.uint16 if dtype == BF16 else np.float32)
    tok = np.empty((n, N), dtype=np.int32)
    copied = np.zeros((n, N), dtype=bool)
    for i, b in enumerate(seqs):
        rng = _rng(seed, b)
        tgt[i] = _store(rng.standard_normal((N, V)), dtype)
        rows = as_f64(tgt[i], dtype)
        tok[i, 0] = -1
        for j in range(1, N):
            if rng.random() < match_prob:
                tok[i, j] = int(np.argmax(rows[parents[j]]))
                copied[i, j] = True
            else:
                tok[i, j] = int(rng.integers(0, V))
    return TreeBatch(n, N, V, dtype, tgt, parents, tok, depth, name=f"tree_B{B}_N{N}", copied=copied)


__all__ = [
    "F32", "BF16", "ChainBatch", "TreeBatch", "SIGMA_B256_V128K", "config_greedy",
    "f32_to_bf16_bits", "bf16_bits_to_f64", "as_f64", "gaussian_chain",
    "config_tiny", "config_zipf", "config_headline", "config_controlled", "gaussian_chain_batch",
    "controlled_chain_batch",
    "config_tree", "config_tree_draft", "bfs_tree", "tree_depths", "config_tree_masks", "KvBatch", "config_kv_commit",
]
