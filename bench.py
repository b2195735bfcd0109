#!/usr/bin/env python
"""Benchmark of batched draft-token verification on GB300.

Default workload ("sample"): one step = one spec_verify_sample call over the
B=256, V=128256, K=5, bf16, T=0.7 batch (target logits [256,6,128256], draft
logits [256,5,128256]): the vocabulary sweep over all 2816 rows plus the
per-sequence accept scan and replacement/bonus draw, all inside one persistent
kernel launch (after a small memset of the workspace's control block).

Other workloads (--workload):
  zipf    spec_verify_sample, B=64, V=32000, K=4, f32, T=1: target 2*N(0,1) with
          a Zipf-like bias -1.1*log(rank) over a random vocabulary permutation,
          draft = target + N(0, 0.7^2)
  zipf_greedy  spec_verify_greedy on the same inputs (the temperature-0 run)
  ctl_B<B>_K<K>  spec_verify_sample over the controlled-acceptance sweep,
          V=151936 bf16 T=1, B in {1, 8, 64, 512}, K in {4, 8}: each draft row is
          a copy of its target row with probability 0.8, else an independent row
  sweep   all eight ctl_B<B>_K<K> workloads in one run, one JSON line each
  acceptance  spec_row_stats + spec_verify_sample on 5 x 10,000 one-draft
          sequences (V=2048 f32) at graded draft noise: the acceptance rate
          against sum min(p,q) and KL(q||p), and tokens per target pass against
          K for alpha ~ 0.5 / 0.7 / 0.9 (controlled copies), in the JSON line
  greedy  spec_verify_greedy, B=256, V=128256, K=5, bf16; draft token t is the
          target row's argmax with probability 0.8
  tree    spec_verify_tree_greedy, B=128, N=64 nodes (BFS [4,3,2,1] truncated),
          V=128256, bf16; node tokens copy the parent's argmax with probability 0.7
  treemask  spec_tree_mask, 4096 per-sequence trees of 256 nodes
  kvcommit  spec_kv_commit, 256 chains, 64 KB entries
  stats     spec_row_stats over the default workload's rows: sum min(p,q), KL, TV
  draft     spec_tree_draft, B=128 trees of 64 nodes, V=128256: top-k children per node
Both read only the rows the greedy rules need (rows up to the first mismatch;
accepted tree nodes), one persistent kernel per call; their algorithmic bytes
are those rows, counted from the generator's own copy draws.

Inputs are generated once (seeded, synthetic), copied to HBM, and the timed
region covers exactly --steps calls bracketed by a barrier and a device
synchronisation, timed with CUDA events; a second pass of --steps calls with
the library's per-kernel event hooks gives the kernel durations the roofline
uses.  Inputs smaller than twice the L2 cache (129 MB) are held in several
device copies that the steps cycle through, so every step reads inputs that
at least one L2's worth of other traffic has passed since their last use; no
flush is needed between steps.

Reported: the metric (verified draft positions/s; tree: candidate nodes/s),
the dominant kernel's achieved HBM bandwidth against the measured copy peak
(roofline: algorithmic bytes per launch over the launch duration taken from
the timed region, the per-call event time beside it), an end-to-end figure with host<->device copies inside the timed
region, the SM clocks seen during the run, and the double-precision CPU
oracle timed on a bounded sample on this host.

The CPU baseline is the double-precision oracle on this host's cores (one
thread per core, sequences split between threads; the single-threaded rate
is reported beside it).  It runs on the first sequences of the timed batch,
and the GPU outputs of those sequences are compared with the oracle's there
(the parity block: bit-exact outside decisions the oracle flags as within
1e-6 of flipping, flags counted).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload sample|zipf|zipf_greedy|ctl_B<B>_K<K>|sweep|greedy|tree|treemask|kvcommit|stats|draft]
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

B, V, K, T = 256, 128256, 5, 0.7
TREE_B, TREE_N = 128, 64
METRIC = "verified draft positions/s"
UNIT = "positions/s"


def sweep_bytes(b=B, k=K, v=V, elem=2):
    """Bytes of one pass over every target and draft row."""
    return b * (2 * k + 1) * v * elem


L2_BYTES = 129 * 10**6


def rotation_copies(nbytes: int) -> int:
    """Device copies of a step's inputs to cycle through so that copies x
    bytes spans at least twice the L2 cache."""
    return max(1, -(-2 * L2_BYTES // max(1, nbytes)))


def metric_bytes(b=B, k=K, v=V, elem=2):
    """Algorithmic bytes of one sampling call: one pass over all rows + one
    stopping target row per sequence."""
    return (b * (k + 1) * v + b * k * v + b * v) * elem


def source_sha(files=None) -> str:
    """Hash of the kernel sources a profile was taken on: the given csrc files
    (the kernel's own header plus the shared helpers), or all of csrc."""
    d = os.path.join(ROOT, "speculative_decoding_verification_52_gb300", "csrc")
    names = sorted(files) if files else sorted(os.listdir(d))
    h = hashlib.sha256()
    for f in names:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary: str, files=None):
    """dram read+write bytes per launch of the dominant kernel from a committed
    ncu summary, only if it was taken on the current kernel sources."""
    try:
        kv = {}
        with open(os.path.join(ROOT, "profiles", summary)) as f:
            for line in f:
                if ":" in line:
                    k_, v_ = line.split(":", 1)
                    kv[k_.strip()] = v_.strip()
        if kv.get("source_sha") != source_sha(files):
            return None
        return int(float(kv["dram_bytes_per_launch"]))
    except (OSError, KeyError, ValueError):
        return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling in the background."""

    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for r in csv.reader(io.StringIO(f.read())):
                if len(r) >= 10:
                    rows.append([c.strip() for c in r])
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "power_w_max": max((float(r[4]) for r in rows if r[4].replace(".", "").isdigit()), default=None)}


# ---------------------------------------------------------------------------
# multi-rank host logic (replicas over sequences, weak scaling)
# ---------------------------------------------------------------------------
def rank_sequences(rank: int, per_rank: int) -> list[int]:
    """Sequence ids of one rank: every rank verifies its own batch, disjoint
    from the others' (sequences are independent; nothing is exchanged)."""
    return list(range(rank * per_rank, (rank + 1) * per_rank))


def max_over_ranks(values, ws: int, device=None):
    """Element-wise max of per-rank timings (the slowest rank sets the job's time)."""
    values = [float(v) for v in values]
    if ws <= 1:
        return values
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
class Workload:
    """One benchmarked call: its batch, the metric's units per step, the
    dominant kernel and its algorithmic bytes, and the oracle's CPU leg."""
    name = ""
    metric = METRIC
    unit = UNIT
    summary = ""
    kernel = ""
    sources = ()             # csrc files the dominant kernel is built from
    per_rank = B
    launches_per_step = 1
    dtype = "f32"            # what the path computes in
    oracle_dtype = "f64"
    seq_noun = "sequence verifications"   # what one oracle sequence of the batch is

    def describe(self) -> dict:
        raise NotImplementedError

    def batch(self, seqs):
        raise NotImplementedError

    def units(self, batch) -> int:
        raise NotImplementedError

    def algorithmic_bytes(self, batch) -> int:
        raise NotImplementedError

    def oracle_call(self, batch, sl):
        raise NotImplementedError

    def oracle_chunk(self) -> int:
        return 4

    def parity(self, batch, outs, n):
        """GPU outputs of the first n sequences against the oracle (None when
        the workload has no parity summary here)."""
        return None

    def extra_report(self, batch) -> dict:
        """Workload-specific measurements added to the JSON line."""
        return {}

    def device_setup(self, batch, dev):
        """Returns (host inputs, device inputs they are copied to, step(),
        device outputs)."""
        raise NotImplementedError


def _bf16_host(x):
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).pin_memory()


def _pinned(x):
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).pin_memory()


def sample_parity(batch, out, nacc, n):
    """Sampling outputs of the first n sequences against the oracle: bit-exact
    except after decisions the oracle flags as within 1e-6 of flipping (a near
    accept test at t excludes slots >= t and the count; a near CDF boundary
    excludes only the drawn token).  Counts flags and mismatches."""
    import numpy as np

    import oracle
    sl = slice(0, n)
    ref = oracle.verify_sample(batch.target[sl], batch.dtype, batch.draft[sl], batch.draft_dtype,
                               batch.draft_is_probs, np.ascontiguousarray(batch.draft_tokens[sl]),
                               np.ascontiguousarray(batch.uniforms[sl]), batch.T)
    na, nc, ro, rn = ref["near_accept"], ref["near_cdf"], ref["out_tokens"], ref["num_accepted"]
    flagged = flagged_mismatch = unflagged_mismatch = 0
    for b in range(n):
        if na[b] >= 0:
            flagged += 1
            t = int(na[b])
            ok = bool((out[b, :t] == ro[b, :t]).all())
            if not ok:
                unflagged_mismatch += 1
            elif nacc[b] != rn[b] or not (out[b] == ro[b]).all():
                flagged_mismatch += 1
            continue
        if nacc[b] != rn[b]:
            unflagged_mismatch += 1
            continue
        if nc[b]:
            flagged += 1
            tsl = int(rn[b]) if rn[b] >= 0 else 0
            keep = np.ones(out.shape[1], dtype=bool)
            keep[tsl] = False
            if not (out[b][keep] == ro[b][keep]).all():
                unflagged_mismatch += 1
            elif out[b, tsl] != ro[b, tsl]:
                flagged_mismatch += 1
            continue
        if not (out[b] == ro[b]).all():
            unflagged_mismatch += 1
    return {"sequences": n, "near_accept": int((na >= 0).sum()), "near_cdf": int((nc != 0).sum()),
            "flagged_sequences": flagged, "flagged_mismatch": flagged_mismatch,
            "unflagged_mismatch": unflagged_mismatch,
            "rule": "bit-exact except after a decision within 1e-6 of flipping (counted)"}


def greedy_parity(batch, out, nacc, n):
    """Greedy outputs of the first n sequences against the oracle, bit for bit."""
    import numpy as np

    import oracle
    ro, rn = oracle.verify_greedy(batch.target[:n], batch.dtype, np.ascontiguousarray(batch.draft_tokens[:n]))
    bad = int(((nacc[:n] != rn) | (out[:n] != ro).any(axis=1)).sum())
    return {"sequences": n, "mismatch": bad, "rule": "bit-exact"}


class ChainWorkload(Workload):
    """One chain-verification call (sampling, or the greedy rule) over a
    ChainBatch, with the batch's inputs held in rotation_copies(...) device
    copies that consecutive steps cycle through."""

    def __init__(self, name, label, make, B_, K_, V_, T_, elem, greedy=False, summary="", kernel=""):
        self.name, self.label, self.make = name, label, make
        self.Bn, self.Kn, self.Vn, self.Tn, self.elem, self.greedy = B_, K_, V_, T_, elem, greedy
        self.per_rank = B_
        self.summary = summary
        self.kernel = kernel or ("tree_greedy_kernel (chain mode)" if greedy else "fused_sample_kernel")
        self.sources = ("common.cuh", "tree.cuh") if greedy else ("common.cuh", "fused.cuh")

    def input_bytes(self):
        if self.greedy:
            return self.Bn * (self.Kn + 1) * self.Vn * self.elem
        return self.Bn * (2 * self.Kn + 1) * self.Vn * self.elem

    def describe(self):
        nb = self.input_bytes()
        c = rotation_copies(nb)
        return {"workload": self.label, "B": self.Bn, "V": self.Vn, "K": self.Kn,
                "temperature": 0.0 if self.greedy else self.Tn, "input_bytes": nb, "input_copies": c,
                "l2": (f"inputs ({nb / 1e6:.1f} MB) larger than twice L2; no flush" if c == 1 else
                       f"{c} device copies of the inputs ({c * nb / 1e6:.1f} MB) cycled: each step reads "
                       f"inputs untouched for at least one L2's worth of traffic; no flush")}

    def batch(self, seqs):
        return self.make(seqs)

    def units(self, batch):
        return batch.B * batch.K

    def algorithmic_bytes(self, batch):
        if not self.greedy:
            return metric_bytes(batch.B, batch.K, batch.V, self.elem)
        # the greedy rule reads rows 0..n of a sequence that accepts n drafts
        # (the argmax of the f32 target rows, first index on ties)
        import numpy as np
        g = np.argmax(batch.target, axis=-1)[:, :batch.K]
        rows = int((leading_true(g == batch.draft_tokens) + 1).sum())
        return rows * batch.V * self.elem

    def oracle_call(self, batch, sl):
        import numpy as np

        import oracle
        tok = np.ascontiguousarray(batch.draft_tokens[sl])
        if self.greedy:
            oracle.verify_greedy(batch.target[sl], batch.dtype, tok)
        else:
            oracle.verify_sample(batch.target[sl], batch.dtype, batch.draft[sl], batch.draft_dtype,
                                 batch.draft_is_probs, tok, np.ascontiguousarray(batch.uniforms[sl]), batch.T)

    def oracle_chunk(self):
        return 1

    def parity(self, batch, outs, n):
        out, nacc = outs[0], outs[1]
        return greedy_parity(batch, out, nacc, n) if self.greedy else sample_parity(batch, out, nacc, n)

    def device_setup(self, batch, dev):
        import torch

        import speculative_decoding_verification_52_gb300 as sv
        conv = _bf16_host if batch.dtype == "bf16" else _pinned
        hs = [conv(batch.target)]
        if not self.greedy:
            hs.append(conv(batch.draft))
        hs += [_pinned(batch.draft_tokens), _pinned(batch.uniforms)]
        copies = rotation_copies(self.input_bytes())
        sets = [[h.to(dev) for h in hs] for _ in range(copies)]
        out = torch.empty((batch.B, batch.K + 1), dtype=torch.int32, device=dev)
        nacc = torch.empty((batch.B,), dtype=torch.int32, device=dev)
        wsb = sv.workspace(sv.spec_workspace_bytes(batch.B, batch.K, batch.V), dev)
        stream = torch.cuda.current_stream()
        i = [0]

        def step():
            d = sets[i[0]]
            i[0] = (i[0] + 1) % copies
            if self.greedy:
                sv.spec_verify_greedy(d[0], d[1], out_tokens=out, num_accepted=nacc, workspace_buf=wsb,
                                      stream=stream)
            else:
                sv.spec_verify_sample(d[0], d[1], d[2], d[3], batch.T, out_tokens=out, num_accepted=nacc,
                                      workspace_buf=wsb, stream=stream)
        # end to end: the host inputs are copied into the set the next step reads
        return hs, _RotatingSets(sets, i), step, [out, nacc]


class _RotatingSets:
    """The device input set the next step reads (for the end-to-end copies)."""

    def __init__(self, sets, index):
        self.sets, self.index = sets, index

    def __iter__(self):
        return iter(self.sets[self.index[0]])


def _zipf(T_):
    def make(seqs):
        from speculative_decoding_verification_52_gb300 import inputs as gen
        return gen.config_zipf(T=T_, B=64, seqs=seqs)
    return make


def _controlled(B_, K_):
    def make(seqs):
        from speculative_decoding_verification_52_gb300 import inputs as gen
        return gen.config_controlled(B_, K_, seqs=seqs)
    return make


SWEEP = [(b, k) for k in (4, 8) for b in (1, 8, 64, 512)]
CHAIN_WORKLOADS = [
    ChainWorkload("zipf", "spec-verify sampling B=64 V=32000 K=4 f32 T=1, Zipf-biased targets "
                  "(2*N(0,1) - 1.1*log(rank)), draft = target + N(0,0.7^2)", _zipf(1.0), 64, 4, 32000, 1.0, 4),
    ChainWorkload("zipf_greedy", "spec-verify greedy B=64 V=32000 K=4 f32, the Zipf-biased inputs "
                  "(rows up to the first mismatch)", _zipf(1.0), 64, 4, 32000, 1.0, 4, greedy=True),
] + [
    ChainWorkload(f"ctl_B{b}_K{k}", f"spec-verify sampling B={b} V=151936 K={k} bf16 T=1, controlled "
                  f"acceptance (draft row = target row w.p. 0.8, else an independent N(0,1) row)",
                  _controlled(b, k), b, k, 151936, 1.0, 2)
    for b, k in SWEEP
]


class AcceptanceWorkload(Workload):
    """The pages' acceptance measurement ("Speculative decoding: draft, verify,
    repeat", step 4: acceptance rate against the divergence of the draft from
    the verifier; "Speculative decoding and EAGLE", exercises: tokens per target
    pass against K).  One step scores and verifies five batches of 10,000
    one-draft sequences (V=2048 f32, T=1) whose drafts are the target plus
    N(0, sigma^2) noise at graded sigma: spec_row_stats gives sum min(p,q) and
    KL(q||p) per position, spec_verify_sample the accept decision."""
    name = "acceptance"
    metric = "draft positions scored and verified/s"
    unit = "positions/s"
    kernel = "row_stats_kernel (a cluster of one per pair) + fused_sample_kernel (f32, V=2048)"
    sources = ("common.cuh", "row_stats.cuh", "fused.cuh")
    SIGMAS = (0.1, 0.3, 0.6, 1.0, 2.0)
    NSEQ, VV = 10_000, 2048
    COPY = (0.04, 0.42, 0.81)      # draft row = target row w.p. c (alpha ~ 0.5, 0.7, 0.9 at T=1)
    KS = (1, 2, 3, 4, 5, 6, 7, 8)
    per_rank = 10_000
    launches_per_step = 2 * len(SIGMAS)

    def describe(self):
        return {"workload": "acceptance against KL(q||p): 5 batches of 10,000 one-draft sequences, V=2048 f32 "
                            "T=1, draft = target + N(0, sigma^2), sigma in (0.1, 0.3, 0.6, 1.0, 2.0); per step "
                            "spec_row_stats and spec_verify_sample on each batch",
                "B": self.NSEQ, "V": self.VV, "K": 1, "temperature": 1.0,
                "input_bytes": len(self.SIGMAS) * self.NSEQ * 3 * self.VV * 4,
                "l2": "inputs (1.23 GB) larger than L2; no flush"}

    class Batches(list):
        """The five sigma batches; B = sequences per batch."""
        B = 0

    def batch(self, seqs):
        from speculative_decoding_verification_52_gb300 import inputs as gen
        out = self.Batches(gen.gaussian_chain_batch(len(seqs), self.VV, 1, sigma=s_, T=1.0, seed=52_600 + i)
                           for i, s_ in enumerate(self.SIGMAS))
        out.B = len(seqs)
        return out

    def units(self, batch):
        return sum(b.B * b.K for b in batch)

    def algorithmic_bytes(self, batch):
        # statistics: target row 0 and draft row 0 of every sequence; verify:
        # every row once plus one stopping target row
        return sum(2 * b.B * b.K * b.V * 4 + metric_bytes(b.B, b.K, b.V, 4) for b in batch)

    def oracle_chunk(self):
        return 64

    def oracle_call(self, batch, sl):
        import numpy as np

        import oracle
        for b in batch:
            oracle.row_stats(b.target[sl], "f32", b.draft[sl], "f32", False, 1.0)
            oracle.verify_sample(b.target[sl], "f32", b.draft[sl], "f32", False,
                                 np.ascontiguousarray(b.draft_tokens[sl]), np.ascontiguousarray(b.uniforms[sl]), 1.0)

    def device_setup(self, batch, dev):
        import torch

        import speculative_decoding_verification_52_gb300 as sv
        hs, ds, res = [], [], []
        for b in batch:
            h = [_pinned(b.target), _pinned(b.draft), _pinned(b.draft_tokens), _pinned(b.uniforms)]
            hs += h
            d = [x.to(dev) for x in h]
            ds += d
            r = dict(d=d, T=b.T, alpha=torch.empty((b.B, 1), dtype=torch.float32, device=dev),
                     kl=torch.empty((b.B, 1), dtype=torch.float32, device=dev),
                     tv=torch.empty((b.B, 1), dtype=torch.float32, device=dev),
                     out=torch.empty((b.B, 2), dtype=torch.int32, device=dev),
                     nacc=torch.empty((b.B,), dtype=torch.int32, device=dev),
                     ws=sv.workspace(sv.spec_workspace_bytes(b.B, 1, b.V), dev))
            res.append(r)
        stream = torch.cuda.current_stream()
        self._res = res

        def step():
            for r in res:
                d = r["d"]
                sv.spec_row_stats(d[0], d[1], r["T"], alpha=r["alpha"], kl=r["kl"], tv=r["tv"], stream=stream)
                sv.spec_verify_sample(d[0], d[1], d[2], d[3], r["T"], out_tokens=r["out"], num_accepted=r["nacc"],
                                      workspace_buf=r["ws"], stream=stream)
        outs = [x for r in res for x in (r["alpha"], r["kl"], r["nacc"])]
        return hs, ds, step, outs

    def extra_report(self, batch):
        """The acceptance curve from the last step's outputs, and tokens per
        target pass against K on controlled-copy batches (2,000 sequences,
        V=1024 f32, run once here)."""
        import numpy as np
        import torch

        import speculative_decoding_verification_52_gb300 as sv
        from speculative_decoding_verification_52_gb300 import inputs as gen
        torch.cuda.synchronize()
        curve = []
        for s_, r in zip(self.SIGMAS, self._res):
            a = r["alpha"].cpu().numpy()[:, 0]
            kl = r["kl"].cpu().numpy()[:, 0]
            acc = (r["nacc"].cpu().numpy() >= 1).astype(np.float64)
            m = float(a.mean())
            curve.append({"sigma": s_, "mean_alpha": m, "mean_kl": float(kl.mean()),
                          "accept_rate": float(acc.mean()), "se": float(np.sqrt(m * (1 - m) / len(acc)))})
        dev = torch.device("cuda", torch.cuda.current_device())
        tpp = []
        for c in self.COPY:
            for k in self.KS:
                b = gen.controlled_chain_batch(2000, k, 1024, c, 1.0, seed=52_650 + k)
                t = torch.from_numpy(b.target).to(dev)
                d = torch.from_numpy(b.draft).to(dev)
                alpha, _, _ = sv.spec_row_stats(t, d, b.T)
                _, n = sv.spec_verify_sample(t, d, torch.from_numpy(b.draft_tokens).to(dev),
                                             torch.from_numpy(b.uniforms).to(dev), b.T)
                al = float(alpha.mean().item())
                tok = n.cpu().numpy().astype(np.float64) + 1.0
                tpp.append({"copy_prob": c, "K": k, "alpha": al, "tokens_per_pass": float(tok.mean()),
                            "closed_form": (1 - al ** (k + 1)) / (1 - al), "se": float(tok.std() / np.sqrt(len(tok)))})
        return {"acceptance_curve": curve, "tokens_per_pass": tpp}


class SampleWorkload(Workload):
    name = "sample"
    summary = "fused_sample_kernel_b256_v128256_k5_bf16.md"
    kernel = "fused_sample_kernel<bf16 target, bf16 draft logits>"
    sources = ("common.cuh", "fused.cuh")

    def describe(self):
        return {"workload": "spec-verify sampling B=256 V=128256 K=5 bf16 T=0.7 (target+draft logits, accept scan, "
                            "residual/bonus draw)", "B": B, "V": V, "K": K, "temperature": T,
                "input_bytes": sweep_bytes(), "metric_bytes_per_step": metric_bytes(),
                "l2": "inputs (722 MB) larger than L2; no flush"}

    def batch(self, seqs):
        from speculative_decoding_verification_52_gb300 import inputs as gen
        return gen.config_headline(seqs=seqs)

    def units(self, batch):
        return batch.B * batch.K

    def algorithmic_bytes(self, batch):
        return metric_bytes(batch.B, batch.K, batch.V)

    def parity(self, batch, outs, n):
        return sample_parity(batch, outs[0], outs[1], n)

    def oracle_call(self, batch, sl):
        import numpy as np

        import oracle
        oracle.verify_sample(batch.target[sl], batch.dtype, batch.draft[sl], batch.dtype, False,
                             np.ascontiguousarray(batch.draft_tokens[sl]), np.ascontiguousarray(batch.uniforms[sl]),
                             batch.T)

    def device_setup(self, batch, dev):
        import torch

        import speculative_decoding_verification_52_gb300 as sv
        hs = [_bf16_host(batch.target), _bf16_host(batch.draft), _pinned(batch.draft_tokens),
              _pinned(batch.uniforms)]
        ds = [h.to(dev) for h in hs]
        out = torch.empty((batch.B, batch.K + 1), dtype=torch.int32, device=dev)
        nacc = torch.empty((batch.B,), dtype=torch.int32, device=dev)
        wsb = sv.workspace(sv.spec_workspace_bytes(batch.B, batch.K, batch.V), dev)
        stream = torch.cuda.current_stream()

        def step():
            sv.spec_verify_sample(ds[0], ds[1], ds[2], ds[3], batch.T, out_tokens=out, num_accepted=nacc,
                                  workspace_buf=wsb, stream=stream)
        return hs, ds, step, [out, nacc]


def leading_true(flags):
    """Per row, the number of leading True entries."""
    import numpy as np
    f = np.asarray(flags, dtype=bool)
    return np.where(f.all(axis=1), f.shape[1], np.argmin(f, axis=1))


class GreedyWorkload(Workload):
    name = "greedy"
    summary = "tree_greedy_kernel_chain_b256_v128256_k5_bf16.md"
    kernel = "tree_greedy_kernel<bf16> (chain mode)"
    sources = ("common.cuh", "tree.cuh")

    def describe(self):
        return {"workload": "spec-verify greedy B=256 V=128256 K=5 bf16, draft = target argmax w.p. 0.8 "
                            "(rows up to the first mismatch)", "B": B, "V": V, "K": K, "temperature": 0.0,
                "input_bytes": B * (K + 1) * V * 2, "l2": "inputs (394 MB) larger than L2; no flush"}

    def batch(self, seqs):
        from speculative_decoding_verification_52_gb300 import inputs as gen
        return gen.config_greedy(seqs=seqs)

    def units(self, batch):
        return batch.B * batch.K

    def algorithmic_bytes(self, batch):
        # rows 0..n per sequence, n = accepted drafts = leading copied positions
        rows = int((leading_true(batch.meta["copied"]) + 1).sum())
        return rows * batch.V * 2

    def oracle_call(self, batch, sl):
        import numpy as np

        import oracle
        oracle.verify_greedy(batch.target[sl], batch.dtype, np.ascontiguousarray(batch.draft_tokens[sl]))

    def parity(self, batch, outs, n):
        return greedy_parity(batch, outs[0], outs[1], n)

    def device_setup(self, batch, dev):
        import torch

        import speculative_decoding_verification_52_gb300 as sv
        hs = [_bf16_host(batch.target), _pinned(batch.draft_tokens)]
        ds = [h.to(dev) for h in hs]
        out = torch.empty((batch.B, batch.K + 1), dtype=torch.int32, device=dev)
        nacc = torch.empty((batch.B,), dtype=torch.int32, device=dev)
        wsb = sv.workspace(sv.spec_workspace_bytes(batch.B, batch.K, batch.V), dev)
        stream = torch.cuda.current_stream()

        def step():
            sv.spec_verify_greedy(ds[0], ds[1], out_tokens=out, num_accepted=nacc, workspace_buf=wsb, stream=stream)
        return hs, ds, step, [out, nacc]


class TreeWorkload(Workload):
    name = "tree"
    metric = "verified candidate tree nodes/s"
    unit = "nodes/s"
    summary = "tree_greedy_kernel_b128_n64_v128256_bf16.md"
    kernel = "tree_greedy_kernel<bf16>"
    sources = ("common.cuh", "tree.cuh")
    per_rank = TREE_B

    def describe(self):
        return {"workload": "spec-verify tree greedy B=128 N=64 (BFS [4,3,2,1] truncated) V=128256 bf16",
                "B": TREE_B, "N": TREE_N, "V": V, "input_bytes": TREE_B * TREE_N * V * 2,
                "l2": "inputs (2.10 GB) larger than L2; no flush"}

    def batch(self, seqs):
        from speculative_decoding_verification_52_gb300 import inputs as gen
        return gen.config_tree(seqs=seqs)

    def units(self, batch):
        return batch.B * (batch.N - 1)

    def algorithmic_bytes(self, batch):
        # accepted nodes' rows: a node is accepted iff every node on its path
        # from the root drew a copy of its parent's argmax
        import numpy as np
        acc = np.zeros((batch.B, batch.N), dtype=bool)
        acc[:, 0] = True
        for j in range(1, batch.N):
            acc[:, j] = acc[:, batch.parents[j]] & batch.copied[:, j]
        return int(acc.sum()) * batch.V * 2

    def oracle_chunk(self):
        return 1

    def oracle_call(self, batch, sl):
        import numpy as np

        import oracle
        oracle.verify_tree_greedy(batch.target[sl], batch.dtype, batch.parents,
                                  np.ascontiguousarray(batch.node_tokens[sl]), batch.max_depth)

    def device_setup(self, batch, dev):
        import numpy as np
        import torch

        import speculative_decoding_verification_52_gb300 as sv
        hs = [_bf16_host(batch.target), _pinned(batch.node_tokens)]
        ds = [h.to(dev) for h in hs]
        parents = torch.from_numpy(np.ascontiguousarray(batch.parents, dtype=np.int32)).to(dev)
        W = batch.max_depth + 1
        out = torch.empty((batch.B, W), dtype=torch.int32, device=dev)
        nacc = torch.empty((batch.B,), dtype=torch.int32, device=dev)
        path = torch.empty((batch.B, W), dtype=torch.int32, device=dev)
        wsb = sv.workspace(sv.spec_tree_workspace_bytes(batch.B, batch.N, batch.V), dev)
        stream = torch.cuda.current_stream()

        def step():
            sv.spec_verify_tree_greedy(ds[0], parents, ds[1], batch.max_depth, out_tokens=out, num_accepted=nacc,
                                       out_path=path, workspace_buf=wsb, stream=stream)
        return hs, ds, step, [out, nacc, path]


class TreeMaskWorkload(Workload):
    name = "treemask"
    metric = "tree-attention mask rows/s"
    unit = "rows/s"
    summary = "tree_mask_kernel_b4096_n256.md"
    kernel = "tree_mask_run_kernel<8>"
    seq_noun = "trees masked"
    sources = ("tree_mask.cuh",)
    dtype = oracle_dtype = "u32"
    per_rank = 4096
    NODES = 256

    def describe(self):
        nw = (self.NODES + 31) // 32
        return {"workload": "tree attention masks, B=4096 per-sequence trees of N=256 nodes (parent uniform over "
                            "earlier nodes)", "B": self.per_rank, "N": self.NODES,
                "input_bytes": 4 * self.per_rank * self.NODES,
                "output_bytes": 4 * self.per_rank * self.NODES * nw,
                "l2": "outputs (33.6 MB) within L2; steps are back to back"}

    def batch(self, seqs):
        from speculative_decoding_verification_52_gb300 import inputs as gen
        par = gen.config_tree_masks(N=self.NODES, seqs=seqs)

        class _B:
            pass
        b = _B()
        b.B, b.N, b.parents = par.shape[0], par.shape[1], par
        return b

    def units(self, batch):
        return batch.B * batch.N

    def algorithmic_bytes(self, batch):
        return 4 * batch.B * batch.N * (1 + (batch.N + 31) // 32) + 4 * batch.B

    def oracle_call(self, batch, sl):
        import oracle
        oracle.tree_mask(batch.parents[sl])

    def device_setup(self, batch, dev):
        import torch

        import speculative_decoding_verification_52_gb300 as sv
        hs = [_pinned(batch.parents)]
        ds = [h.to(dev) for h in hs]
        masks = torch.empty((batch.B, batch.N, (batch.N + 31) // 32), dtype=torch.int32, device=dev)
        status = torch.empty((batch.B,), dtype=torch.int32, device=dev)
        stream = torch.cuda.current_stream()

        def step():
            sv.spec_tree_mask(ds[0], masks=masks, status=status, stream=stream)
        return hs, ds, step, [masks, status]


class KvCommitWorkload(Workload):
    name = "kvcommit"
    metric = "KV entries committed/s"
    unit = "entries/s"
    summary = "kv_commit_kernel_b256_e64k.md"
    kernel = "kv_commit_kernel"
    seq_noun = "chains committed"
    sources = ("kv_commit.cuh",)
    dtype = oracle_dtype = "u8"

    def describe(self):
        return {"workload": "KV commit-on-accept, B=256 chains of K=5 drafts (i.i.d. acceptance 0.75), 64 KB "
                            "entries (32 layers x 8 KV heads x 128 x bf16), cache of 64 slots per sequence",
                "B": B, "K": 5, "entry_bytes": 65536, "Lmax": 64,
                "l2": "scratch (101 MB) and cache (1.07 GB) beyond L2 in total; steps re-commit the same entries",
                "e2e_note": "the cache is resident state: end to end copies the scratch, lengths and counts"}

    def batch(self, seqs):
        from speculative_decoding_verification_52_gb300 import inputs as gen
        return gen.config_kv_commit(seqs=seqs)

    def units(self, batch):
        return int(batch.count[batch.count > 0].sum())

    def algorithmic_bytes(self, batch):
        return 2 * self.units(batch) * batch.E + 12 * batch.B

    def oracle_call(self, batch, sl):
        import oracle
        oracle.kv_commit(batch.cache[sl], batch.lengths[sl], batch.scratch[sl], None, batch.count[sl])

    def device_setup(self, batch, dev):
        import torch

        import speculative_decoding_verification_52_gb300 as sv
        hs = [_pinned(batch.scratch), _pinned(batch.lengths), _pinned(batch.count)]
        ds = [h.to(dev) for h in hs]
        cache = torch.from_numpy(batch.cache).to(dev)
        newl = torch.empty((batch.B,), dtype=torch.int32, device=dev)
        stream = torch.cuda.current_stream()

        def step():
            sv.spec_kv_commit(cache, ds[1], ds[0], ds[2], new_lengths=newl, stream=stream)
        return hs, ds, step, [newl]


class StatsWorkload(Workload):
    name = "stats"
    metric = "draft positions scored/s"
    unit = "positions/s"
    summary = "row_stats_stream_kernel_b256_v128256_k5_bf16.md"
    kernel = "row_stats_stream_kernel<bf16>"
    seq_noun = "sequences' statistics"
    sources = ("common.cuh", "row_stats.cuh", "row_stats_stream.cuh")

    def describe(self):
        return {"workload": "acceptance statistics (sum min(p,q), KL(q||p), TV) per drafted position, B=256 "
                            "V=128256 K=5 bf16 T=0.7, the headline sampling inputs", "B": B, "V": V, "K": K,
                "temperature": T, "input_bytes": 2 * B * K * V * 2,
                "l2": "inputs (657 MB read once from HBM) larger than L2; no flush; the second pass over each "
                      "pair's rows is meant to hit L2 (DRAM traffic in profiles/)"}

    def batch(self, seqs):
        from speculative_decoding_verification_52_gb300 import inputs as gen
        return gen.config_headline(seqs=seqs)

    def units(self, batch):
        return batch.B * batch.K

    def algorithmic_bytes(self, batch):
        # every target row t < K and every draft row, read once
        return 2 * batch.B * batch.K * batch.V * 2

    def oracle_call(self, batch, sl):
        import oracle
        oracle.row_stats(batch.target[sl], batch.dtype, batch.draft[sl], batch.dtype, False, batch.T)

    def device_setup(self, batch, dev):
        import torch

        import speculative_decoding_verification_52_gb300 as sv
        hs = [_bf16_host(batch.target), _bf16_host(batch.draft)]
        ds = [h.to(dev) for h in hs]
        outs = [torch.empty((batch.B, batch.K), dtype=torch.float32, device=dev) for _ in range(3)]
        stream = torch.cuda.current_stream()

        def step():
            sv.spec_row_stats(ds[0], ds[1], batch.T, alpha=outs[0], kl=outs[1], tv=outs[2], stream=stream)
        return hs, ds, step, outs


class DraftWorkload(Workload):
    name = "draft"
    metric = "drafted tree nodes/s"
    unit = "nodes/s"
    summary = "tree_draft_kernel_b128_n64_v128256_bf16.md"
    kernel = "tree_draft_kernel<bf16>"
    seq_noun = "trees drafted"
    sources = ("common.cuh", "tree_draft.cuh")
    per_rank = TREE_B

    def describe(self):
        return {"workload": "top-k tree drafting, B=128 trees of N=64 nodes (BFS [4,3,2,1] truncated), one draft "
                            "row per node, V=128256 bf16, T=0.7: each node's children take its row's top tokens",
                "B": TREE_B, "N": TREE_N, "V": V, "temperature": T, "max_children": 4,
                "l2": "rows read (1.35 GB) larger than L2; no flush"}

    def batch(self, seqs):
        from speculative_decoding_verification_52_gb300 import inputs as gen
        par, draft = gen.config_tree_draft(seqs=seqs)

        class _B:
            pass
        b = _B()
        b.B, b.N, b.parents, b.draft = draft.shape[0], draft.shape[1], par, draft
        return b

    def units(self, batch):
        return batch.B * (batch.N - 1)

    def algorithmic_bytes(self, batch):
        import numpy as np
        internal = len(set(np.asarray(batch.parents[1:]).tolist()))
        return batch.B * internal * V * 2

    def oracle_chunk(self):
        return 1

    def oracle_call(self, batch, sl):
        import numpy as np

        import oracle
        oracle.tree_draft(np.ascontiguousarray(batch.draft[sl]), "bf16", batch.parents, T, 4)

    def device_setup(self, batch, dev):
        import torch

        import speculative_decoding_verification_52_gb300 as sv
        hs = [_bf16_host(batch.draft), _pinned(batch.parents)]
        ds = [h.to(dev) for h in hs]
        tok = torch.empty((batch.B, batch.N), dtype=torch.int32, device=dev)
        lq = torch.empty((batch.B, batch.N), dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream()

        def step():
            sv.spec_tree_draft(ds[0], ds[1], T, 4, node_tokens=tok, node_logq=lq, stream=stream)
        return hs, ds, step, [tok, lq]


WORKLOADS = {w.name: w for w in (SampleWorkload(), GreedyWorkload(), TreeWorkload(), TreeMaskWorkload(),
                                 KvCommitWorkload(), StatsWorkload(), DraftWorkload(), AcceptanceWorkload(),
                                 *CHAIN_WORKLOADS)}


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_rate(wl: Workload, batch, budget_s: float, min_seqs: int, threads: int = 1):
    """The oracle, as it stands, over the batch's sequences (cycled, a few per
    call) until about budget_s of wall time; `threads` host threads each run
    their own calls (the oracle's C calls release the interpreter lock, so the
    threads run on separate cores).  Returns (units/s, sequences, seconds)."""
    import oracle
    oracle.build()
    oracle.lib()
    per_seq_units = wl.units(batch) / batch.B
    chunk = wl.oracle_chunk()
    if threads <= 1:
        done, t_used = 0, 0.0
        while t_used < budget_s or done < min_seqs:
            s0 = done % batch.B
            sl = slice(s0, min(batch.B, s0 + chunk))
            t0 = time.perf_counter()
            wl.oracle_call(batch, sl)
            t_used += time.perf_counter() - t0
            done += sl.stop - sl.start
        return done * per_seq_units / t_used, done, t_used
    from concurrent.futures import ThreadPoolExecutor
    slices = [slice(s0, min(batch.B, s0 + chunk)) for s0 in range(0, batch.B, chunk)]
    done, k = 0, 0
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as pool:
        while time.perf_counter() - t0 < budget_s or done < min_seqs:
            rnd = [slices[(k + i) % len(slices)] for i in range(threads)]
            k += threads
            list(pool.map(lambda sl: wl.oracle_call(batch, sl), rnd))
            done += sum(sl.stop - sl.start for sl in rnd)
    t_used = time.perf_counter() - t0
    return done * per_seq_units / t_used, done, t_used


def cpu_baseline(wl: Workload, batch, budget_s: float, outs=None, parity_seqs: int = 32):
    """The CPU-baseline leg: the oracle on every host core (and on one, for
    reference) over a bounded sample of the workload; when the GPU outputs are
    given, the same leg compares the first sequences' outputs with the
    oracle's (the parity block)."""
    cores = host_cores()
    rate, done, t_used = oracle_rate(wl, batch, budget_s, 4 * cores, threads=cores)
    rate1, done1, t1 = oracle_rate(wl, batch, max(1.0, budget_s / 4), 2, threads=1)
    cpu = {"value": rate, "unit": wl.unit, "cores": cores, "kind": "oracle",
           "sample": f"{done} {wl.seq_noun} (the {batch.B} of the same workload, cycled) "
                     f"on {cores} threads, {t_used:.1f} s; single-threaded double-precision C oracle per call",
           "value_1core": rate1, "sample_1core": f"{done1} {wl.seq_noun} on 1 thread, {t1:.1f} s"}
    parity = None
    if outs is not None:
        n = min(batch.B, parity_seqs)
        parity = wl.parity(batch, outs, n)
    return cpu, parity


def run_reference(args, wl: Workload, ws, rank):
    """The oracle arm: the double-precision CPU oracle on this host's cores,
    each step a bounded sample of the same workload."""
    if rank != 0:
        return
    cores = host_cores()
    per_step = wl.oracle_chunk() * cores
    batch = wl.batch(list(range(min(per_step, wl.per_rank))))
    per_step = batch.B
    for _ in range(max(0, args.warmup)):
        oracle_rate(wl, batch, 0.0, per_step, threads=cores)
    t = 0.0
    for _ in range(args.steps):
        _, _, dt = oracle_rate(wl, batch, 0.0, per_step, threads=cores)
        t += dt
    value = args.steps * wl.units(batch) / t
    sample = f"{per_step} of the {wl.per_rank} sequences per step, on {cores} threads"
    line = {"impl": "reference", "metric": wl.metric, "value": value, "unit": wl.unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.oracle_dtype,
            "data": "synthetic", "config": wl.describe(),
            "cpu_baseline": {"value": value, "unit": wl.unit, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": wl.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, wl: Workload, ws, rank, local):
    import torch

    import speculative_decoding_verification_52_gb300 as sv

    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sv.lib()

    batch = wl.batch(rank_sequences(rank, wl.per_rank))
    hs, ds, step, douts = wl.device_setup(batch, dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # the timed steps: plain calls, nothing else on the stream
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = e0.elapsed_time(e1) / args.steps

    # the same steps again with the library's timing hooks on (CUDA events
    # around the kernels of each call: part 1 = the sweep, or the whole fused
    # kernel; part 2 = the finishing kernel, none when fused) for the roofline
    sv.spec_profile_begin(args.steps * wl.launches_per_step)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    kern_ms, fin_ms, ncalls = sv.spec_profile_end()

    # end to end through the public API: pinned host inputs -> HBM -> verify -> host outputs
    houts = [torch.empty(d.shape, dtype=d.dtype).pin_memory() for d in douts]
    e2e_steps = max(3, min(args.steps, 50))

    def e2e_step():
        for h, d in zip(hs, ds):
            d.copy_(h, non_blocking=True)
        step()
        for h, d in zip(houts, douts):
            h.copy_(d, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = f0.elapsed_time(f1) / e2e_steps
    clk = clocks.stop()

    n = max(1, ncalls)
    ms, e2e_ms, kern_avg_ms, fin_avg_ms = max_over_ranks([ms, e2e_ms, kern_ms / n, fin_ms / n], ws, dev)
    if rank != 0:
        return
    peaks, src = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    alg = wl.algorithmic_bytes(batch)
    # The launch duration is taken over the timed region: a step is nothing but
    # the library's launches, back to back, so the timed region divided by the
    # launches it holds bounds each launch's duration from above (launch gaps
    # included).  Per-call events from the second pass are reported beside it;
    # they bracket every launch separately and read a little higher.
    launch_ms = ms / wl.launches_per_step
    achieved = alg / wl.launches_per_step / (launch_ms * 1e-3) / 1e9   # bytes per launch / launch time
    units = wl.units(batch)
    cpu = parity = None
    if ws == 1:
        step()   # one more call: its outputs are the ones the parity block checks
        torch.cuda.synchronize()
        cpu, parity = cpu_baseline(wl, batch, args.cpu_budget, [o.cpu().numpy() for o in douts])
    cfg = wl.describe()
    cfg["parallelism"] = f"replicas over sequences x{ws}"
    cfg["algorithmic_bytes_per_step"] = alg
    cfg["metric_GBps"] = alg / (ms * 1e-3) / 1e9
    cfg["metric_frac_of_8TBps"] = alg / (ms * 1e-3) / 8e12
    roof = {"bound": "hbm", "kernel": wl.kernel, "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "peak_source": f"{src} hbm_gbs (burst copy)",
            "traffic": profiled_traffic(wl.summary, wl.sources), "algorithmic_bytes": alg, "avg_launch_ms": launch_ms,
            "avg_launch_ms_per_call_events": kern_avg_ms}
    if wl.launches_per_step > 1:
        roof["launches_per_step"] = wl.launches_per_step
    extra = wl.extra_report(batch)
    line = {
        "metric": wl.metric, "value": ws * units / (ms * 1e-3), "unit": wl.unit, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic", "config": cfg, "roofline": roof,
        "e2e": {"value": ws * units / (e2e_ms * 1e-3), "unit": wl.unit,
                "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in hs),
                "d2h_bytes_per_step": sum(x.numel() * x.element_size() for x in houts), "ms_per_step": e2e_ms},
        # our kernels per step: one persistent kernel (plus one cudaMemsetAsync of
        # its control block)
        "gpu_launches": wl.launches_per_step * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    if parity is not None:
        line["parity"] = parity
    if extra:
        line.update(extra)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + ["sweep"], default="sample")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_setup()
    names = [f"ctl_B{b}_K{k}" for b, k in SWEEP] if args.workload == "sweep" else [args.workload]
    for name in names:
        wl = WORKLOADS[name]
        if args.impl == "reference":
            run_reference(args, wl, ws, rank)
        else:
            run_ours(args, wl, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
