#!/usr/bin/env python
"""Benchmark of batched draft-token verification on GB300.

Default workload ("sample"): one step = one spec_verify_sample call over the
B=256, V=128256, K=5, bf16, T=0.7 batch (target logits [256,6,128256], draft
logits [256,5,128256]): the vocabulary sweep over all 2816 rows plus the
per-sequence accept scan and replacement/bonus draw, all inside one persistent
kernel launch (after a small memset of the workspace's control block).

Other workloads (--workload):
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
uses.  Every workload's inputs are larger
than the L2 cache (129 MB), so no flush is needed between steps.

Reported: the metric (verified draft positions/s; tree: candidate nodes/s),
the dominant kernel's achieved HBM bandwidth against the measured copy peak
(roofline), an end-to-end figure with host<->device copies inside the timed
region, the SM clocks seen during the run, and the double-precision CPU
oracle timed on a bounded sample on this host.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload sample|greedy|tree|treemask|kvcommit|stats|draft]
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
    kernel = "tree_mask_reg_kernel<8>"
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
    summary = "row_stats_kernel_b256_v128256_k5_bf16.md"
    kernel = "row_stats_kernel<bf16, bf16 logits>"
    sources = ("common.cuh", "row_stats.cuh")

    def describe(self):
        return {"workload": "acceptance statistics (sum min(p,q), KL(q||p), TV) per drafted position, B=256 "
                            "V=128256 K=5 bf16 T=0.7, the headline sampling inputs", "B": B, "V": V, "K": K,
                "temperature": T, "input_bytes": 2 * B * K * V * 2,
                "l2": "inputs (657 MB read) larger than L2; no flush"}

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
    kernel = "tree_draft_kernel<bf16, 4>"
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
                                 KvCommitWorkload(), StatsWorkload(), DraftWorkload())}


def oracle_rate(wl: Workload, batch, budget_s: float, min_seqs: int):
    """The oracle, as it stands, over the batch's sequences (cycled, a few per
    call) until about budget_s of CPU work; returns (units/s, sequences, seconds)."""
    import oracle
    oracle.build()
    per_seq_units = wl.units(batch) / batch.B
    done, t_used = 0, 0.0
    while t_used < budget_s or done < min_seqs:
        s0 = done % batch.B
        sl = slice(s0, min(batch.B, s0 + wl.oracle_chunk()))
        t0 = time.perf_counter()
        wl.oracle_call(batch, sl)
        t_used += time.perf_counter() - t0
        done += sl.stop - sl.start
    return done * per_seq_units / t_used, done, t_used


def run_reference(args, wl: Workload, ws, rank):
    """The oracle arm: the double-precision CPU oracle on this host's cores,
    each step a bounded sample of the same workload."""
    if rank != 0:
        return
    per_step = wl.oracle_chunk()
    batch = wl.batch(list(range(per_step)))
    for _ in range(max(0, args.warmup)):
        oracle_rate(wl, batch, 0.0, per_step)
    t = 0.0
    for _ in range(args.steps):
        _, _, dt = oracle_rate(wl, batch, 0.0, per_step)
        t += dt
    value = args.steps * wl.units(batch) / t
    sample = f"{per_step} of the {wl.per_rank} sequences per step"
    line = {"impl": "reference", "metric": wl.metric, "value": value, "unit": wl.unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.oracle_dtype,
            "data": "synthetic", "config": wl.describe(),
            "cpu_baseline": {"value": value, "unit": wl.unit, "cores": 1, "kind": "oracle", "sample": sample},
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
    sv.spec_profile_begin(args.steps)
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
    achieved = alg / (kern_avg_ms * 1e-3) / 1e9
    units = wl.units(batch)
    cpu = None
    if ws == 1:
        cpu_rate, done, cpu_t = oracle_rate(wl, batch, args.cpu_budget, 4)
        cpu = {"value": cpu_rate, "unit": wl.unit, "cores": 1, "kind": "oracle",
               "sample": f"{done} sequence verifications (the {batch.B} sequences of the same workload, cycled), "
                         f"single-threaded double-precision C oracle, {cpu_t:.1f} s"}
    cfg = wl.describe()
    cfg["parallelism"] = f"replicas over sequences x{ws}"
    cfg["algorithmic_bytes_per_step"] = alg
    cfg["metric_GBps"] = alg / (ms * 1e-3) / 1e9
    cfg["metric_frac_of_8TBps"] = alg / (ms * 1e-3) / 8e12
    roof = {"bound": "hbm", "kernel": wl.kernel, "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "peak_source": f"{src} hbm_gbs (burst copy)",
            "traffic": profiled_traffic(wl.summary, wl.sources), "algorithmic_bytes": alg, "avg_launch_ms": kern_avg_ms}
    if wl.launches_per_step > 1:
        roof["finish_avg_ms"] = fin_avg_ms
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
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="sample")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    wl = WORKLOADS[args.workload]
    ws, rank, local = dist_setup()
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
