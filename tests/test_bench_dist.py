"""bench.py's multi-rank host logic on CPU with the gloo backend, world size 2:
disjoint per-rank sequence sets (replicas over sequences, no exchange), the
max-over-ranks timing reduction, and the torchrun launch of the oracle arm
(rank 0 prints the one JSON line, the other rank exits 0 without work)."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        seqs = bench.rank_sequences(rank, 256)
        # per-rank timings that differ by rank; the job's time is the slowest rank's
        mine = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)]
        red = bench.max_over_ranks(mine, ws)
        q.put((rank, seqs[0], seqs[-1], len(seqs), red))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_rank_sharding_and_max_reduction_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, a0, z0, n0, red0), (r1, a1, z1, n1, red1) = res
    assert (a0, z0, n0) == (0, 255, 256) and (a1, z1, n1) == (256, 511, 256)   # disjoint, same size
    assert red0 == red1 == [2.0, 5.0, 0.5]


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3, 1.5], 1) == [3.0, 1.5]
    assert bench.rank_sequences(0, 4) == [0, 1, 2, 3]


def test_reference_arm_under_torchrun_two_ranks():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--gpus", "2", "--impl", "reference",
           "--workload", "greedy", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
