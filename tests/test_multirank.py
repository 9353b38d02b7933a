"""bench.py's multi-rank logic on CPU: two gloo ranks on 127.0.0.1. The path
shards as independent replicas (no data-path collective); the only
cross-rank operations are the barrier around the timed region and the
max-over-ranks of the elapsed time, and the reference arm runs on rank 0
alone."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        dist.barrier()
        q.put((rank, bench.max_over_ranks(1.0 + 2.5 * rank, world), bench.max_over_ranks(7.0 - rank, world)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert got == [(0, 3.5, 7.0), (1, 3.5, 7.0)]


def test_max_over_ranks_single():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.25, 1) == 4.25


def test_reference_arm_two_ranks():
    """torch.distributed.run with 2 ranks: rank 0 prints one JSON line for
    the reference arm, rank 1 exits 0 without output."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "2", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_single_rank_line():
    """The reference arm at N = 1: one JSON line with the contract's keys, the
    CPU-baseline record describing this run, and zero-byte e2e transfers."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in rec, key
    assert rec["impl"] == "reference" and rec["n_gpus"] == 1 and rec["steps"] == 2 and rec["value"] > 0
    cpu = rec["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == rec["value"] and cpu["cores"] >= 1 and cpu["sample"]
    assert rec["e2e"] == {"value": rec["value"], "unit": rec["unit"], "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}
    # The same configuration as the GPU arm's line, key for key.
    sys.path.insert(0, ROOT)
    import bench
    assert rec["config"] == bench.headline_config(bench.parse([]), 1)
