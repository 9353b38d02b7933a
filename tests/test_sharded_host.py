"""Row-sharded search, host side, on CPU: the partition of the rows, the
global row offsets and the exchange of every shard's K best over two gloo
ranks, checked against the oracle on the whole corpus. Each rank's local
search is stood in for by the oracle on its shard (the GPU path is
tests/test_gpu_sharded.py); what is checked here is that partition, offsets
and exchange lose nothing: the top-K of the gathered candidates is the
whole corpus's top-K."""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from resident_brute_force_gb300.sharded import shard_rows  # noqa: E402


def test_shard_rows_partition():
    for n, world in [(10, 1), (10, 3), (1_000_000, 8), (7, 7), (1001, 4)]:
        parts = [shard_rows(n, world, r) for r in range(world)]
        assert parts[0][0] == 0
        for (r0, m), (r1, _) in zip(parts, parts[1:]):
            assert r0 + m == r1            # contiguous, rank order
        assert parts[-1][0] + parts[-1][1] == n
        sizes = [m for _, m in parts]
        assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
    for bad in [(5, 0, 0), (5, 2, 2), (5, 2, -1), (3, 4, 0)]:
        with pytest.raises(ValueError):
            shard_rows(*bad)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _corpus(kind, n, d):
    import workloads
    if kind == "gauss":
        return workloads.unit_corpus(n, d, seed=1)
    # Tie-heavy: a few distinct rows repeated across the shard boundary, so
    # equal scores in different shards must come out in global index order.
    base = workloads.dyadic_grid(37, d, seed=5)
    return base[np.arange(n) % 37]


def _worker(rank, world, port, n, d, k, kind, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        import workloads
        from resident_brute_force_gb300.sharded import exchange, shard_rows
        row0, rows = shard_rows(n, world, rank)
        if kind == "gauss":
            shard = workloads.unit_corpus_rows(row0, rows, d, seed=1)
        else:
            shard = _corpus(kind, n, d)[row0:row0 + rows]
        queries = workloads.unit_queries(3, d, seed=2)
        out = []
        for qv in queries:
            li, ls = oracle.topk(shard, qv, k)       # the shard's local top-K (local indices)
            gi = torch.from_numpy((li + row0).astype(np.int32))   # global indices
            gs = torch.from_numpy(ls.astype(np.float32))
            ai, as_ = exchange(gi, gs)
            out.append((ai.numpy().copy(), as_.numpy().copy()))
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("kind,n,d,k,world", [("gauss", 20_011, 64, 16, 2), ("ties", 5_003, 32, 50, 2),
                                              ("gauss", 3_001, 48, 100, 3)])
def test_exchange_gives_the_whole_corpus_topk(kind, n, d, k, world):
    import torch.multiprocessing as mp

    import oracle
    import workloads
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n, d, k, kind, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    corpus = _corpus(kind, n, d)
    queries = workloads.unit_queries(3, d, seed=2)
    for j, qv in enumerate(queries):
        gi, gs = got[0][j]
        assert gi.shape == (world, k)
        for r in range(1, world):       # every rank holds the same gathered lists
            assert np.array_equal(got[r][j][0], gi) and np.array_equal(got[r][j][1], gs)
        for r in range(world):          # rank r's list sits at [r], with its own rows' global indices
            r0, m = shard_rows(n, world, r)
            assert np.all((gi[r] >= r0) & (gi[r] < r0 + m))
        # The merge, done by the oracle over the gathered candidates (sorted
        # by global index, so that the oracle's tie rule on candidate
        # positions is the tie rule on global indices).
        cand = np.unique(gi.reshape(-1))
        ci, cs = oracle.topk(corpus[cand], qv, k)
        o_idx, o_sc = oracle.topk(corpus, qv, k)
        assert np.array_equal(cand[ci], o_idx) and np.array_equal(cs, o_sc)
