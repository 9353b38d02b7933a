"""Row-sharded search on one GPU through the C ABI: G engines, each holding
one contiguous row shard (upload_corpus_shard, global row offsets), each
searched on its own, the G lists merged by merge_shard_topk_dev. The result
must be what the oracle gives on the whole corpus: bit for bit on dyadic
data (exact scores, heavy ties across shard boundaries), within the fp32 rule
on the 1M x 1024 planted configuration. On several GPUs the lists travel
through one all-gather instead of a device copy (resident_brute_force_gb300
.sharded); the kernels are the same."""
import os

import numpy as np
import pytest

import oracle
import workloads
from tests.parity import check_exact, check_float_topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rbf():
    import resident_brute_force_gb300 as rbf
    rbf.load_library()
    return rbf


def _shard_engines(rbf, corpus, g, max_k=256, max_batch=1, flags=0, bounds=None):
    from resident_brute_force_gb300.sharded import shard_rows
    n = corpus.shape[0]
    bounds = bounds or [shard_rows(n, g, r) for r in range(g)]
    engines = []
    for r0, m in bounds:
        e = rbf.Engine(m, corpus.shape[1], max_k, max_batch=max_batch, flags=flags)
        e.upload_corpus_shard(corpus[r0:r0 + m], r0)
        engines.append(e)
    return engines, bounds


def _sharded_search(engines, bounds, q, k):
    """Every shard's top-min(K, rows) into slot s of a [G, K] buffer (missing
    entries -1), then the merge on engine 0."""
    import torch
    g = len(engines)
    gi = torch.full((g, k), -1, dtype=torch.int32, device="cuda")
    gs = torch.zeros((g, k), dtype=torch.float32, device="cuda")
    dq = torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32)).cuda()
    for s, (e, (_, m)) in enumerate(zip(engines, bounds)):
        ks = min(k, m)
        e.search_resident_dev(dq, ks, gi[s, :ks], gs[s, :ks])
    torch.cuda.synchronize()
    oi = torch.empty(k, dtype=torch.int32, device="cuda")
    osc = torch.empty(k, dtype=torch.float32, device="cuda")
    engines[0].merge_shard_topk_dev(gi, gs, k, oi, osc)
    torch.cuda.synchronize()
    return oi.cpu().numpy(), osc.cpu().numpy()


def _close(engines):
    for e in engines:
        e.close()


@pytest.mark.parametrize("g", [2, 4])
def test_dyadic_shards_bit_exact(rbf, g):
    n, d = 40_003, 128
    rng = np.random.default_rng(3)
    base = workloads.dyadic_grid(2_000, d, seed=81)
    c = base[rng.integers(0, 2_000, size=n)]   # every row has duplicates, most in other shards
    qs = workloads.dyadic_grid(3, d, seed=82)
    engines, bounds = _shard_engines(rbf, c, g)
    try:
        for q in qs:
            for k in (1, 8, 33, 100, 256):
                check_exact(*_sharded_search(engines, bounds, q, k), *oracle.topk(c, q, k))
    finally:
        _close(engines)


def test_shard_smaller_than_k(rbf):
    """A shard of 40 rows answers with 40 entries and pads its list with -1."""
    n, d = 9_000, 64
    c = workloads.dyadic_grid(n, d, seed=83)
    bounds = [(0, 4_000), (4_000, 40), (4_040, 4_960)]
    engines, bounds = _shard_engines(rbf, c, 3, bounds=bounds)
    q = workloads.dyadic_grid(1, d, seed=84)[0]
    try:
        for k in (32, 100, 256):
            check_exact(*_sharded_search(engines, bounds, q, k), *oracle.topk(c, q, k))
    finally:
        _close(engines)


def test_views_and_batched_shards(rbf):
    """Views of a shard engine report global indices too, and the batched
    path (bf16 tensor cores; exact on dyadic data) merges [G, B, K] lists."""
    import torch
    n, d, b, k = 30_011, 64, 40, 16
    c = workloads.dyadic_grid(n, d, seed=85)
    qs = workloads.dyadic_grid(b, d, seed=86)
    engines, bounds = _shard_engines(rbf, c, 2, max_k=32, max_batch=b, flags=rbf.RBF_FLAG_BF16_CORPUS)
    try:
        with engines[1].view() as v:
            idx, sc = v.search_resident(qs[0], k)
            r0, m = bounds[1]
            o_idx, o_sc = oracle.topk(c[r0:r0 + m], qs[0], k)
            check_exact(idx, sc, o_idx + r0, o_sc)
        dq = torch.from_numpy(qs).cuda()
        gi = torch.empty((2, b, k), dtype=torch.int32, device="cuda")
        gs = torch.empty((2, b, k), dtype=torch.float32, device="cuda")
        for s, e in enumerate(engines):
            e.search_resident_batch_dev(dq, k, gi[s], gs[s])
        torch.cuda.synchronize()
        oi = torch.empty((b, k), dtype=torch.int32, device="cuda")
        osc = torch.empty((b, k), dtype=torch.float32, device="cuda")
        engines[0].merge_shard_topk_dev(gi, gs, k, oi, osc)
        torch.cuda.synchronize()
        oi, osc = oi.cpu().numpy(), osc.cpu().numpy()
        for j in range(b):
            check_exact(oi[j], osc[j], *oracle.topk(c, qs[j], k))
    finally:
        _close(engines)


def test_full_size_planted_four_shards(rbf):
    """The 1,000,000 x 1024 planted configuration split into 4 shards of
    250,000 rows: planted rows lead, and sampled queries meet the fp32 rule
    against the oracle on the whole corpus."""
    n, d, nq = 1_000_000, 1024, 1000
    c = workloads.unit_corpus(n, d, seed=1)
    qs = workloads.unit_queries(nq, d, seed=2)
    planted = workloads.plant_near_duplicates(c, qs, per_query=10, noise=0.05, seed=3)
    engines, bounds = _shard_engines(rbf, c, 4)
    try:
        for j in range(0, nq, 50):
            idx, _ = _sharded_search(engines, bounds, qs[j], 32)
            assert set(idx[:10].tolist()) == set(planted[j].tolist()), j
        for j in (0, 999):
            sigma = oracle.scores(c, qs[j])
            for k in (8, 32, 100):
                check_float_topk(*_sharded_search(engines, bounds, qs[j], k), sigma, k)
    finally:
        _close(engines)


def test_shard_argument_errors(rbf):
    import torch
    c = workloads.dyadic_grid(100, 16, seed=87)
    with rbf.Engine(100, 16, 64, max_batch=2) as e:
        for off in (-1, 2**31 - 100):
            with pytest.raises(rbf.RbfError) as ei:
                e.upload_corpus_shard(c, off)
            assert ei.value.status == rbf.RBF_ERR_INVALID_VALUE
        e.upload_corpus_shard(c, 2**31 - 101)        # the last row is 2^31 - 2
        idx, _ = e.search_resident(c[5], 4)
        assert np.all(idx >= 2**31 - 101)
        gi = torch.zeros((2, 8), dtype=torch.int32, device="cuda")
        gs = torch.zeros((2, 8), dtype=torch.float32, device="cuda")
        oi = torch.empty(8, dtype=torch.int32, device="cuda")
        osc = torch.empty(8, dtype=torch.float32, device="cuda")
        lib = e.lib
        for g, b, k in ((0, 1, 8), (2, 0, 8), (2, 3, 8), (2, 1, 65), (2, 1, 0), (1025, 1, 8)):
            assert lib.merge_shard_topk_dev(e._h, gi.data_ptr(), gs.data_ptr(), g, b, k, oi.data_ptr(),
                                            osc.data_ptr()) == rbf.RBF_ERR_INVALID_VALUE, (g, b, k)
        assert e.check_device_error() == rbf.RBF_OK


_ONE_RANK = r'''
import os, sys, json
sys.path.insert(0, os.getcwd())
import numpy as np, torch, torch.distributed as dist
import oracle, workloads
import resident_brute_force_gb300 as rbf
from resident_brute_force_gb300.sharded import ShardedSearch
torch.cuda.set_device(0)
dist.init_process_group("nccl", rank=0, world_size=1)
n, d = 20_011, 64
c = workloads.dyadic_grid(n, d, seed=88)
qs = workloads.dyadic_grid(4, d, seed=89)
s = ShardedSearch(rbf, n, d, 128, 1, 0)
s.upload(c[s.row0:s.row0 + s.rows])
ok = True
for q in qs:
    for k in (1, 16, 128):
        idx, sc = s.search(q, k)
        o_idx, o_sc = oracle.topk(c, q, k)
        ok = ok and np.array_equal(idx.astype(np.int64), o_idx) and np.array_equal(sc.astype(np.float64), o_sc)
s.close()
dist.destroy_process_group()
print("RESULT " + json.dumps({"ok": bool(ok)}), flush=True)
'''


def test_sharded_search_one_rank_nccl(tmp_path):
    """ShardedSearch end to end in a one-rank NCCL group (its own process):
    the local search, the all-gather and the merge, bit for bit against the
    oracle. Several ranks need several GPUs; their host logic is
    tests/test_sharded_host.py."""
    import json
    import socket
    import subprocess
    import sys
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), NCCL_NVLS_ENABLE="0")
    r = subprocess.run([sys.executable, "-c", _ONE_RANK], cwd=root, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    # Libraries may print to stdout too: the result is the line marked RESULT.
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")]
    assert lines, r.stdout[-2000:] + r.stderr[-2000:]
    assert json.loads(lines[-1][len("RESULT "):])["ok"]
