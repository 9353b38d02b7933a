"""Parity on shapes drawn at random (fixed seed): corpus sizes from a few
hundred rows to past the batched pre-pass threshold, D from 1 to 1,100 (odd
and ragged widths included), every K bucket, batches of 1 to 256 queries, the
three float paths (fp32 single query, bf16 and tf32 batched). Dyadic data make
every score exact on every path, so each sampled query must equal the oracle
bit for bit; the batched host call must also equal its device variant."""
import numpy as np
import pytest

import oracle
import workloads
from tests.parity import check_exact

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rbf():
    import resident_brute_force_gb300 as rbf
    rbf.load_library()
    return rbf


def _shapes(seed, count, n_max):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        n = int(rng.integers(257, n_max))
        d = int(rng.choice([1, 3, 7, 64, 96, 130, 257, 384, 768, 1024, 1100]))
        k = int(min(n, rng.choice([1, 5, 8, 16, 31, 32, 33, 64, 100, 129, 256])))
        b = int(rng.choice([1, 2, 17, 64, 129, 256]))
        out.append((n, d, b, k))
    return out


@pytest.mark.parametrize("n,d,b,k", _shapes(2026, 8, 40_000))
def test_single_query_random_shapes(rbf, n, d, b, k):
    c = workloads.dyadic_grid(n, d, seed=n + 3 * d)
    qs = workloads.dyadic_grid(3, d, seed=n + 3 * d + 1)
    with rbf.Engine(n, d, 256) as e:
        e.upload_corpus_rowmajor(c)
        for q in qs:
            check_exact(*e.search_resident(q, k), *oracle.topk(c, q, k))


@pytest.mark.parametrize("kind", ["bf16", "tf32"])
@pytest.mark.parametrize("n,d,b,k", _shapes(2027, 5, 30_000) + [(90_001, 64, 40, 32), (70_144, 130, 9, 100)])
def test_batched_random_shapes(rbf, kind, n, d, b, k):
    import torch
    c = workloads.dyadic_grid(n, d, seed=n + 5 * d)
    qs = workloads.dyadic_grid(b, d, seed=n + 5 * d + 1)
    flags = rbf.RBF_FLAG_BF16_CORPUS if kind == "bf16" else 0
    with rbf.Engine(n, d, 256, max_batch=b, flags=flags) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        di = torch.empty((b, k), dtype=torch.int32, device="cuda")
        ds = torch.empty((b, k), dtype=torch.float32, device="cuda")
        e.search_resident_batch_dev(torch.from_numpy(qs).cuda(), k, di, ds)
        torch.cuda.synchronize()
        assert np.array_equal(di.cpu().numpy(), idx) and np.array_equal(ds.cpu().numpy(), sc)
        for j in sorted({0, b - 1, b // 2}):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], k))
