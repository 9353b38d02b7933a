"""Batched search on an engine without a bf16 copy: tcgen05 kind::tf32 on
the resident fp32 corpus (fp32 queries, tf32 operands, fp32 accumulate),
through the C ABI against the oracle.

Dyadic inputs (multiples of 2^-6, at most 7 significant bits) are exact in
tf32 and their sums exact in fp32, so there the result must match bit for
bit. On unit-norm data each operand keeps 10 mantissa bits, so every score is
within 2^-9 of the exact one (the sum of |c_d q_d| is at most 1): checked at
2e-3 absolute, inside the 2e-2 rule for the reduced-precision batched path."""
import numpy as np
import pytest

import oracle
import workloads
from tests.parity import BF16_ABS, check_exact, check_float_topk, check_sorted_distinct

pytestmark = pytest.mark.gpu

TF32_ABS = 2e-3


@pytest.fixture(scope="module")
def rbf():
    import resident_brute_force_gb300 as rbf
    rbf.load_library()
    return rbf


@pytest.mark.parametrize("n,d,b,k", [
    (1000, 64, 5, 8), (300, 128, 1, 1), (4099, 768, 130, 32), (2000, 100, 256, 16), (777, 36, 300, 32),
    (70_001, 64, 40, 32),
])
def test_dyadic_bit_exact(rbf, n, d, b, k):
    c = workloads.dyadic_grid(n, d, seed=n + d)
    qs = workloads.dyadic_grid(b, d, seed=n + d + 1)
    with rbf.Engine(n, d, 32, max_batch=b) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(b):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], k))


@pytest.mark.parametrize("b", [64, 256])
def test_unit_gaussian(rbf, b):
    n, d, k = 100_003, 768, 32
    c = workloads.unit_corpus(n, d, seed=3)
    qs = workloads.unit_queries(b, d, seed=4)
    with rbf.Engine(n, d, 32, max_batch=b) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(0, b, 11):
            check_float_topk(idx[j], sc[j], oracle.scores(c, qs[j]), k, tol_abs=TF32_ABS)
        for j in range(b):
            check_sorted_distinct(idx[j].astype(np.int64), sc[j].astype(np.float64), n)


def test_dev_matches_host(rbf):
    import torch
    n, d, b = 20_000, 384, 200
    c = workloads.unit_corpus(n, d, seed=5)
    qs = workloads.unit_queries(b, d, seed=6)
    with rbf.Engine(n, d, 32, max_batch=b) as e:
        e.upload_corpus_rowmajor(c)
        h_idx, h_sc = e.search_resident_batch(qs, 32)
        dq = torch.from_numpy(qs).cuda()
        d_idx = torch.empty((b, 32), dtype=torch.int32, device="cuda")
        d_sc = torch.empty((b, 32), dtype=torch.float32, device="cuda")
        e.search_resident_batch_dev(dq, 32, d_idx, d_sc)
        torch.cuda.synchronize()
        assert np.array_equal(d_idx.cpu().numpy(), h_idx) and np.array_equal(d_sc.cpu().numpy(), h_sc)
        assert e.check_device_error() == rbf.RBF_OK


def test_cosine_tf32(rbf):
    n, d, b, k = 30_011, 256, 150, 32
    rng = np.random.default_rng(7)
    c = (workloads.gaussian_rows(n, d, 8).astype(np.float64) * rng.uniform(0.1, 10, size=n)[:, None]).astype(np.float32)
    qs = (workloads.gaussian_rows(b, d, 9).astype(np.float64) * rng.uniform(0.1, 10, size=b)[:, None]).astype(np.float32)
    with rbf.Engine(n, d, 32, max_batch=b, flags=rbf.RBF_FLAG_COSINE) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(0, b, 7):
            check_float_topk(idx[j], sc[j], oracle.scores_cosine(c, qs[j]), k, tol_abs=TF32_ABS)


def test_full_size_planted(rbf):
    """B = 256 x N = 1,000,000 x D = 768 on the fp32 corpus: planted rows lead
    for every query."""
    n, d, b, k = 1_000_000, 768, 256, 32
    c = workloads.unit_corpus(n, d, seed=1)
    qs = workloads.unit_queries(b, d, seed=2)
    planted = workloads.plant_near_duplicates(c, qs, per_query=10, noise=0.05, seed=3)
    with rbf.Engine(n, d, k, max_batch=b) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(b):
            assert set(idx[j][:10].tolist()) == set(planted[j].tolist()), j
        for j in (0, 255):
            check_float_topk(idx[j], sc[j], oracle.scores(c, qs[j]), k, tol_abs=BF16_ABS)
