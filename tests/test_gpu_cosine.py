"""Cosine mode (RBF_FLAG_COSINE) through the C ABI against the oracle's
cosine: the inner product over the product of the L2 norms, -inf for a
non-positive denominator (GPU-Resident Top-K for Agentic RAG, section 4 step
2, cosine mode). The engine divides rows by their norms at upload and the
query at every call; scores follow the fp32 rule (1e-5 relative, 1e-2
floor), batched scores the bf16 rules."""
import numpy as np
import pytest

import oracle
import workloads
from tests.parity import BF16_ABS, check_float_topk, check_sorted_distinct

pytestmark = pytest.mark.gpu

BF16_ACC_ABS = 1e-4


@pytest.fixture(scope="module")
def rbf():
    import resident_brute_force_gb300 as rbf
    rbf.load_library()
    return rbf


def scaled_rows(n, d, seed, lo=0.1, hi=10.0):
    """Gaussian rows times a per-row scale in [lo, hi]: cosine and inner
    product rank them differently."""
    rng = np.random.default_rng(seed)
    g = workloads.gaussian_rows(n, d, seed)
    s = rng.uniform(lo, hi, size=n)
    return (g.astype(np.float64) * s[:, None]).astype(np.float32)


@pytest.mark.parametrize("d", [384, 1024, 100, 3])
def test_scaled_rows_match_oracle(rbf, d):
    n = 20011
    c = scaled_rows(n, d, seed=d)
    qs = scaled_rows(4, d, seed=d + 1)
    with rbf.Engine(n, d, 256, flags=rbf.RBF_FLAG_COSINE) as e:
        e.upload_corpus_rowmajor(c)
        for j, k in enumerate((1, 8, 100, 256)):
            idx, sc = e.search_resident(qs[j], k)
            check_float_topk(idx, sc, oracle.scores_cosine(c, qs[j]), k)


def test_power_of_two_copies_tie_by_index(rbf):
    """Copies of one row scaled by powers of two have bit-identical cosines,
    so they tie and come back in index order."""
    n, d = 5000, 768
    c = scaled_rows(n, d, seed=5)
    pos = [11, 900, 2500, 4999]
    for p, s in zip(pos, (1.0, 4.0, 0.125, 1024.0)):
        c[p] = c[77] * np.float32(s)
    q = c[77] * np.float32(3.0) + np.float32(0.01) * scaled_rows(1, d, seed=6)[0]
    with rbf.Engine(n, d, 32, flags=rbf.RBF_FLAG_COSINE) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident(q, 8)
        assert idx[:5].tolist() == [11, 77, 900, 2500, 4999]
        assert len(set(sc[:5].tolist())) == 1
        check_float_topk(idx, sc, oracle.scores_cosine(c, q), 8)


def test_zero_rows_and_zero_query(rbf):
    n, d = 250, 64
    c = scaled_rows(n, d, seed=7)
    zero = [0, 5, 150, 249]
    c[zero] = 0.0
    q = scaled_rows(1, d, seed=8)[0]
    with rbf.Engine(n, d, 256, flags=rbf.RBF_FLAG_COSINE) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident(q, n)
        assert idx[-4:].tolist() == zero and np.all(np.isneginf(sc[-4:]))
        check_float_topk(idx[:n - 4], sc[:n - 4], oracle.scores_cosine(c, q), n - 4)
        idx, sc = e.search_resident(np.zeros(d, np.float32), 10)
        assert idx.tolist() == list(range(10)) and np.all(np.isneginf(sc))
        o_idx, o_sc = oracle.topk_cosine(c, np.zeros(d, np.float32), 10)
        assert o_idx.tolist() == idx.tolist() and np.all(np.isneginf(o_sc))


def test_device_entry_points_match_host(rbf):
    import torch
    n, d = 30000, 1024
    c = scaled_rows(n, d, seed=9)
    q = scaled_rows(1, d, seed=10)[0]
    with rbf.Engine(n, d, 64, flags=rbf.RBF_FLAG_COSINE) as e:
        e.upload_corpus_rowmajor(c)
        h_idx, h_sc = e.search_resident(q, 64)
        dq = torch.from_numpy(q).cuda()
        d_idx = torch.empty(64, dtype=torch.int32, device="cuda")
        d_sc = torch.empty(64, dtype=torch.float32, device="cuda")
        for _ in range(2):
            e.search_resident_dev(dq, 64, d_idx, d_sc)
            torch.cuda.synchronize()
            assert np.array_equal(d_idx.cpu().numpy(), h_idx) and np.array_equal(d_sc.cpu().numpy(), h_sc)
        assert e.check_device_error() == rbf.RBF_OK


def test_planted_rows_with_random_scales(rbf):
    """Planted near-duplicates scaled by random factors: the inner product
    would rank the large-scale rows first, cosine ranks the planted rows."""
    n, d = 200_000, 768
    c = workloads.unit_corpus(n, d, seed=11)
    qs = workloads.unit_queries(3, d, seed=12)
    planted = workloads.plant_near_duplicates(c, qs, per_query=10, noise=0.05, seed=13)
    rng = np.random.default_rng(14)
    c = (c.astype(np.float64) * rng.uniform(0.05, 20.0, size=n)[:, None]).astype(np.float32)
    with rbf.Engine(n, d, 32, flags=rbf.RBF_FLAG_COSINE) as e:
        e.upload_corpus_rowmajor(c)
        for j in range(3):
            idx, sc = e.search_resident(qs[j], 32)
            assert set(idx[:10].tolist()) == set(planted[j].tolist())
            check_float_topk(idx, sc, oracle.scores_cosine(c, qs[j]), 32)


def _unit_bf16(x):
    """Unit length in double, fp32, then bf16: the inputs the tensor cores
    multiply in cosine mode (up to the last bit of the norms)."""
    x64 = x.astype(np.float64)
    nrm = np.sqrt(np.sum(x64 * x64, axis=1, keepdims=True))
    return oracle.round_bf16((x64 / nrm).astype(np.float32))


@pytest.mark.parametrize("b", [64, 200])
def test_batched_cosine(rbf, b):
    n, d, k = 70_001, 384, 32
    c = scaled_rows(n, d, seed=15)
    qs = scaled_rows(b, d, seed=16)
    c16 = _unit_bf16(c)
    q16 = _unit_bf16(qs)
    with rbf.Engine(n, d, 32, max_batch=b, flags=rbf.RBF_FLAG_BF16_CORPUS | rbf.RBF_FLAG_COSINE) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(0, b, 13):
            check_float_topk(idx[j], sc[j], oracle.scores_cosine(c, qs[j]), k, tol_abs=BF16_ABS)
            check_float_topk(idx[j], sc[j], oracle.scores(c16, q16[j]), k, tol_abs=BF16_ACC_ABS)
        for j in range(b):
            check_sorted_distinct(idx[j].astype(np.int64), sc[j].astype(np.float64), n)
