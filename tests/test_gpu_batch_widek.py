"""Batched search with 32 < K <= 256 through the C ABI against the oracle.

For K above 32 each epilogue thread keeps its best-first list in the partials
buffer (global memory) instead of registers, with its length beside it, and
the merge reads only each list's valid prefix. Both engine kinds are covered:
bf16 copy (kind::f16) and fp32 only (kind::tf32). Dyadic inputs are exact in
both and their sums exact in fp32, so there the result must match the oracle
bit for bit, ties and order included.
"""
import numpy as np
import pytest

import oracle
import workloads
from tests.parity import BF16_ABS, check_exact, check_float_topk, check_sorted_distinct

pytestmark = pytest.mark.gpu

BF16_ACC_ABS = 1e-4
KINDS = ["bf16", "tf32"]


@pytest.fixture(scope="module")
def rbf():
    import resident_brute_force_gb300 as rbf
    rbf.load_library()
    return rbf


def engine(rbf, kind, n, d, b, k=256, cosine=False):
    flags = rbf.RBF_FLAG_BF16_CORPUS if kind == "bf16" else rbf.RBF_FLAG_FP32_CORPUS
    if cosine:
        flags |= rbf.RBF_FLAG_COSINE
    return rbf.Engine(n, d, k, max_batch=b, flags=flags)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("n,d,b,k", [
    (1000, 64, 5, 33), (300, 128, 1, 128), (4099, 768, 130, 100), (2000, 100, 256, 256), (777, 64, 300, 64),
    (256, 64, 3, 256),
])
def test_dyadic_bit_exact(rbf, kind, n, d, b, k):
    c = workloads.dyadic_grid(n, d, seed=n + d)
    qs = workloads.dyadic_grid(b, d, seed=n + d + 1)
    with engine(rbf, kind, n, d, b) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(b):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], k))


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("k", [100, 256])
def test_sample_bound_dyadic_exact(rbf, kind, k):
    """N >= 65,536: the bound from the first 16,384 rows (the K-th largest of
    512 chunk maxima) is in force in the main pass."""
    n, d, b = 70_001, 64, 40
    c = workloads.dyadic_grid(n, d, seed=31)
    qs = workloads.dyadic_grid(b, d, seed=32)
    with engine(rbf, kind, n, d, b) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(b):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], k))


@pytest.mark.parametrize("k", [64, 100, 256])
def test_large_sample_dyadic_exact(rbf, k):
    """N = 300,000: the sample grows with K (32,768 rows at K = 64, 65,536
    at K = 100 and 256, capped at a quarter of N), several 128-row tiles per
    CTA folded into each chunk maximum."""
    n, d, b = 300_000, 64, 24
    c = workloads.dyadic_grid(n, d, seed=33)
    qs = workloads.dyadic_grid(b, d, seed=34)
    with engine(rbf, "bf16", n, d, b) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(b):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], k))


@pytest.mark.parametrize("kind", KINDS)
def test_ascending_scores_every_row_beats_the_list(rbf, kind):
    """Row i is (alpha_i, 0, ..., 0) with alpha_i = floor(255 i / n): along +e0
    every row a thread meets beats its whole list, so each flush shifts the
    full list; along -e0 the first rows win and every later row is dropped."""
    n, d, k = 80_000, 64, 200
    c = np.zeros((n, d), dtype=np.float32)
    c[:, 0] = np.floor(np.arange(n) * 255.0 / n)
    e0 = np.zeros(d, dtype=np.float32)
    e0[0] = 1.0
    qs = np.stack([e0, -e0, workloads.dyadic_grid(1, d, seed=42)[0]])
    with engine(rbf, kind, n, d, 3) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(3):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], k))
        first = int(np.argmax(c[:, 0] == 254.0))
        assert idx[0][:32].tolist() == list(range(first, first + 32))
        assert idx[1].tolist() == list(range(k))


@pytest.mark.parametrize("kind", KINDS)
def test_all_equal_rows(rbf, kind):
    n, d, k = 70_000, 64, 256
    c = np.full((n, d), 0.25, dtype=np.float32)
    qs = np.ones((2, d), dtype=np.float32)
    with engine(rbf, kind, n, d, 2) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        assert idx[0].tolist() == list(range(k)) and idx[1].tolist() == list(range(k))
        assert np.all(sc == 16.0)


@pytest.mark.parametrize("n", [20_011, 100_003])
def test_unit_gaussian_both_references(rbf, n):
    d, b, k = 768, 256, 100
    c = workloads.unit_corpus(n, d, seed=1)
    qs = workloads.unit_queries(b, d, seed=2)
    c16 = oracle.round_bf16(c)
    q16 = oracle.round_bf16(qs)
    with engine(rbf, "bf16", n, d, b) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(0, b, 17):
            check_float_topk(idx[j], sc[j], oracle.scores(c16, q16[j]), k, tol_abs=BF16_ACC_ABS)
            check_float_topk(idx[j], sc[j], oracle.scores(c, qs[j]), k, tol_abs=BF16_ABS)


def test_many_groups_dev_matches_host(rbf):
    """1,000 queries = four 256-query groups, each scored and merged in turn
    through the same partials buffer; the device-pointer call and repeated
    calls give the same bytes."""
    import torch
    n, d, b, k = 5000, 64, 1000, 256
    c = workloads.dyadic_grid(n, d, seed=51)
    qs = workloads.dyadic_grid(b, d, seed=52)
    with engine(rbf, "bf16", n, d, b) as e:
        e.upload_corpus_rowmajor(c)
        h_idx, h_sc = e.search_resident_batch(qs, k)
        for j in range(0, b, 37):
            check_exact(h_idx[j], h_sc[j], *oracle.topk(c, qs[j], k))
        dq = torch.from_numpy(qs).cuda()
        d_idx = torch.empty((b, k), dtype=torch.int32, device="cuda")
        d_sc = torch.empty((b, k), dtype=torch.float32, device="cuda")
        for _ in range(2):
            e.search_resident_batch_dev(dq, k, d_idx, d_sc)
            torch.cuda.synchronize()
            assert np.array_equal(d_idx.cpu().numpy(), h_idx)
            assert np.array_equal(d_sc.cpu().numpy(), h_sc)
        # K <= 32 after K > 32 on the same engine, and back.
        idx8, sc8 = e.search_resident_batch(qs[:50], 8)
        for j in range(50):
            check_exact(idx8[j], sc8[j], *oracle.topk(c, qs[j], 8))
        idx2, sc2 = e.search_resident_batch(qs, k)
        assert np.array_equal(idx2, h_idx) and np.array_equal(sc2, h_sc)
        assert e.check_device_error() == rbf.RBF_OK


def test_cosine_wide(rbf):
    n, d, b, k = 3000, 96, 20, 150
    c = workloads.dyadic_grid(n, d, seed=61) * np.float32(3.0)
    qs = workloads.dyadic_grid(b, d, seed=62)
    with engine(rbf, "bf16", n, d, b, cosine=True) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(b):
            sig = oracle.scores_cosine(c, qs[j])
            check_float_topk(idx[j], sc[j], sig, k, tol_abs=BF16_ABS)


def test_k_limits(rbf):
    c = workloads.dyadic_grid(500, 64, seed=21)
    qs = workloads.dyadic_grid(4, 64, seed=22)
    with engine(rbf, "bf16", 500, 64, 4, k=100) as e:
        e.upload_corpus_rowmajor(c)
        for bad in (101, 0):
            with pytest.raises(rbf.RbfError) as ei:
                e.search_resident_batch(qs, bad)
            assert ei.value.status == rbf.RBF_ERR_INVALID_VALUE
        idx, sc = e.search_resident_batch(qs, 100)
        for j in range(4):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], 100))


def test_full_size_planted_k100(rbf):
    """B = 256 x N = 1,000,000 x D = 768 at K = 100 with 10 planted
    near-duplicates per query: they lead for every query; sampled queries
    match both references."""
    n, d, b, k = 1_000_000, 768, 256, 100
    c = workloads.unit_corpus(n, d, seed=1)
    qs = workloads.unit_queries(b, d, seed=2)
    planted = workloads.plant_near_duplicates(c, qs, per_query=10, noise=0.05, seed=3)
    with engine(rbf, "bf16", n, d, b, k=k) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(b):
            assert set(idx[j][:10].tolist()) == set(planted[j].tolist()), j
            check_sorted_distinct(idx[j].astype(np.int64), sc[j].astype(np.float64), n)
        c16 = oracle.round_bf16(c)
        for j in (0, 131):
            q16 = oracle.round_bf16(qs[j])
            check_float_topk(idx[j], sc[j], oracle.scores(c16, q16), k, tol_abs=BF16_ACC_ABS)
            check_float_topk(idx[j], sc[j], oracle.scores(c, qs[j]), k, tol_abs=BF16_ABS)


@pytest.mark.parametrize("sample", [0, 256, 16_384, 49_152, 70_144])
@pytest.mark.parametrize("k", [8, 32, 100])
def test_sample_option_changes_nothing(rbf, sample, k):
    """RBF_OPT_BATCH_SAMPLE picks the pre-pass rows (0: none; up to all of
    N): the result is bit-identical to the automatic choice and exact."""
    n, d, b = 70_144, 64, 12
    c = workloads.dyadic_grid(n, d, seed=71)
    qs = workloads.dyadic_grid(b, d, seed=72)
    with engine(rbf, "bf16", n, d, b) as e:
        e.upload_corpus_rowmajor(c)
        ref_idx, ref_sc = e.search_resident_batch(qs, k)
        e.set_option(rbf.RBF_OPT_BATCH_SAMPLE, sample)
        idx, sc = e.search_resident_batch(qs, k)
        assert np.array_equal(idx, ref_idx) and np.array_equal(sc, ref_sc)
        for j in range(0, b, 5):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], k))
        for bad in (-2, 100):
            with pytest.raises(rbf.RbfError):
                e.set_option(rbf.RBF_OPT_BATCH_SAMPLE, bad)
