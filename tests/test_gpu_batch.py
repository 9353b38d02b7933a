"""Batched search (tcgen05 bf16 scoring + fused epilogue select) through the C
ABI against the oracle.

Two references: the oracle on the original fp32 data (the true answer; rule:
2e-2 absolute on unit-norm data) and the oracle on the bf16-rounded corpus and
queries (what the tensor cores multiply; products are exact in fp32, so only
the fp32 accumulation differs: 1e-4 absolute). Dyadic inputs are exact in bf16
and their sums exact in fp32, so there the result must match bit for bit.
"""
import numpy as np
import pytest

import oracle
import workloads
from tests.parity import BF16_ABS, check_exact, check_float_topk, check_sorted_distinct

pytestmark = pytest.mark.gpu

BF16_ACC_ABS = 1e-4


@pytest.fixture(scope="module")
def rbf():
    import resident_brute_force_gb300 as rbf
    rbf.load_library()
    return rbf


def engine(rbf, n, d, b, k=32):
    return rbf.Engine(n, d, k, max_batch=b, flags=rbf.RBF_FLAG_BF16_CORPUS)


@pytest.mark.parametrize("n,d,b,k", [
    (1000, 64, 5, 8), (300, 128, 1, 1), (4099, 768, 130, 32), (2000, 100, 256, 16), (777, 64, 300, 32),
])
def test_dyadic_bit_exact(rbf, n, d, b, k):
    c = workloads.dyadic_grid(n, d, seed=n + d)
    qs = workloads.dyadic_grid(b, d, seed=n + d + 1)
    with engine(rbf, n, d, b, 32) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(b):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], k))


@pytest.mark.parametrize("d", [768, 384, 1024])
def test_unit_gaussian_both_references(rbf, d):
    n, b, k = 20_011, 256, 32
    c = workloads.unit_corpus(n, d, seed=1)
    qs = workloads.unit_queries(b, d, seed=2)
    c16 = oracle.round_bf16(c)
    q16 = oracle.round_bf16(qs)
    with engine(rbf, n, d, b) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(0, b, 17):
            sig16 = oracle.scores(c16, q16[j])
            check_float_topk(idx[j], sc[j], sig16, k, tol_abs=BF16_ACC_ABS)
            sig = oracle.scores(c, qs[j])
            check_float_topk(idx[j], sc[j], sig, k, tol_abs=BF16_ABS)


def test_duplicates_and_ties(rbf):
    rng = np.random.default_rng(5)
    base = workloads.dyadic_grid(40, 128, seed=6)
    c = base[rng.integers(0, 40, size=5000)]
    qs = workloads.dyadic_grid(64, 128, seed=7)
    with engine(rbf, 5000, 128, 64) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, 32)
        for j in range(64):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], 32))


def test_dev_matches_host_and_repeats(rbf):
    import torch
    n, d, b = 30_000, 768, 200
    c = workloads.unit_corpus(n, d, seed=11)
    qs = workloads.unit_queries(b, d, seed=12)
    with engine(rbf, n, d, b) as e:
        e.upload_corpus_rowmajor(c)
        h_idx, h_sc = e.search_resident_batch(qs, 32)
        dq = torch.from_numpy(qs).cuda()
        d_idx = torch.empty((b, 32), dtype=torch.int32, device="cuda")
        d_sc = torch.empty((b, 32), dtype=torch.float32, device="cuda")
        for _ in range(3):
            e.search_resident_batch_dev(dq, 32, d_idx, d_sc)
            torch.cuda.synchronize()
            assert np.array_equal(d_idx.cpu().numpy(), h_idx)
            assert np.array_equal(d_sc.cpu().numpy(), h_sc)
        assert e.check_device_error() == rbf.RBF_OK


@pytest.mark.parametrize("flags", ["bf16", "tf32", "cosine"])
def test_host_read_in_place_matches_staging(rbf, flags):
    """search_resident_batch reads the caller's query buffer in place where the
    device reads pageable host memory through the host's page tables
    (RBF_OPT_HOST_READ = 1, the default there) and through the pinned staging
    block otherwise (0): the results are identical, and exact on dyadic data.
    The queries are a strided view copied to a fresh buffer by the binding,
    and a plain numpy array, so both fresh and long-lived pages are read."""
    n, d, b, k = 20_011, 96, 37, 16
    c = workloads.dyadic_grid(n, d, seed=13)
    qs = workloads.dyadic_grid(2 * b, d, seed=14)[::2]
    f = {"bf16": rbf.RBF_FLAG_BF16_CORPUS, "tf32": 0, "cosine": rbf.RBF_FLAG_BF16_CORPUS | rbf.RBF_FLAG_COSINE}[flags]
    with rbf.Engine(n, d, k, max_batch=b, flags=f) as e:
        e.upload_corpus_rowmajor(c)
        with pytest.raises(rbf.RbfError) as ei:
            e.set_option(rbf.RBF_OPT_HOST_READ, 2)
        assert ei.value.status == rbf.RBF_ERR_INVALID_VALUE
        e.set_option(rbf.RBF_OPT_HOST_READ, 0)
        ref_idx, ref_sc = e.search_resident_batch(qs, k)
        try:
            e.set_option(rbf.RBF_OPT_HOST_READ, 1)
        except rbf.RbfError as err:
            assert err.status == rbf.RBF_ERR_UNSUPPORTED
            pytest.skip("the device does not read pageable host memory")
        for q in (qs, np.ascontiguousarray(qs)):
            idx, sc = e.search_resident_batch(q, k)
            assert np.array_equal(idx, ref_idx) and np.array_equal(sc, ref_sc)
        if flags == "bf16":
            for j in range(0, b, 6):
                check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], k))


def test_unaligned_query_buffers(rbf):
    """Query buffers that start 4 bytes past a 16-byte boundary (host and
    device) take the element-wise conversion path; the results equal those of
    aligned buffers, and D not a multiple of 4 leaves a partial group per row."""
    import torch
    for d in (96, 98):
        n, b, k = 9_001, 19, 8
        c = workloads.dyadic_grid(n, d, seed=15)
        qs = workloads.dyadic_grid(b, d, seed=16)
        raw = np.zeros(b * d + 8, dtype=np.float32)
        base = (-raw.ctypes.data // 4) % 4  # first 16-byte aligned element
        off = np.ndarray((b, d), dtype=np.float32, buffer=raw, offset=4 * (base + 1))
        off[...] = qs
        assert off.ctypes.data % 16 == 4
        with engine(rbf, n, d, b, k) as e:
            e.upload_corpus_rowmajor(c)
            ref_idx, ref_sc = e.search_resident_batch(np.ascontiguousarray(qs), k)
            idx, sc = e.search_resident_batch(off, k)
            assert np.array_equal(idx, ref_idx) and np.array_equal(sc, ref_sc)
            flat = torch.zeros(b * d + 1, dtype=torch.float32, device="cuda")
            dq = flat[1:].view(b, d)
            dq.copy_(torch.from_numpy(qs))
            di = torch.empty((b, k), dtype=torch.int32, device="cuda")
            ds = torch.empty((b, k), dtype=torch.float32, device="cuda")
            e.search_resident_batch_dev(dq, k, di, ds)
            torch.cuda.synchronize()
            assert np.array_equal(di.cpu().numpy(), ref_idx) and np.array_equal(ds.cpu().numpy(), ref_sc)
            for j in range(0, b, 6):
                check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], k))


def test_invalid_and_k_above_32(rbf):
    c = workloads.dyadic_grid(500, 64, seed=21)
    qs = workloads.dyadic_grid(4, 64, seed=22)
    with engine(rbf, 500, 64, 4, k=64) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, 33)       # lists in global memory from K = 33 on
        for j in range(4):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], 33))
        with pytest.raises(rbf.RbfError) as ei:
            e.search_resident_batch(qs, 65)
        assert ei.value.status == rbf.RBF_ERR_INVALID_VALUE
        with pytest.raises(rbf.RbfError) as ei:
            e.search_resident_batch(np.concatenate([qs, qs]), 8)
        assert ei.value.status == rbf.RBF_ERR_INVALID_VALUE
        idx, sc = e.search_resident_batch(qs, 8)
        for j in range(4):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], 8))


def test_full_size_planted(rbf):
    """B = 256 queries x N = 1,000,000 x D = 768, K = 32, with 10 planted
    near-duplicates per query: planted rows lead for every query, and 16
    queries spread over the batch (both CTAs of a pair, every 32-query
    epilogue warp) match both oracle references."""
    n, d, b, k = 1_000_000, 768, 256, 32
    c = workloads.unit_corpus(n, d, seed=1)
    qs = workloads.unit_queries(b, d, seed=2)
    planted = workloads.plant_near_duplicates(c, qs, per_query=10, noise=0.05, seed=3)
    with engine(rbf, n, d, b) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(b):
            assert set(idx[j][:10].tolist()) == set(planted[j].tolist()), j
            check_sorted_distinct(idx[j].astype(np.int64), sc[j].astype(np.float64), n)
        c16 = oracle.round_bf16(c)
        for j in range(0, b, 17):
            q16 = oracle.round_bf16(qs[j])
            check_float_topk(idx[j], sc[j], oracle.scores(c16, q16), k, tol_abs=BF16_ACC_ABS)
            check_float_topk(idx[j], sc[j], oracle.scores(c, qs[j]), k, tol_abs=BF16_ABS)


# N >= 65,536 rows: the batched path first takes, for each query, the K-th
# largest of its 32-row chunk maxima over the first 16,384 rows (K <= 32) and
# drops every key below it in the main pass.

@pytest.mark.parametrize("k", [1, 8, 32])
def test_sample_bound_dyadic_exact(rbf, k):
    n, d, b = 70_001, 64, 40
    c = workloads.dyadic_grid(n, d, seed=31)
    qs = workloads.dyadic_grid(b, d, seed=32)
    with engine(rbf, n, d, b) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, k)
        for j in range(b):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], k))


def test_sample_bound_best_rows_outside_sample(rbf):
    """Row i is (alpha_i, 0, ..., 0) with alpha_i = floor(255 i / n), exact in
    bf16: the sample (the first rows) holds only small alphas, so for a query
    along +e0 the bound is weak and almost every row passes it, and the answer
    (the first 32 rows with alpha = 254) lies outside the sample."""
    n, d = 80_000, 64
    c = np.zeros((n, d), dtype=np.float32)
    c[:, 0] = np.floor(np.arange(n) * 255.0 / n)
    e0 = np.zeros(d, dtype=np.float32)
    e0[0] = 1.0
    qs = np.stack([e0, -e0, workloads.dyadic_grid(1, d, seed=42)[0]])
    with engine(rbf, n, d, 3) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, 32)
        for j in range(3):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], 32))
        first = int(np.argmax(c[:, 0] == 254.0))
        assert idx[0].tolist() == list(range(first, first + 32))


def test_sample_bound_all_equal_rows(rbf):
    """Every row ties: the K-th key of the sample is row K-1 itself, and the
    answer is rows 0..K-1, all inside the sample."""
    n, d = 70_000, 64
    c = np.full((n, d), 0.25, dtype=np.float32)
    qs = np.ones((2, d), dtype=np.float32)
    with engine(rbf, n, d, 2) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, 32)
        assert idx[0].tolist() == list(range(32)) and idx[1].tolist() == list(range(32))
        assert np.all(sc == 16.0)
