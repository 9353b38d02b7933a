"""Single-query resident search through the C ABI against the oracle."""
import json
import os

import numpy as np
import pytest

import oracle
import workloads
from tests.parity import check_exact, check_float_topk, check_sorted_distinct

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def rbf():
    import resident_brute_force_gb300 as rbf
    rbf.load_library()
    return rbf


def make_engine(rbf, max_n, max_d, max_k=256, **kw):
    return rbf.Engine(max_n, max_d, max_k, **kw)


def test_golden_tiny(rbf):
    with open(os.path.join(GOLDEN, "tiny_ip.json")) as f:
        g = json.load(f)
    c = np.array(g["corpus"], dtype=np.float32)
    with make_engine(rbf, 8, 4) as e:
        e.upload_corpus_rowmajor(c)
        for case in g["cases"]:
            idx, sc = e.search_resident(np.array(case["query"], np.float32), case["k"])
            assert idx.tolist() == case["idx"]
            assert sc.tolist() == case["score"]


# Widths: the register-query specialisations (384, 768, 1024) and the
# generic path (1, 3, 100, 130, 2000), each over several tiles with a tail.
@pytest.mark.parametrize("d", [384, 768, 1024, 1, 3, 100, 130, 2000])
def test_dyadic_bit_exact(rbf, d):
    n = 4099 if d <= 1024 else 1501
    c = workloads.dyadic_grid(n, d, seed=200 + d)
    q = workloads.dyadic_grid(1, d, seed=300 + d)[0]
    with make_engine(rbf, n, d) as e:
        e.upload_corpus_rowmajor(c)
        for k in (1, 8, 9, 32, 33, 100, 128, 200, 256):
            if k > n:
                continue
            idx, sc = e.search_resident(q, k)
            o_idx, o_sc = oracle.topk(c, q, k)
            check_exact(idx, sc, o_idx, o_sc)


@pytest.mark.parametrize("d", [384, 768, 1024])
def test_unit_gaussian_tolerance(rbf, d):
    n = 20011
    c = workloads.unit_corpus(n, d, seed=1)
    qs = workloads.unit_queries(3, d, seed=2)
    with make_engine(rbf, n, d) as e:
        e.upload_corpus_rowmajor(c)
        for q in qs:
            sigma = oracle.scores(c, q)
            for k in (8, 32, 100):
                idx, sc = e.search_resident(q, k)
                check_float_topk(idx, sc, sigma, k)


def test_duplicate_rows_tie_by_index(rbf):
    rng = np.random.default_rng(7)
    base = workloads.dyadic_grid(50, 256, seed=8)
    c = base[rng.integers(0, 50, size=6000)]
    q = workloads.dyadic_grid(1, 256, seed=9)[0]
    with make_engine(rbf, 6000, 256) as e:
        e.upload_corpus_rowmajor(c)
        for k in (1, 17, 64, 256):
            idx, sc = e.search_resident(q, k)
            check_exact(idx, sc, *oracle.topk(c, q, k))


def test_all_equal_rows(rbf):
    c = np.full((3000, 384), 0.5, dtype=np.float32)
    q = np.ones(384, dtype=np.float32)
    with make_engine(rbf, 3000, 384) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident(q, 100)
        assert idx.tolist() == list(range(100))
        assert np.all(sc == 192.0)


def test_small_n_and_k_equals_n(rbf):
    for n, d in [(1, 384), (2, 7), (31, 1024), (257, 33)]:
        c = workloads.dyadic_grid(n, d, seed=n)
        q = workloads.dyadic_grid(1, d, seed=n + 1)[0]
        with make_engine(rbf, n, d) as e:
            e.upload_corpus_rowmajor(c)
            k = min(n, 256)
            check_exact(*e.search_resident(q, k), *oracle.topk(c, q, k))
            check_exact(*e.search_resident(q, 1), *oracle.topk(c, q, 1))


def test_nan_and_inf_rows(rbf):
    c = workloads.dyadic_grid(500, 128, seed=11)
    c[3, 5] = np.nan
    c[10, 0] = np.inf
    c[11, 0] = -np.inf
    q = np.abs(workloads.dyadic_grid(1, 128, seed=12)[0]) + 0.5
    with make_engine(rbf, 500, 128) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident(q, 256)
        o_idx, o_sc = oracle.topk(c, q, 256)
        check_exact(idx, sc, o_idx, o_sc)
        assert idx[0] == 10 and sc[0] == np.inf


def test_device_entry_points_match_host(rbf):
    import torch
    n, d = 10007, 768
    c = workloads.unit_corpus(n, d, seed=21)
    q = workloads.unit_queries(1, d, seed=22)[0]
    with make_engine(rbf, n, d) as e:
        e.upload_corpus_rowmajor(torch.from_numpy(c).cuda())   # device-pointer upload
        h_idx, h_sc = e.search_resident(q, 32)
        dq = torch.from_numpy(q).cuda()
        d_idx = torch.empty(32, dtype=torch.int32, device="cuda")
        d_sc = torch.empty(32, dtype=torch.float32, device="cuda")
        e.search_resident_dev(dq, 32, d_idx, d_sc)
        torch.cuda.synchronize()
        assert np.array_equal(d_idx.cpu().numpy(), h_idx)
        assert np.array_equal(d_sc.cpu().numpy(), h_sc)
        d_idx.zero_()
        e.score_select_partials_dev(dq, 32)
        e.merge_partial_topk_dev(32, d_idx, d_sc)
        torch.cuda.synchronize()
        assert np.array_equal(d_idx.cpu().numpy(), h_idx)
        assert e.check_device_error() == rbf.RBF_OK
        # an unaligned device query (4-byte offset) is accepted
        buf = torch.zeros(d + 1, dtype=torch.float32, device="cuda")
        buf[1:] = dq
        e.search_resident_dev(buf[1:], 32, d_idx, d_sc)
        torch.cuda.synchronize()
        assert np.array_equal(d_idx.cpu().numpy(), h_idx)


@pytest.mark.parametrize("opts", [
    {"RBF_OPT_SCHEDULE": 1},
    {"RBF_OPT_CTAS_PER_SM": 2},
    {"RBF_OPT_STAGE_BYTES": 8192},
    {"RBF_OPT_STAGE_BYTES": 65536, "RBF_OPT_SCHEDULE": 1},
    {"RBF_OPT_CTAS_PER_SM": 3, "RBF_OPT_SCHEDULE": 1},
    {"RBF_OPT_CTAS_PER_SM": 4},      # more than 512 lists: the merge takes its general path
])
def test_launch_shapes_same_result(rbf, opts):
    n, d = 30001, 1024
    c = workloads.dyadic_grid(n, d, seed=31)
    q = workloads.dyadic_grid(1, d, seed=32)[0]
    with make_engine(rbf, n, d) as e:
        e.upload_corpus_rowmajor(c)
        ref = e.search_resident(q, 100)
        for name, val in opts.items():
            e.set_option(getattr(rbf, name), val)
        for _ in range(3):   # repeated calls re-arm the tile counter
            check_exact(*e.search_resident(q, 100), *ref)
        check_exact(*ref, *oracle.topk(c, q, 100))


def test_deterministic_repeats(rbf):
    n, d = 50000, 384
    c = workloads.unit_corpus(n, d, seed=41)
    c[1000:1010] = c[77]     # exact duplicates of one row
    q = c[77].copy()
    with make_engine(rbf, n, d) as e:
        e.upload_corpus_rowmajor(c)
        e.set_option(rbf.RBF_OPT_SCHEDULE, 1)
        first = e.search_resident(q, 32)
        for _ in range(30):
            check_exact(*e.search_resident(q, 32), *first)
        # the duplicates share one bit-identical score and come in index order
        assert first[0][:11].tolist() == [77] + list(range(1000, 1010))
        assert len(set(first[1][:11].tolist())) == 1


def test_argument_errors(rbf):
    c = workloads.dyadic_grid(100, 16, seed=51)
    q = c[0]
    with make_engine(rbf, 100, 16, max_k=64) as e:
        with pytest.raises(rbf.RbfError) as ei:
            e.search_resident(q, 8)
        assert ei.value.status == rbf.RBF_ERR_NOT_READY
        with pytest.raises(rbf.RbfError) as ei:
            e.upload_corpus_rowmajor(np.zeros((101, 16), np.float32))
        assert ei.value.status == rbf.RBF_ERR_INVALID_VALUE
        with pytest.raises(rbf.RbfError):
            e.upload_corpus_rowmajor(np.zeros((10, 17), np.float32))
        with pytest.raises(rbf.RbfError) as ei:
            e.upload_corpus_rowmajor(np.zeros((0, 16), np.float32))   # empty corpus
        assert ei.value.status == rbf.RBF_ERR_INVALID_VALUE
        e.upload_corpus_rowmajor(c[:50])
        with pytest.raises(rbf.RbfError) as ei:
            e.search_resident_batch(np.zeros((0, 16), np.float32), 4)  # empty batch
        assert ei.value.status == rbf.RBF_ERR_INVALID_VALUE
        for k in (0, -1, 65, 51):
            with pytest.raises(rbf.RbfError) as ei:
                e.search_resident(q, k)
            assert ei.value.status == rbf.RBF_ERR_INVALID_VALUE
        with pytest.raises(rbf.RbfError) as ei:
            e.search_resident_batch(np.stack([q, q]), 4)
        assert ei.value.status == rbf.RBF_ERR_INVALID_VALUE   # b > max_batch
        check_exact(*e.search_resident(q, 50), *oracle.topk(c[:50], q, 50))
    with pytest.raises(rbf.RbfError):
        rbf.Engine(0, 16)
    with pytest.raises(rbf.RbfError):
        rbf.Engine(10, 16, max_k=257)


def test_binding_refuses_short_buffers(rbf):
    """The C entry points read and write exactly the sizes they are given; the
    binding refuses a query of the wrong length or an output that is too short
    before any pointer reaches the library, and the engine stays usable."""
    import torch
    n, d, k = 2000, 64, 16
    c = workloads.dyadic_grid(n, d, seed=52)
    with make_engine(rbf, n, d, max_k=64, max_batch=4) as e:
        e.upload_corpus_rowmajor(c)
        assert (e.n, e.d) == (n, d)
        dq = torch.from_numpy(c[3]).cuda()
        di = torch.empty(k, dtype=torch.int32, device="cuda")
        ds = torch.empty(k, dtype=torch.float32, device="cuda")
        bad = [
            lambda: e.search_resident(c[3][:d - 1], k),
            lambda: e.search_resident_dev(dq[:d - 1], k, di, ds),
            lambda: e.search_resident_dev(dq, k, di[:k - 1], ds),
            lambda: e.search_resident_dev(dq, k, di, ds[:k - 1]),
            lambda: e.score_select_partials_dev(dq[:d - 1], k),
            lambda: e.merge_partial_topk_dev(k, di[:k - 1], ds),
            lambda: e.search_resident_batch(c[:2, :d - 1], k),
            lambda: e.search_resident_batch(c[3], k),
            lambda: e.search_resident_batch_dev(torch.from_numpy(c[:2]).cuda(), k, di, ds),
            lambda: e.topk_int32_dev(di, k, di[:k - 1], torch.empty(k, dtype=torch.int64, device="cuda")),
            lambda: rbf.topk_int32_noalloc(di, k, di, torch.empty(k - 1, dtype=torch.int64, device="cuda")),
            lambda: e.upload_corpus_rowmajor(c[0]),
        ]
        for j, call in enumerate(bad):
            with pytest.raises(ValueError):
                call()
        torch.cuda.synchronize()
        check_exact(*e.search_resident(c[3], k), *oracle.topk(c, c[3], k))
        assert e.check_device_error() == rbf.RBF_OK


def test_bounded_wait_timeout_reports_and_context_survives(rbf):
    c = workloads.dyadic_grid(1000, 64, seed=61)
    with make_engine(rbf, 1000, 64) as e:
        assert e.selftest_wait_timeout(2_000_000) == rbf.RBF_ERR_TIMEOUT
        e.upload_corpus_rowmajor(c)
        check_exact(*e.search_resident(c[5], 8), *oracle.topk(c, c[5], 8))


def test_host_fault_injection_leaves_outputs_untouched(rbf):
    c = workloads.dyadic_grid(1000, 64, seed=71)
    q = c[3]
    with make_engine(rbf, 1000, 64) as e:
        e.upload_corpus_rowmajor(c)
        lib = e.lib
        idx = np.full(8, -7, np.int32)
        sc = np.full(8, -7.0, np.float32)
        for kind in (rbf.FAULT_COPY, rbf.FAULT_LAUNCH):
            e.inject_host_fault(kind, 1)
            st = lib.search_resident(e._h, q.ctypes.data, 8, idx.ctypes.data, sc.ctypes.data)
            assert st == rbf.RBF_ERR_CUDA
            assert np.all(idx == -7) and np.all(sc == -7.0)
        check_exact(*e.search_resident(q, 8), *oracle.topk(c, q, 8))


def test_sweep_cells_sampled(rbf):
    """The pages' sweep N x D x K on unit Gaussian data: one query per cell,
    fewer rows than the full sweep for the larger N (the full sizes are the
    configuration test below and the bench)."""
    for d in (384, 768, 1024):
        full = workloads.unit_corpus(100_000, d, seed=1)
        q = workloads.unit_queries(1, d, seed=2)[0]
        with make_engine(rbf, 100_000, d) as e:
            for n in (10_000, 50_000, 100_000):
                c = full[:n]
                e.upload_corpus_rowmajor(c)
                sigma = oracle.scores(c, q)
                for k in (8, 32, 100):
                    idx, sc = e.search_resident(q, k)
                    check_float_topk(idx, sc, sigma, k)


@pytest.mark.parametrize("d", [384, 768, 1024])
def test_sweep_cells_full_size(rbf, d):
    """The sweep's two largest row counts (500k and 1M) at every D of the
    sweep, in the launch shape the bench uses: one sampled query per cell
    against the oracle at K = 8, 32 and 100 (1M x 1024 is also the planted
    configuration below)."""
    n_max = 1_000_000
    full = workloads.unit_corpus(n_max, d, seed=1)
    qs = workloads.unit_queries(2, d, seed=2)
    with make_engine(rbf, n_max, d) as e:
        for n, q in ((500_000, qs[0]), (1_000_000, qs[1])):
            c = full[:n]
            e.upload_corpus_rowmajor(c)
            sigma = oracle.scores(c, q)
            for k in (8, 32, 100):
                idx, sc = e.search_resident(q, k)
                check_float_topk(idx, sc, sigma, k)


def test_full_size_planted(rbf):
    """1,000,000 x 1024 fp32 unit-norm corpus with 10 planted near-duplicates
    per query: full oracle comparison on a sample of queries and the planted
    rows checked on many, in the launch shape the bench uses."""
    n, d, nq = 1_000_000, 1024, 1000
    c = workloads.unit_corpus(n, d, seed=1)
    qs = workloads.unit_queries(nq, d, seed=2)
    planted = workloads.plant_near_duplicates(c, qs, per_query=10, noise=0.05, seed=3)
    import torch
    with make_engine(rbf, n, d) as e:
        e.upload_corpus_rowmajor(c)
        for j in range(0, nq, 25):
            idx, sc = e.search_resident(qs[j], 32)
            assert set(idx[:10].tolist()) == set(planted[j].tolist())
            check_sorted_distinct(idx, sc, n)
        for j in (0, 499, 999):
            sigma = oracle.scores(c, qs[j])
            for k in (8, 32, 100):
                idx, sc = e.search_resident(qs[j], k)
                check_float_topk(idx, sc, sigma, k)
        del torch


def test_out_of_memory_paths(rbf, monkeypatch):
    """rbf_create reports RBF_ERR_OUT_OF_MEMORY and leaks nothing: for a real
    over-size request (64 TB of corpus) and for an injected allocation
    failure (RBF_FAULT=alloc), for engines and views; afterwards engines work."""
    with pytest.raises(rbf.RbfError) as ei:
        rbf.Engine(2**31 - 1, 8192, 8)
    assert ei.value.status == rbf.RBF_ERR_OUT_OF_MEMORY
    c = workloads.dyadic_grid(500, 32, seed=73)
    base = rbf.Engine(500, 32, 8)
    try:
        base.upload_corpus_rowmajor(c)
        monkeypatch.setenv("RBF_FAULT", "alloc")
        for make in (lambda: rbf.Engine(500, 32, 8), lambda: base.view()):
            with pytest.raises(rbf.RbfError) as ei:
                make()
            assert ei.value.status == rbf.RBF_ERR_OUT_OF_MEMORY
        monkeypatch.delenv("RBF_FAULT")
        with base.view() as v:
            check_exact(*v.search_resident(c[7], 8), *oracle.topk(c, c[7], 8))
    finally:
        base.close()


def test_repeated_calls_are_bit_identical(rbf):
    """The same query 100 times (single query, batched and int32): every result
    is the same bytes, so no ordering inside a kernel leaks into the output."""
    import torch
    n, d = 30_000, 256
    c = workloads.unit_corpus(n, d, seed=74)
    qs = workloads.unit_queries(16, d, seed=75)
    x = torch.from_numpy(workloads.int32_uniform(1_000_000, seed=76)).cuda()
    with rbf.Engine(n, d, 100, max_batch=16, flags=rbf.RBF_FLAG_BF16_CORPUS) as e:
        e.upload_corpus_rowmajor(c)
        first = e.search_resident(qs[0], 100)
        first_b = e.search_resident_batch(qs, 100)
        first_i = e.topk_int32(x, 64)
        for _ in range(100):
            idx, sc = e.search_resident(qs[0], 100)
            assert np.array_equal(idx, first[0]) and np.array_equal(sc, first[1])
        for _ in range(100):
            idx, sc = e.search_resident_batch(qs, 100)
            assert np.array_equal(idx, first_b[0]) and np.array_equal(sc, first_b[1])
            v, p = e.topk_int32(x, 64)
            assert np.array_equal(v, first_i[0]) and np.array_equal(p, first_i[1])
        check_float_topk(first[0], first[1], oracle.scores(c, qs[0]), 100)
