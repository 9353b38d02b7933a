"""Views (rbf_create_view): several handles on one resident corpus, each with
its own stream and per-call buffers, so that queries run concurrently, on
different streams and from different host threads. Every result must equal
the one the base engine gives alone, bit for bit, and the oracle's."""
import threading

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


def test_views_share_the_corpus(rbf):
    n, d, k = 20_000, 96, 16
    c = workloads.dyadic_grid(n, d, seed=81)
    qs = workloads.dyadic_grid(8, d, seed=82)
    base = rbf.Engine(n, d, 64, max_batch=8, flags=rbf.RBF_FLAG_BF16_CORPUS)
    base.upload_corpus_rowmajor(c)
    views = [base.view() for _ in range(3)]
    try:
        for v in views:
            assert v.num_partials == base.num_partials
            for j in range(0, 8, 3):
                check_exact(*v.search_resident(qs[j], k), *oracle.topk(c, qs[j], k))
            idx, sc = v.search_resident_batch(qs, 40)
            for j in range(8):
                check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], 40))
    finally:
        for v in views:
            v.close()
        base.close()


def test_concurrent_streams_device_calls(rbf):
    """Four handles issue single-query searches on four streams without any
    synchronisation between them; every result equals the sequential one."""
    import torch
    n, d, k, nq = 50_000, 384, 8, 64
    c = workloads.unit_corpus(n, d, seed=83)
    qs = workloads.unit_queries(nq, d, seed=84)
    streams = [torch.cuda.Stream() for _ in range(4)]
    base = rbf.Engine(n, d, k, stream=streams[0])
    base.upload_corpus_rowmajor(c)
    handles = [base] + [base.view(stream=s) for s in streams[1:]]
    try:
        dq = torch.from_numpy(qs).cuda()
        ref_i = torch.empty((nq, k), dtype=torch.int32, device="cuda")
        ref_s = torch.empty((nq, k), dtype=torch.float32, device="cuda")
        with torch.cuda.stream(streams[0]):
            for j in range(nq):
                base.search_resident_dev(dq[j], k, ref_i[j], ref_s[j])
        torch.cuda.synchronize()
        out_i = torch.zeros((nq, k), dtype=torch.int32, device="cuda")
        out_s = torch.zeros((nq, k), dtype=torch.float32, device="cuda")
        for rep in range(3):
            out_i.zero_()
            out_s.zero_()
            torch.cuda.synchronize()
            for j in range(nq):
                h = handles[j % 4]
                with torch.cuda.stream(streams[j % 4]):
                    h.search_resident_dev(dq[j], k, out_i[j], out_s[j])
            torch.cuda.synchronize()
            assert torch.equal(out_i, ref_i) and torch.equal(out_s, ref_s), rep
        for j in range(0, nq, 13):
            check_float_topk(ref_i[j].cpu().numpy(), ref_s[j].cpu().numpy(), oracle.scores(c, qs[j]), k)
        for h in handles:
            assert h.check_device_error() == rbf.RBF_OK
    finally:
        for h in handles[1:]:
            h.close()
        base.close()


def test_concurrent_host_threads(rbf):
    """Host-buffer searches (each a captured graph on its handle's stream) from
    four threads at once, 40 queries each."""
    n, d, k = 30_000, 128, 32
    c = workloads.dyadic_grid(n, d, seed=85)
    qs = workloads.dyadic_grid(160, d, seed=86)
    base = rbf.Engine(n, d, k)
    base.upload_corpus_rowmajor(c)
    expect = [base.search_resident(qs[j], k) for j in range(160)]
    views = [base.view() for _ in range(3)]
    handles = [base] + views
    errors = []

    def worker(t):
        try:
            h = handles[t]
            for j in range(t, 160, 4):
                idx, sc = h.search_resident(qs[j], k)
                if not (np.array_equal(idx, expect[j][0]) and np.array_equal(sc, expect[j][1])):
                    errors.append((t, j))
        except Exception as ex:  # pragma: no cover - reported below
            errors.append((t, repr(ex)))

    try:
        threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
        for th in threads:
            th.start()
        for th in threads:
            th.join()
        assert not errors, errors[:5]
        for j in range(0, 160, 31):
            check_exact(*expect[j], *oracle.topk(c, qs[j], k))
    finally:
        for v in views:
            v.close()
        base.close()


def test_upload_on_base_reaches_views_and_rules(rbf):
    n, d, k = 4000, 64, 8
    c1 = workloads.dyadic_grid(n, d, seed=87)
    c2 = workloads.dyadic_grid(n // 2, d + 3, seed=88)
    q1 = workloads.dyadic_grid(1, d, seed=89)[0]
    q2 = workloads.dyadic_grid(1, d + 3, seed=90)[0]
    base = rbf.Engine(n, d + 3, k)
    v = base.view()
    try:
        with pytest.raises(rbf.RbfError) as ei:
            v.search_resident(q1, k)                    # nothing uploaded yet
        assert ei.value.status == rbf.RBF_ERR_NOT_READY
        base.upload_corpus_rowmajor(c1)
        check_exact(*v.search_resident(q1, k), *oracle.topk(c1, q1, k))  # captures a graph
        base.upload_corpus_rowmajor(c2)                 # new shape: the view's graph must go
        assert (v.n, v.d) == (n // 2, d + 3)
        check_exact(*v.search_resident(q2, k), *oracle.topk(c2, q2, k))
        with pytest.raises(rbf.RbfError) as ei:
            v.upload_corpus_rowmajor(c1)                # views cannot upload
        assert ei.value.status == rbf.RBF_ERR_INVALID_VALUE
        with pytest.raises(rbf.RbfError):
            base.close()                                # a view is still open
        with pytest.raises(rbf.RbfError) as ei:
            v.view()                                    # no view of a view
        assert ei.value.status == rbf.RBF_ERR_INVALID_VALUE
        v.set_option(rbf.RBF_OPT_CTAS_PER_SM, 2)        # the view's own launch shape
        check_exact(*v.search_resident(q2, k), *oracle.topk(c2, q2, k))
        check_exact(*base.search_resident(q2, k), *oracle.topk(c2, q2, k))
    finally:
        v.close()
        base.close()


def test_concurrent_batched_and_int32_on_views(rbf):
    """Batched searches (K = 32 and K = 100, the latter through per-thread lists in each handle's
    own partials buffer) and int32 top-K calls issued on three handles' streams without
    synchronisation in between: every result equals the one computed alone."""
    import torch
    n, d, b = 70_144, 128, 40
    c = workloads.dyadic_grid(n, d, seed=91)
    qs = workloads.dyadic_grid(3 * b, d, seed=92)
    x = torch.from_numpy(workloads.int32_uniform(2_000_000, seed=93)).cuda()
    streams = [torch.cuda.Stream() for _ in range(3)]
    base = rbf.Engine(n, d, 128, max_batch=b, flags=rbf.RBF_FLAG_BF16_CORPUS, stream=streams[0])
    base.upload_corpus_rowmajor(c)
    hs = [base] + [base.view(stream=s) for s in streams[1:]]
    try:
        dq = torch.from_numpy(qs).cuda()
        jobs = [(32, 0), (100, 1), (32, 2)]
        ref = []
        for k, part in jobs:
            di = torch.empty((b, k), dtype=torch.int32, device="cuda")
            ds = torch.empty((b, k), dtype=torch.float32, device="cuda")
            base.search_resident_batch_dev(dq[part * b:(part + 1) * b], k, di, ds)
            torch.cuda.synchronize()
            ref.append((di.clone(), ds.clone()))
        dv_ref = torch.empty(50, dtype=torch.int32, device="cuda")
        dp_ref = torch.empty(50, dtype=torch.int64, device="cuda")
        base.topk_int32_dev(x, 50, dv_ref, dp_ref)
        torch.cuda.synchronize()
        for rep in range(3):
            outs = []
            for h, s, (k, part) in zip(hs, streams, jobs):
                di = torch.zeros((b, k), dtype=torch.int32, device="cuda")
                ds = torch.zeros((b, k), dtype=torch.float32, device="cuda")
                dv = torch.zeros(50, dtype=torch.int32, device="cuda")
                dp = torch.zeros(50, dtype=torch.int64, device="cuda")
                torch.cuda.synchronize()
                outs.append((di, ds, dv, dp))
            for h, s, (k, part), (di, ds, dv, dp) in zip(hs, streams, jobs, outs):
                with torch.cuda.stream(s):
                    h.search_resident_batch_dev(dq[part * b:(part + 1) * b], k, di, ds)
                    h.topk_int32_dev(x, 50, dv, dp)
            torch.cuda.synchronize()
            for j, (di, ds, dv, dp) in enumerate(outs):
                assert torch.equal(di, ref[j][0]) and torch.equal(ds, ref[j][1]), (rep, j)
                assert torch.equal(dv, dv_ref) and torch.equal(dp, dp_ref), (rep, j)
        for j, (k, part) in enumerate(jobs):
            for q in range(0, b, 13):
                idx = ref[j][0][q].cpu().numpy()
                sc = ref[j][1][q].cpu().numpy()
                check_exact(idx, sc, *oracle.topk(c, qs[part * b + q], k))
        for h in hs:
            assert h.check_device_error() == rbf.RBF_OK
    finally:
        for h in hs[1:]:
            h.close()
        base.close()


def test_upload_waits_for_searches_queued_on_views(rbf):
    """A view queues device searches over a 400 MB corpus (a few ms of work in
    flight) and the base uploads a different corpus right away: every queued
    search must still see the old corpus, and the next one the new."""
    import torch
    n, d, k, nq = 100_000, 1024, 8, 24
    c1 = workloads.unit_corpus(n, d, seed=94)
    c2 = -c1                                            # same shape, every score negated
    qs = workloads.unit_queries(nq, d, seed=95)
    st = torch.cuda.Stream()
    base = rbf.Engine(n, d, k)
    base.upload_corpus_rowmajor(c1)
    v = base.view(stream=st)
    try:
        dq = torch.from_numpy(qs).cuda()
        dc2 = torch.from_numpy(c2).cuda()
        out_i = torch.zeros((nq, k), dtype=torch.int32, device="cuda")
        out_s = torch.zeros((nq, k), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            for j in range(nq):
                v.search_resident_dev(dq[j], k, out_i[j], out_s[j])
        base.upload_corpus_rowmajor(dc2)                # no synchronisation with the view's stream
        torch.cuda.synchronize()
        for j in range(0, nq, 5):
            check_float_topk(out_i[j].cpu().numpy(), out_s[j].cpu().numpy(), oracle.scores(c1, qs[j]), k)
        check_float_topk(*v.search_resident(qs[0], k), oracle.scores(c2, qs[0]), k)
        assert v.check_device_error() == rbf.RBF_OK
    finally:
        v.close()
        base.close()


def test_views_made_and_destroyed_from_threads(rbf):
    """Four host threads each make a view, search with it and destroy it, five
    times over, while the others do the same: every result equals the base's
    and the base can be closed afterwards (no view left behind)."""
    n, d, k = 20_000, 128, 16
    c = workloads.dyadic_grid(n, d, seed=96)
    qs = workloads.dyadic_grid(40, d, seed=97)
    base = rbf.Engine(n, d, k)
    base.upload_corpus_rowmajor(c)
    expect = [base.search_resident(qs[j], k) for j in range(40)]
    errors = []

    def worker(t):
        try:
            for rep in range(5):
                with base.view() as v:
                    for j in range(t, 40, 4):
                        idx, sc = v.search_resident(qs[j], k)
                        if not (np.array_equal(idx, expect[j][0]) and np.array_equal(sc, expect[j][1])):
                            errors.append((t, rep, j))
        except Exception as ex:  # pragma: no cover - reported below
            errors.append((t, repr(ex)))

    try:
        threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
        for th in threads:
            th.start()
        for th in threads:
            th.join()
        assert not errors, errors[:5]
        check_exact(*expect[7], *oracle.topk(c, qs[7], k))
    finally:
        base.close()
