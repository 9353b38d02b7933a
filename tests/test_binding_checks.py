"""The binding's argument checks, on the CPU: a query whose length is not the
resident D, an output shorter than the call writes, or an array of the wrong
rank is refused with ValueError before any pointer reaches the library (so
these run without a GPU: the engine object is never connected to one)."""
import numpy as np
import pytest
import torch

from resident_brute_force_gb300 import _binding as b


class _NoLibrary:
    """Stands in for the loaded library: any call into it fails the test."""

    def __getattr__(self, name):
        def reached(*args):
            raise AssertionError(f"{name} reached the library")
        return reached


def _engine(n=100, d=64, base=None):
    e = object.__new__(b.Engine)   # no rbf_create: nothing below reaches the library
    e.lib = _NoLibrary()
    e._h = None
    e._base = base
    e._n, e._d = (None, None) if base is not None else (n, d)
    return e


def test_views_report_their_base_shape():
    base = _engine(100, 64)
    v = _engine(base=base)
    assert (v.n, v.d) == (100, 64)
    base._n, base._d = 50, 67
    assert (v.n, v.d) == (50, 67)


def test_short_or_misshapen_arguments_are_refused():
    e = _engine(100, 64)
    k = 16
    q = torch.zeros(64)
    i32 = torch.zeros(k, dtype=torch.int32)
    f32 = torch.zeros(k)
    i64 = torch.zeros(k, dtype=torch.int64)
    bad = [
        lambda: e.search_resident(np.zeros(63, np.float32), k),
        lambda: e.search_resident(np.zeros(65, np.float32), k),
        lambda: e.search_resident_dev(q[:63], k, i32, f32),
        lambda: e.search_resident_dev(q, k, i32[:k - 1], f32),
        lambda: e.search_resident_dev(q, k, i32, f32[:k - 1]),
        lambda: e.score_select_partials_dev(q[:63], k),
        lambda: e.merge_partial_topk_dev(k, i32, f32[:k - 1]),
        lambda: e.search_resident_batch(np.zeros((2, 63), np.float32), k),
        lambda: e.search_resident_batch(np.zeros(64, np.float32), k),
        lambda: e.search_resident_batch_dev(torch.zeros(64), k, i32, f32),
        lambda: e.search_resident_batch_dev(torch.zeros(2, 64), k, i32, f32),
        lambda: e.topk_int32_dev(i32, k, i32[:k - 1], i64),
        lambda: e.topk_int32_dev(i32, k, i32, i64[:k - 1]),
        lambda: b.topk_int32_noalloc(i32, k, i32, i64[:k - 1]),
        lambda: e.upload_corpus_rowmajor(np.zeros(64, np.float32)),
    ]
    for j, call in enumerate(bad):
        with pytest.raises(ValueError):
            call()


def test_sizes_that_fit_pass_the_checks():
    """Right sizes get past the checks to the pointer conversion, which wants
    CUDA tensors (so, here, a TypeError and still no library call)."""
    e = _engine(100, 64)
    k = 16
    with pytest.raises(TypeError):
        e.search_resident_dev(torch.zeros(64), k, torch.zeros(k, dtype=torch.int32), torch.zeros(k))
    with pytest.raises(TypeError):
        e.search_resident_batch_dev(torch.zeros(2, 64), k, torch.zeros(2 * k, dtype=torch.int32),
                                    torch.zeros(2 * k))
    unknown = _engine(None, None)  # nothing uploaded: the library reports NOT_READY itself
    unknown._d = None
    with pytest.raises(TypeError):
        unknown.search_resident_dev(torch.zeros(5), k, torch.zeros(k, dtype=torch.int32), torch.zeros(k))
