"""ctypes binding of librbf.so (include/rbf.h), argument marshalling only.

Every step of the search runs in the library's CUDA kernels. This module only
turns numpy arrays / torch tensors into pointers and sizes, calls the C entry
point of the same name, and raises ``RbfError`` on a non-zero status. If the
library is missing it raises at once: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import _build

RBF_OK = 0
RBF_ERR_INVALID_VALUE = 1
RBF_ERR_NOT_READY = 2
RBF_ERR_OUT_OF_MEMORY = 3
RBF_ERR_CUDA = 4
RBF_ERR_TIMEOUT = 5
RBF_ERR_UNSUPPORTED = 6
RBF_ERR_BOUNDS = 7

RBF_MAX_K = 256
RBF_MAX_D = 8192
RBF_FLAG_FP32_CORPUS = 0x1
RBF_FLAG_BF16_CORPUS = 0x2
RBF_FLAG_COSINE = 0x4

RBF_OPT_CTAS_PER_SM = 1
RBF_OPT_STAGE_BYTES = 2
RBF_OPT_SMEM_BUDGET = 3
RBF_OPT_TIMEOUT_NS = 4
RBF_OPT_SCHEDULE = 5
RBF_OPT_BATCH_SAMPLE = 6
RBF_OPT_HOST_READ = 7

FAULT_COPY = 1
FAULT_LAUNCH = 2

# Every symbol the header declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_U32 = ctypes.c_uint32
_U64 = ctypes.c_uint64
_S = ctypes.c_int
SIGNATURES = {
    "rbf_create": (_S, [_I64, _I32, _I32, _I32, _U32, _P, ctypes.POINTER(_P)]),
    "rbf_create_view": (_S, [_P, _P, ctypes.POINTER(_P)]),
    "rbf_destroy": (_S, [_P]),
    "rbf_stream": (_P, [_P]),
    "rbf_num_sms": (_I32, [_P]),
    "rbf_num_partials": (_I32, [_P]),
    "rbf_set_option": (_S, [_P, _S, _I64]),
    "rbf_status_string": (ctypes.c_char_p, [_S]),
    "rbf_last_cuda_error": (_I32, [_P]),
    "rbf_last_launches": (_I32, [_P]),
    "rbf_check_device_error": (_S, [_P]),
    "upload_corpus_rowmajor": (_S, [_P, _P, _I64, _I32]),
    "upload_corpus_shard": (_S, [_P, _P, _I64, _I32, _I64]),
    "merge_shard_topk_dev": (_S, [_P, _P, _P, _I32, _I32, _I32, _P, _P]),
    "search_resident": (_S, [_P, _P, _I32, _P, _P]),
    "search_resident_dev": (_S, [_P, _P, _I32, _P, _P]),
    "score_select_partials_dev": (_S, [_P, _P, _I32]),
    "merge_partial_topk_dev": (_S, [_P, _I32, _P, _P]),
    "search_resident_batch": (_S, [_P, _P, _I32, _I32, _P, _P]),
    "search_resident_batch_dev": (_S, [_P, _P, _I32, _I32, _P, _P]),
    "topk_int32": (_S, [_P, _P, _I64, _I32, _P, _P]),
    "topk_int32_dev": (_S, [_P, _P, _I64, _I32, _P, _P]),
    "topk_int32_noalloc": (_S, [_P, _I64, _I32, _P, _P, _P]),
    "rbf_selftest_wait_timeout": (_S, [_P, _U64]),
    "rbf_inject_host_fault": (_S, [_P, _I32, _I32]),
}

_lib = None


def lib_path() -> str:
    """The library to load: RBF_LIB if set (e.g. the checked build), else the
    in-tree librbf.so."""
    return os.environ.get("RBF_LIB") or _build.LIB_PATH


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load librbf.so. Raises if it has not been built."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        p = lib_path()
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with __graft_entry__.build() (nvcc, sm_103a)")
        _lib = _declare(ctypes.CDLL(p))
    return _lib


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


def topk_int32_noalloc(d_data, k: int, d_val, d_pos, stream=None) -> int:
    """Call topk_int32_noalloc (no engine, no device allocation); returns the
    status code. All tensors are CUDA tensors on the current device."""
    _need(d_val.numel() >= max(int(k), 0) and d_pos.numel() >= max(int(k), 0),
          f"d_val / d_pos hold {d_val.numel()} / {d_pos.numel()} entries, the call writes {k}")
    s = None
    if stream is not None:
        s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return load_library().topk_int32_noalloc(_dev_ptr(d_data, "int32"), int(d_data.numel()), int(k),
                                             _dev_ptr(d_val, "int32"), _dev_ptr(d_pos, "int64"),
                                             ctypes.c_void_p(s) if s else None)


class RbfError(RuntimeError):
    def __init__(self, status: int, where: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        name = load_library().rbf_status_string(status).decode()
        extra = f" (cudaError {cuda_error})" if status == RBF_ERR_CUDA else ""
        super().__init__(f"{where}: {name}{extra}")


def status_string(status: int) -> str:
    return load_library().rbf_status_string(status).decode()


def _host_ptr(a: np.ndarray, dtype) -> tuple[np.ndarray, int]:
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


_TORCH_DTYPES: dict = {}


def _dev_ptr(t, dtype_name: str) -> int:
    """Device pointer of a contiguous CUDA torch tensor of the given dtype."""
    if not getattr(t, "is_cuda", False):
        raise TypeError("expected a CUDA tensor")
    want = _TORCH_DTYPES.get(dtype_name)
    if want is None:
        import torch
        want = _TORCH_DTYPES.setdefault(dtype_name, getattr(torch, dtype_name))
    if t.dtype != want:
        raise TypeError(f"expected torch.{dtype_name}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


class _HostBuffers:
    """An engine's host arrays for its single-query and int32 host-buffer
    calls, with their addresses taken once: numpy builds a helper object each
    time an array's address is read (~2 us), while copying a query into a
    fixed buffer and the K results out of one costs well under that."""

    def __init__(self):
        self.q = np.empty(RBF_MAX_D, np.float32)
        self.idx = np.empty(RBF_MAX_K, np.int32)
        self.sc = np.empty(RBF_MAX_K, np.float32)
        self.pos = np.empty(RBF_MAX_K, np.int64)
        self.q_p = self.q.ctypes.data
        self.idx_p = self.idx.ctypes.data
        self.sc_p = self.sc.ctypes.data
        self.pos_p = self.pos.ctypes.data


def _need(ok: bool, msg: str) -> None:
    """The library reads and writes exactly the sizes it is given; a buffer
    that is too short is refused here, before any pointer reaches it."""
    if not ok:
        raise ValueError(msg)


def _any_ptr(x, np_dtype, torch_dtype_name: str) -> tuple[object, int]:
    """Pointer to host (numpy / CPU tensor) or device (CUDA tensor) data."""
    if hasattr(x, "data_ptr"):
        if x.is_cuda:
            return x, _dev_ptr(x, torch_dtype_name)
        x = x.numpy()
    return _host_ptr(x, np_dtype)


class Engine:
    """An engine with every buffer preallocated (see ``rbf_create``).

    Like the handle it wraps, one Engine serves one call at a time (its
    host-buffer calls also share small host arrays); concurrent callers each
    take their own ``view()``."""

    def __init__(self, max_n: int, max_d: int, max_k: int = RBF_MAX_K, max_batch: int = 1,
                 flags: int = 0, stream=None, _view_of=None):
        self.lib = load_library()
        handle = ctypes.c_void_p()
        s = None
        if stream is not None:
            s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        if _view_of is not None:
            st = self.lib.rbf_create_view(_view_of._h, ctypes.c_void_p(s) if s else None, ctypes.byref(handle))
            where = "rbf_create_view"
        else:
            st = self.lib.rbf_create(int(max_n), int(max_d), int(max_k), int(max_batch), int(flags),
                                     ctypes.c_void_p(s) if s else None, ctypes.byref(handle))
            where = "rbf_create"
        if st != RBF_OK:
            raise RbfError(st, where)
        self._h = handle
        self._stream_ref = stream
        self._base = _view_of  # a view keeps its base alive
        self._n = None
        self._d = None

    @property
    def n(self):
        """Rows of the resident corpus (None before an upload); a view reports its base's."""
        return self._base.n if self._base is not None else self._n

    @property
    def d(self):
        """Dimension of the resident corpus (None before an upload); a view reports its base's."""
        return self._base.d if self._base is not None else self._d

    def _host_buffers(self) -> _HostBuffers:
        hb = getattr(self, "_hb", None)
        if hb is None:
            hb = self._hb = _HostBuffers()
        return hb

    def _out_len(self, t, count: int, what: str) -> None:
        if t.numel() < count:
            raise ValueError(f"{what} holds {t.numel()} entries, the call writes {count}")

    def _query_len(self, size: int, what: str) -> None:
        d = self.d
        if d is not None and size != d:
            raise ValueError(f"{what} has {size} elements, the corpus has D = {d}")

    def view(self, stream=None) -> "Engine":
        """A second handle on this engine's resident corpus with its own stream
        and per-call buffers (rbf_create_view): calls on different handles may
        run concurrently. Close views before their base."""
        return Engine(0, 0, _view_of=self, stream=stream)

    # -- lifetime
    def close(self) -> None:
        if getattr(self, "_h", None):
            st = self.lib.rbf_destroy(self._h)
            if st != RBF_OK:
                raise RbfError(st, "rbf_destroy (close the views first)")
            self._h = None
            self._base = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def _check(self, st: int, where: str) -> None:
        if st != RBF_OK:
            raise RbfError(st, where, self.lib.rbf_last_cuda_error(self._h))

    # -- info / options
    @property
    def stream_handle(self) -> int:
        return self.lib.rbf_stream(self._h) or 0

    @property
    def num_sms(self) -> int:
        return self.lib.rbf_num_sms(self._h)

    @property
    def num_partials(self) -> int:
        return self.lib.rbf_num_partials(self._h)

    def last_cuda_error(self) -> int:
        return self.lib.rbf_last_cuda_error(self._h)

    @property
    def last_launches(self) -> int:
        """Kernels the most recent search / top-K call enqueued."""
        return self.lib.rbf_last_launches(self._h)

    def set_option(self, option: int, value: int) -> None:
        self._check(self.lib.rbf_set_option(self._h, int(option), int(value)), "rbf_set_option")

    def check_device_error(self) -> int:
        return self.lib.rbf_check_device_error(self._h)

    def selftest_wait_timeout(self, timeout_ns: int) -> int:
        return self.lib.rbf_selftest_wait_timeout(self._h, int(timeout_ns))

    def inject_host_fault(self, kind: int, count: int) -> None:
        self._check(self.lib.rbf_inject_host_fault(self._h, int(kind), int(count)), "rbf_inject_host_fault")

    # -- ingest
    def upload_corpus_rowmajor(self, corpus) -> None:
        _need(len(corpus.shape) == 2, "the corpus is a 2-D [N, D] array")
        keep, ptr = _any_ptr(corpus, np.float32, "float32")
        n, d = corpus.shape
        self._check(self.lib.upload_corpus_rowmajor(self._h, ptr, int(n), int(d)), "upload_corpus_rowmajor")
        self._n, self._d = int(n), int(d)
        del keep

    def upload_corpus_shard(self, corpus, row_offset: int) -> None:
        """Rows [row_offset, row_offset + N) of a larger corpus: results report
        global row indices (upload_corpus_shard)."""
        _need(len(corpus.shape) == 2, "the corpus is a 2-D [N, D] array")
        keep, ptr = _any_ptr(corpus, np.float32, "float32")
        n, d = corpus.shape
        self._check(self.lib.upload_corpus_shard(self._h, ptr, int(n), int(d), int(row_offset)),
                    "upload_corpus_shard")
        self._n, self._d = int(n), int(d)
        del keep

    # -- single query
    def search_resident(self, query, k: int):
        q = np.asarray(query)
        if q.ndim != 1:
            q = q.reshape(-1)
        self._query_len(q.shape[0], "the query")
        if q.shape[0] > RBF_MAX_D:
            raise ValueError(f"the query has {q.shape[0]} elements, more than RBF_MAX_D")
        hb = self._host_buffers()
        k = int(k)
        hb.q[:q.shape[0]] = q  # the library reads D floats from here (cast to float32)
        self._check(self.lib.search_resident(self._h, hb.q_p, k, hb.idx_p, hb.sc_p), "search_resident")
        return hb.idx[:k].copy(), hb.sc[:k].copy()

    def search_resident_dev(self, d_query, k: int, d_idx, d_score) -> None:
        self._query_len(d_query.numel(), "d_query")
        self._out_len(d_idx, k, "d_idx")
        self._out_len(d_score, k, "d_score")
        self._check(self.lib.search_resident_dev(self._h, _dev_ptr(d_query, "float32"), int(k),
                                                 _dev_ptr(d_idx, "int32"), _dev_ptr(d_score, "float32")),
                    "search_resident_dev")

    def score_select_partials_dev(self, d_query, k: int) -> None:
        self._query_len(d_query.numel(), "d_query")
        self._check(self.lib.score_select_partials_dev(self._h, _dev_ptr(d_query, "float32"), int(k)),
                    "score_select_partials_dev")

    def merge_partial_topk_dev(self, k: int, d_idx, d_score) -> None:
        self._out_len(d_idx, k, "d_idx")
        self._out_len(d_score, k, "d_score")
        self._check(self.lib.merge_partial_topk_dev(self._h, int(k), _dev_ptr(d_idx, "int32"),
                                                    _dev_ptr(d_score, "float32")), "merge_partial_topk_dev")

    # -- batched
    def search_resident_batch(self, queries, k: int):
        q, qp = _host_ptr(np.asarray(queries), np.float32)
        _need(q.ndim == 2, "the queries are a 2-D [B, D] array")
        self._query_len(q.shape[1], "each query")
        b = q.shape[0]
        idx = np.empty((b, max(int(k), 0)), dtype=np.int32)
        sc = np.empty((b, max(int(k), 0)), dtype=np.float32)
        self._check(self.lib.search_resident_batch(self._h, qp, int(b), int(k), idx.ctypes.data,
                                                   sc.ctypes.data), "search_resident_batch")
        return idx, sc

    def search_resident_batch_dev(self, d_queries, k: int, d_idx, d_score) -> None:
        _need(d_queries.dim() == 2, "d_queries is a 2-D [B, D] tensor")
        self._query_len(d_queries.shape[1], "each query of d_queries")
        b = d_queries.shape[0]
        self._out_len(d_idx, b * int(k), "d_idx")
        self._out_len(d_score, b * int(k), "d_score")
        self._check(self.lib.search_resident_batch_dev(self._h, _dev_ptr(d_queries, "float32"), int(b), int(k),
                                                       _dev_ptr(d_idx, "int32"), _dev_ptr(d_score, "float32")),
                    "search_resident_batch_dev")

    # -- row shards
    def merge_shard_topk_dev(self, d_idx, d_score, k: int, d_out_idx, d_out_score) -> None:
        """Merge g shards' best-first lists, d_idx / d_score of shape [g, b, k]
        (or [g, k] for one query), into [b, k] (merge_shard_topk_dev)."""
        _need(d_idx.dim() in (2, 3) and tuple(d_idx.shape) == tuple(d_score.shape),
              "d_idx and d_score are [g, k] or [g, b, k] tensors of one shape")
        g = d_idx.shape[0]
        b = d_idx.shape[1] if d_idx.dim() == 3 else 1
        _need(d_idx.shape[-1] == int(k), f"the lists hold {d_idx.shape[-1]} entries, k = {k}")
        self._out_len(d_out_idx, b * int(k), "d_out_idx")
        self._out_len(d_out_score, b * int(k), "d_out_score")
        self._check(self.lib.merge_shard_topk_dev(self._h, _dev_ptr(d_idx, "int32"), _dev_ptr(d_score, "float32"),
                                                  int(g), int(b), int(k), _dev_ptr(d_out_idx, "int32"),
                                                  _dev_ptr(d_out_score, "float32")), "merge_shard_topk_dev")

    # -- flat int32
    def topk_int32(self, d_data, k: int):
        hb = self._host_buffers()
        k = int(k)
        self._check(self.lib.topk_int32(self._h, _dev_ptr(d_data, "int32"), int(d_data.numel()), k, hb.idx_p,
                                        hb.pos_p), "topk_int32")
        return hb.idx[:k].copy(), hb.pos[:k].copy()

    def topk_int32_dev(self, d_data, k: int, d_val, d_pos) -> None:
        self._out_len(d_val, k, "d_val")
        self._out_len(d_pos, k, "d_pos")
        self._check(self.lib.topk_int32_dev(self._h, _dev_ptr(d_data, "int32"), int(d_data.numel()), int(k),
                                            _dev_ptr(d_val, "int32"), _dev_ptr(d_pos, "int64")), "topk_int32_dev")
