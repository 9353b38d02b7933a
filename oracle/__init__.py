"""Plain CPU oracle for exact brute-force top-K retrieval.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package. The
product path (``resident_brute_force_gb300``) never imports it, and it never
imports the product path.

The arithmetic lives in ``oracle.c`` (plain C, double accumulation, full
sort under the tie rule); this module only compiles it on demand with gcc and
marshals numpy arrays. Every function states the passage it follows in the C
source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    cmd = ["gcc", *CFLAGS, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _stale() -> bool:
    return (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building if needed) the oracle library. ``path`` loads another
    build of the same source, e.g. a deliberately broken copy in a test."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _stale():
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    i64, i32 = ctypes.c_int64, ctypes.c_int32
    lib.oracle_scores.argtypes = [P, i64, i32, P, P]
    lib.oracle_scores_cosine.argtypes = [P, i64, i32, P, P]
    lib.oracle_topk.argtypes = [P, i64, i32, P, i32, P, P]
    lib.oracle_topk_cosine.argtypes = [P, i64, i32, P, i32, P, P]
    lib.oracle_topk_batch.argtypes = [P, i64, i32, P, i32, i32, P, P]
    lib.oracle_topk_int32.argtypes = [P, i64, i32, P, P]
    lib.oracle_round_bf16.argtypes = [P, P, i64]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    for f in ("oracle_scores", "oracle_scores_cosine", "oracle_topk", "oracle_topk_cosine", "oracle_topk_batch",
              "oracle_topk_int32", "oracle_round_bf16"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


class Oracle:
    """Bound view of one oracle build (the default build, or a test's copy)."""

    def __init__(self, lib: ctypes.CDLL):
        self.lib = lib

    def scores(self, corpus, query) -> np.ndarray:
        """All N double scores of one query (see ``oracle_scores``)."""
        c, q = _f32(corpus), _f32(query).reshape(-1)
        n, d = c.shape
        if q.shape[0] != d:
            raise ValueError("query length != D")
        out = np.empty(n, dtype=np.float64)
        if self.lib.oracle_scores(_ptr(c), n, d, _ptr(q), _ptr(out)):
            raise ValueError("oracle_scores rejected its arguments")
        return out

    def topk(self, corpus, query, k: int):
        """(indices int64[K], scores float64[K]) best-first (``oracle_topk``)."""
        c, q = _f32(corpus), _f32(query).reshape(-1)
        n, d = c.shape
        idx = np.empty(k, dtype=np.int64)
        sc = np.empty(k, dtype=np.float64)
        if self.lib.oracle_topk(_ptr(c), n, d, _ptr(q), k, _ptr(idx), _ptr(sc)):
            raise ValueError("oracle_topk rejected its arguments")
        return idx, sc

    def scores_cosine(self, corpus, query) -> np.ndarray:
        """All N double cosine scores of one query (``oracle_scores_cosine``)."""
        c, q = _f32(corpus), _f32(query).reshape(-1)
        n, d = c.shape
        if q.shape[0] != d:
            raise ValueError("query length != D")
        out = np.empty(n, dtype=np.float64)
        if self.lib.oracle_scores_cosine(_ptr(c), n, d, _ptr(q), _ptr(out)):
            raise ValueError("oracle_scores_cosine rejected its arguments")
        return out

    def topk_cosine(self, corpus, query, k: int):
        """(indices int64[K], cosine scores float64[K]) best-first (``oracle_topk_cosine``)."""
        c, q = _f32(corpus), _f32(query).reshape(-1)
        n, d = c.shape
        idx = np.empty(k, dtype=np.int64)
        sc = np.empty(k, dtype=np.float64)
        if self.lib.oracle_topk_cosine(_ptr(c), n, d, _ptr(q), k, _ptr(idx), _ptr(sc)):
            raise ValueError("oracle_topk_cosine rejected its arguments")
        return idx, sc

    def topk_batch(self, corpus, queries, k: int):
        """(indices int64[B, K], scores float64[B, K]) (``oracle_topk_batch``)."""
        c, q = _f32(corpus), _f32(queries)
        n, d = c.shape
        b = q.shape[0]
        idx = np.empty((b, k), dtype=np.int64)
        sc = np.empty((b, k), dtype=np.float64)
        if self.lib.oracle_topk_batch(_ptr(c), n, d, _ptr(q), b, k, _ptr(idx), _ptr(sc)):
            raise ValueError("oracle_topk_batch rejected its arguments")
        return idx, sc

    def topk_int32(self, x, k: int):
        """(values int32[K], positions int64[K]) (``oracle_topk_int32``)."""
        a = np.ascontiguousarray(x, dtype=np.int32).reshape(-1)
        val = np.empty(k, dtype=np.int32)
        pos = np.empty(k, dtype=np.int64)
        if self.lib.oracle_topk_int32(_ptr(a), a.shape[0], k, _ptr(val), _ptr(pos)):
            raise ValueError("oracle_topk_int32 rejected its arguments")
        return val, pos

    def round_bf16(self, x) -> np.ndarray:
        """fp32 values rounded to bf16 (RN-even), returned as fp32."""
        a = _f32(x)
        out = np.empty_like(a)
        self.lib.oracle_round_bf16(_ptr(a), _ptr(out), a.size)
        return out

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        self.lib.oracle_set_num_threads(int(n))


_default: Oracle | None = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(load())
    return _default


def scores(corpus, query):
    return get().scores(corpus, query)


def topk(corpus, query, k):
    return get().topk(corpus, query, k)


def topk_batch(corpus, queries, k):
    return get().topk_batch(corpus, queries, k)


def scores_cosine(corpus, query):
    return get().scores_cosine(corpus, query)


def topk_cosine(corpus, query, k):
    return get().topk_cosine(corpus, query, k)


def topk_int32(x, k):
    return get().topk_int32(x, k)


def round_bf16(x):
    return get().round_bf16(x)
