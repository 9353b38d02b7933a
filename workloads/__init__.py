"""Seeded synthetic inputs shaped like the workloads of the retrieval pages.

This module is shared by the oracle side and the CUDA side of the tests and
the bench. It holds no scoring and no selection arithmetic: it only draws
random numbers and lays them out. Everything is a deterministic function of
(seed, sizes): rows are generated in fixed blocks of ``BLOCK_ROWS`` rows, block
``b`` drawing from its own PCG64 stream seeded by ``SeedSequence([seed, stream,
b])``, so the result does not depend on how many threads fill the blocks.

Workloads (GPU-Resident Top-K for Agentic RAG, section 5 "the receipts"):
Gaussian embeddings, L2-normalised, inner-product scoring, corpus seed 1 and
query seed 2 ("seed+1"). The flat int32 workload (CUDA programming model
series 9, section 1) is 1e8 values drawn uniformly over the full int32 range.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

BLOCK_ROWS = 8192
INT_BLOCK = 1 << 22

# Stream identifiers keep independent draws with the same seed apart.
STREAM_CORPUS = 0
STREAM_QUERY = 1
STREAM_PLANT_POS = 2
STREAM_PLANT_NOISE = 3
STREAM_INT32 = 4
STREAM_GRID = 5


def _rng(seed: int, stream: int, block: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, block])))


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _parallel(fn, count: int) -> None:
    if count <= 1:
        for b in range(count):
            fn(b)
        return
    with ThreadPoolExecutor(max_workers=_threads()) as ex:
        list(ex.map(fn, range(count)))


def gaussian_rows(n: int, d: int, seed: int, stream: int = STREAM_CORPUS,
                  normalize: bool = True) -> np.ndarray:
    """(n, d) float32 rows with i.i.d. N(0, 1) entries, each row L2-normalised
    in float64 before the cast when ``normalize`` is set."""
    out = np.empty((n, d), dtype=np.float32)
    nblocks = (n + BLOCK_ROWS - 1) // BLOCK_ROWS

    def fill(b: int) -> None:
        r0 = b * BLOCK_ROWS
        r1 = min(n, r0 + BLOCK_ROWS)
        g = _rng(seed, stream, b).standard_normal((r1 - r0, d))
        if normalize:
            norms = np.sqrt(np.einsum("ij,ij->i", g, g))
            norms[norms == 0.0] = 1.0
            g /= norms[:, None]
        out[r0:r1] = g

    _parallel(fill, nblocks)
    return out


def unit_corpus(n: int, d: int, seed: int = 1) -> np.ndarray:
    """Unit-norm Gaussian corpus (the pages' synthetic embeddings)."""
    return gaussian_rows(n, d, seed, STREAM_CORPUS)


def unit_corpus_rows(row0: int, n: int, d: int, seed: int = 1) -> np.ndarray:
    """Rows [row0, row0 + n) of the unit-norm Gaussian corpus of any size
    larger than row0 + n: the same bytes as unit_corpus(N, d, seed)[row0:row0 + n]
    (block b of rows always draws from its own stream, and a short last block
    draws a prefix of the same sequence), without generating the other rows.
    This is how one row shard of a corpus too large for one GPU is made."""
    out = np.empty((n, d), dtype=np.float32)
    b0 = row0 // BLOCK_ROWS
    b1 = (row0 + n + BLOCK_ROWS - 1) // BLOCK_ROWS

    def fill(i: int) -> None:
        b = b0 + i
        lo = max(row0, b * BLOCK_ROWS)
        hi = min(row0 + n, (b + 1) * BLOCK_ROWS)
        if hi <= lo:
            return
        g = _rng(seed, STREAM_CORPUS, b).standard_normal((hi - b * BLOCK_ROWS, d))[lo - b * BLOCK_ROWS:]
        norms = np.sqrt(np.einsum("ij,ij->i", g, g))
        norms[norms == 0.0] = 1.0
        g /= norms[:, None]
        out[lo - row0:hi - row0] = g

    _parallel(fill, b1 - b0)
    return out


def unit_queries(b: int, d: int, seed: int = 2) -> np.ndarray:
    """Unit-norm Gaussian queries: the corpus distribution under seed+1."""
    return gaussian_rows(b, d, seed, STREAM_QUERY)


def plant_near_duplicates(corpus: np.ndarray, queries: np.ndarray, per_query: int = 10,
                          noise: float = 0.05, seed: int = 3) -> np.ndarray:
    """Replace ``per_query`` distinct random rows per query with
    normalise(q + noise * g), g ~ N(0, I). All planted rows are distinct across
    queries. Returns the planted row indices, shape (len(queries), per_query).

    Modifies ``corpus`` in place.
    """
    n = corpus.shape[0]
    pos, rows = _planted(n, queries, per_query, noise, seed)
    corpus[pos.reshape(-1)] = rows
    return pos


def plant_near_duplicates_shard(shard: np.ndarray, row0: int, n_total: int, queries: np.ndarray,
                                per_query: int = 10, noise: float = 0.05, seed: int = 3) -> np.ndarray:
    """plant_near_duplicates on a corpus of n_total rows of which ``shard``
    holds rows [row0, row0 + len(shard)): the rows planted there are the ones
    the whole-corpus call would plant in that range. Returns every planted
    global row index, shape (len(queries), per_query). Modifies ``shard``."""
    pos, rows = _planted(n_total, queries, per_query, noise, seed)
    flat = pos.reshape(-1)
    mine = (flat >= row0) & (flat < row0 + shard.shape[0])
    shard[flat[mine] - row0] = rows[mine]
    return pos


def _planted(n: int, queries: np.ndarray, per_query: int, noise: float, seed: int):
    """Planted positions (nq, per_query) over n rows and the planted rows (nq * per_query, d), fp32."""
    nq, d = queries.shape
    total = nq * per_query
    if total > n:
        raise ValueError("more planted rows than corpus rows")
    pos = _rng(seed, STREAM_PLANT_POS, 0).choice(n, size=total, replace=False)
    pos = pos.reshape(nq, per_query).astype(np.int64)
    g = _rng(seed, STREAM_PLANT_NOISE, 0).standard_normal((total, d))
    rows = queries.astype(np.float64).repeat(per_query, axis=0) + noise * g
    rows /= np.sqrt(np.einsum("ij,ij->i", rows, rows))[:, None]
    return pos, rows.astype(np.float32)


def int32_uniform(n: int, seed: int = 1) -> np.ndarray:
    """n int32 values uniform over the full int32 range (raw 32-bit draws)."""
    out = np.empty(n, dtype=np.int32)
    nblocks = (n + INT_BLOCK - 1) // INT_BLOCK

    def fill(b: int) -> None:
        i0 = b * INT_BLOCK
        i1 = min(n, i0 + INT_BLOCK)
        raw = _rng(seed, STREAM_INT32, b).integers(0, 1 << 32, size=i1 - i0, dtype=np.uint64)
        out[i0:i1] = raw.astype(np.uint32).view(np.int32)

    _parallel(fill, nblocks)
    return out


def dyadic_grid(n: int, d: int, seed: int, bits: int = 6, stream: int = STREAM_GRID) -> np.ndarray:
    """(n, d) float32 entries k / 2**bits with k uniform in [-2**bits, 2**bits].

    Every such value is exact in fp32 and in bf16 (at most 7 significant bits
    for bits <= 6), every product of two is a multiple of 2**(-2*bits), and a
    sum of up to 2**(24 - 2*bits - 1) of them is exact in fp32 in any order.
    The grid is coarse, so exact score ties are common.
    """
    scale = 1 << bits
    out = np.empty((n, d), dtype=np.float32)
    nblocks = max(1, (n + BLOCK_ROWS - 1) // BLOCK_ROWS)

    def fill(b: int) -> None:
        r0 = b * BLOCK_ROWS
        r1 = min(n, r0 + BLOCK_ROWS)
        if r1 <= r0:
            return
        k = _rng(seed, stream, b).integers(-scale, scale + 1, size=(r1 - r0, d))
        out[r0:r1] = k.astype(np.float32) / np.float32(scale)

    _parallel(fill, nblocks)
    return out


def small_int_rows(n: int, d: int, seed: int, lo: int = -3, hi: int = 3,
                   stream: int = STREAM_GRID) -> np.ndarray:
    """(n, d) float32 small integers in [lo, hi]: tie-heavy, exactly scorable."""
    k = _rng(seed, stream, 0).integers(lo, hi + 1, size=(n, d))
    return k.astype(np.float32)


def int32_small_range(n: int, seed: int, lo: int, hi: int) -> np.ndarray:
    """n int32 values uniform in [lo, hi]: a narrow range makes ties common."""
    return _rng(seed, STREAM_INT32, 1 << 20).integers(lo, hi + 1, size=n).astype(np.int32)
