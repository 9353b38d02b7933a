"""Parity rules between the CUDA path and the oracle.

Float scoring (fp32 path): every GPU score within 1e-5 relative of the
oracle's double score of the same row, with a floor of 1e-2 on the magnitude
(a relative bound is meaningless near zero). Index sets: equal except where
the oracle's K-th and (K+1)-th scores are closer than the tolerance, read as:
every returned row scores at least sigma_(K) - tol, and every row scoring more
than sigma_(K) + tol is returned. The GPU list must be sorted by its own
scores under the ordering rule and its indices distinct.

bf16 path: the same with an absolute tolerance of 2e-2 on unit-norm data.

int32 and exactly representable float inputs: bit-exact indices, order and
values.
"""
from __future__ import annotations

import numpy as np

FP32_REL = 1e-5
FP32_FLOOR = 1e-2
BF16_ABS = 2e-2


def fp32_tol(s):
    return FP32_REL * np.maximum(np.abs(s), FP32_FLOOR)


def check_sorted_distinct(idx: np.ndarray, score: np.ndarray, n: int) -> None:
    assert len(set(idx.tolist())) == len(idx), "duplicate indices"
    assert np.all((idx >= 0) & (idx < n)), "index out of range"
    for a in range(len(idx) - 1):
        sa, sb = score[a], score[a + 1]
        assert sa > sb or (sa == sb and idx[a] < idx[a + 1]), f"not best-first at {a}"


def check_float_topk(idx, score, sigma: np.ndarray, k: int, tol_abs=None) -> None:
    """idx/score: GPU result; sigma: oracle double scores of ALL rows."""
    idx = np.asarray(idx).astype(np.int64)
    score = np.asarray(score).astype(np.float64)
    n = sigma.shape[0]
    assert idx.shape == (k,) and score.shape == (k,)
    check_sorted_distinct(idx, score, n)
    ref = sigma[idx]
    tol = fp32_tol(ref) if tol_abs is None else np.full_like(ref, tol_abs)
    bad = np.abs(score - ref) > tol
    assert not bad.any(), f"score mismatch at {np.nonzero(bad)[0][:5]}: {score[bad][:5]} vs {ref[bad][:5]}"
    part = np.partition(-sigma, k - 1)[k - 1]
    sk = -part
    t = float(fp32_tol(np.array([sk]))[0]) if tol_abs is None else tol_abs
    assert np.all(sigma[idx] >= sk - t), "returned a row clearly below the K-th"
    must = np.nonzero(sigma > sk + t)[0]
    missing = np.setdiff1d(must, idx)
    assert missing.size == 0, f"missing rows clearly above the K-th: {missing[:5]}"


def check_exact(idx, score, o_idx, o_score) -> None:
    assert np.array_equal(np.asarray(idx).astype(np.int64), np.asarray(o_idx).astype(np.int64)), \
        f"indices differ: {idx[:8]} vs {o_idx[:8]}"
    assert np.array_equal(np.asarray(score).astype(np.float64), np.asarray(o_score).astype(np.float64)), \
        f"scores differ: {score[:8]} vs {o_score[:8]}"
