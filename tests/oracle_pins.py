"""Pins that tie the oracle to something other than itself.

Each ``pin_*`` function takes a bound oracle (``oracle.Oracle``) and raises
``AssertionError`` when the oracle disagrees with what the pages and the
mathematics fix. The pin tests run them against the real oracle; the mutation
test runs them against copies of the oracle with planted mistakes and expects
every mistake to trip at least one pin.

What each pin rests on:
  - exhaustive search over all K-subsets (tiny N) with exact integer scores;
  - library routines: Python's stable ``sorted``, numpy ``lexsort`` /
    ``argsort(kind="stable")``, torch's CPU bf16 cast;
  - closed forms: D = 1, rows that are multiples of the query, scaled basis
    vectors, all-equal and duplicated rows, planted near-duplicates;
  - exact arithmetic: dyadic-grid data scored with int64 matrix products;
  - the standard error bound of a double dot product against exact rationals;
  - invariants every correct top-K satisfies.
"""
from __future__ import annotations

import itertools
from fractions import Fraction

import numpy as np

import workloads

INT32_MIN = -(2 ** 31)
INT32_MAX = 2 ** 31 - 1


def _better(sa, ia, sb, ib) -> bool:
    """The pages' ordering rule on one pair of (score, index) candidates."""
    if sa != sb:
        return sa > sb
    return ia < ib


def _exact_int_scores(c: np.ndarray, q: np.ndarray) -> list[int]:
    ci = c.astype(np.int64)
    qi = q.astype(np.int64)
    return [int(sum(int(a) * int(b) for a, b in zip(row, qi))) for row in ci]


# ---------------------------------------------------------------- float pins

def pin_subsets(o) -> None:
    """Tiny N: the oracle's set is the unique K-subset whose every member beats
    every non-member, listed best-first."""
    cases = [(6, 3, 11), (8, 4, 12), (9, 2, 13), (7, 5, 14)]
    for n, d, seed in cases:
        c = workloads.small_int_rows(n, d, seed, lo=-2, hi=2)
        q = workloads.small_int_rows(1, d, seed + 100, lo=-2, hi=2)[0]
        s = _exact_int_scores(c, q)
        for k in range(1, n + 1):
            winners = []
            for sub in itertools.combinations(range(n), k):
                rest = [j for j in range(n) if j not in sub]
                if all(_better(s[a], a, s[b], b) for a in sub for b in rest):
                    winners.append(sub)
            assert len(winners) == 1, "rule must single out one subset"
            want = sorted(winners[0], key=lambda j: (-s[j], j))
            idx, sc = o.topk(c, q, k)
            assert list(idx) == want, (n, d, k, list(idx), want)
            assert [float(x) for x in sc] == [float(s[j]) for j in want]


def pin_full_order_stable_sort(o) -> None:
    """K = N equals a stable sort of row indices by descending score."""
    for n, d, seed in [(40, 5, 21), (64, 17, 22), (33, 1, 23)]:
        c = workloads.small_int_rows(n, d, seed, lo=-1, hi=1)
        q = workloads.small_int_rows(1, d, seed + 7, lo=-1, hi=1)[0]
        s = _exact_int_scores(c, q)
        want = sorted(range(n), key=lambda j: -s[j])  # stable: index order on ties
        idx, _ = o.topk(c, q, n)
        assert list(idx) == want


def pin_d1_closed_form(o) -> None:
    """D = 1: sigma_i = c_i * q exactly; order by numpy's stable argsort."""
    rng = np.random.default_rng(31)
    c = rng.standard_normal((257, 1)).astype(np.float32)
    c[10] = c[3]  # one exact tie
    for qv in (1.75, -0.5):
        q = np.array([qv], dtype=np.float32)
        sig = c[:, 0].astype(np.float64) * np.float64(qv)
        want = np.argsort(-sig, kind="stable")
        idx, sc = o.topk(c, q, 257)
        assert np.array_equal(idx, want)
        assert np.array_equal(sc, sig[want])
        np.testing.assert_array_equal(o.scores(c, q), sig)


def pin_scaled_query_rows(o) -> None:
    """Rows alpha_i * q (N != D): sigma_i = alpha_i * |q|^2 exactly, so the
    top-K are the K largest alphas."""
    n, d = 37, 13
    rng = np.random.default_rng(41)
    alpha = rng.permutation(np.arange(-18, 19)).astype(np.float64)
    q = (rng.integers(-8, 9, size=d) / 8.0).astype(np.float32)
    q[0] = 0.625
    c = (alpha[:, None] * q[None, :].astype(np.float64)).astype(np.float32)
    qq = float(np.dot(q.astype(np.float64), q.astype(np.float64)))
    order = np.argsort(-alpha, kind="stable")
    for k in (1, 5, 37):
        idx, sc = o.topk(c, q, k)
        assert np.array_equal(idx, order[:k])
        assert np.array_equal(sc, alpha[order[:k]] * qq)


def pin_basis_rows(o) -> None:
    """Row i = w_i * e_{p_i}: sigma_i = w_i * q[p_i]; covers the first and
    last coordinates."""
    n, d = 50, 24
    rng = np.random.default_rng(51)
    p = rng.integers(0, d, size=n)
    p[0], p[1], p[2] = 0, d - 1, d - 1
    w = rng.integers(1, 9, size=n).astype(np.float64)
    c = np.zeros((n, d), dtype=np.float32)
    c[np.arange(n), p] = w
    q = (np.arange(d, dtype=np.float64) - 7.5).astype(np.float32)
    q[d - 1] = 100.0
    sig = w * q.astype(np.float64)[p]
    np.testing.assert_array_equal(o.scores(c, q), sig)
    order = np.lexsort((np.arange(n), -sig))
    idx, sc = o.topk(c, q, 10)
    assert np.array_equal(idx, order[:10])
    assert idx[0] in (1, 2)


def pin_duplicates_and_all_equal(o) -> None:
    """All-equal rows give indices 0..K-1; duplicated rows come out in
    ascending index order."""
    c = np.full((30, 8), 0.25, dtype=np.float32)
    q = np.ones(8, dtype=np.float32)
    idx, sc = o.topk(c, q, 7)
    assert list(idx) == list(range(7))
    assert np.all(sc == 2.0)
    rng = np.random.default_rng(61)
    base = rng.standard_normal((10, 16)).astype(np.float32)
    c = base[rng.integers(0, 10, size=80)]
    q = rng.standard_normal(16).astype(np.float32)
    idx, sc = o.topk(c, q, 80)
    for a, b, sa, sb in zip(idx[:-1], idx[1:], sc[:-1], sc[1:]):
        assert sa > sb or (sa == sb and a < b)


def pin_dyadic_exact(o) -> None:
    """Multiples of 2^-6: 4096 * sigma is an integer computed exactly by an
    int64 matrix product; scores and order must match bit for bit."""
    n, d = 300, 1024
    c = workloads.dyadic_grid(n, d, seed=71)
    q = workloads.dyadic_grid(1, d, seed=72)[0]
    ci = np.rint(c.astype(np.float64) * 64).astype(np.int64)
    qi = np.rint(q.astype(np.float64) * 64).astype(np.int64)
    s_int = ci @ qi
    sig = s_int.astype(np.float64) / 4096.0
    np.testing.assert_array_equal(o.scores(c, q), sig)
    order = np.lexsort((np.arange(n), -s_int))
    idx, sc = o.topk(c, q, 64)
    assert np.array_equal(idx, order[:64])
    assert np.array_equal(sc, sig[order[:64]])


def pin_planted(o) -> None:
    """Planted near-duplicates of each query are its best rows."""
    n, d, nq = 6000, 64, 3
    c = workloads.unit_corpus(n, d, seed=81)
    qs = workloads.unit_queries(nq, d, seed=82)
    planted = workloads.plant_near_duplicates(c, qs, per_query=10, noise=0.05, seed=83)
    for j in range(nq):
        idx8, _ = o.topk(c, qs[j], 8)
        assert set(idx8) <= set(planted[j])
        idx32, sc32 = o.topk(c, qs[j], 32)
        assert set(idx32[:10]) == set(planted[j])
        assert sc32[9] > 0.8 > sc32[10]


def pin_error_bound(o) -> None:
    """Against exact rationals, the double sum stays within the standard
    bound gamma_D * sum |c_d q_d| with unit roundoff 2^-53."""
    n, d = 24, 384
    c = workloads.unit_corpus(n, d, seed=91)
    q = workloads.unit_queries(1, d, seed=92)[0]
    sig = o.scores(c, q)
    u = 2.0 ** -53
    gamma = d * u / (1 - d * u)
    qf = [Fraction(float(x)) for x in q]
    for i in range(n):
        exact = sum(Fraction(float(a)) * b for a, b in zip(c[i], qf))
        absum = float(np.sum(np.abs(c[i].astype(np.float64) * q.astype(np.float64))))
        assert abs(Fraction(float(sig[i])) - exact) <= Fraction(gamma * absum), i


def pin_invariants(o) -> None:
    """Sorted output, distinct indices, nothing left out beats the K-th."""
    n, d = 2000, 96
    c = workloads.unit_corpus(n, d, seed=101)
    q = workloads.unit_queries(1, d, seed=102)[0]
    sig = o.scores(c, q)
    for k in (1, 8, 100, 256):
        idx, sc = o.topk(c, q, k)
        assert len(set(idx.tolist())) == k
        assert np.all((idx >= 0) & (idx < n))
        assert np.array_equal(sc, sig[idx])
        for a in range(k - 1):
            assert _better(sc[a], idx[a], sc[a + 1], idx[a + 1])
        rest = np.setdiff1d(np.arange(n), idx)
        kth_s, kth_i = sc[-1], idx[-1]
        assert np.all(sig[rest] <= kth_s)
        assert np.all(rest[sig[rest] == kth_s] > kth_i)


def pin_nan_and_signed_zero(o) -> None:
    """NaN scores rank as -inf; -0.0 ties +0.0 and the index decides."""
    c = np.array([[np.nan, 1.0], [0.0, 0.0], [-0.0, 0.0], [1.0, 1.0], [-1.0, 0.0]],
                 dtype=np.float32)
    q = np.array([1.0, 1.0], dtype=np.float32)
    idx, sc = o.topk(c, q, 5)
    assert list(idx) == [3, 1, 2, 4, 0]
    assert sc[-1] == -np.inf
    c2 = np.array([[-1.0], [1.0]], dtype=np.float32)
    q2 = np.array([0.0], dtype=np.float32)   # -0.0 vs +0.0 scores
    idx, _ = o.topk(c2, q2, 2)
    assert list(idx) == [0, 1]


def pin_batch_matches_rows(o) -> None:
    """The batched oracle answers each query exactly as the single one does,
    checked on rows that are multiples of each query (closed form)."""
    rng = np.random.default_rng(111)
    d, b = 12, 4
    qs = (rng.integers(-4, 5, size=(b, d)) / 4.0).astype(np.float32)
    qs[:, 0] = 1.0
    alpha = rng.permutation(np.arange(1, 26)).astype(np.float64)
    c = (alpha[:, None] * qs[0][None, :].astype(np.float64)).astype(np.float32)
    idx, sc = o.topk_batch(c, qs, 6)
    assert np.array_equal(idx[0], np.argsort(-alpha, kind="stable")[:6])
    for j in range(b):
        ij, sj = o.topk(c, qs[j], 6)
        assert np.array_equal(idx[j], ij) and np.array_equal(sc[j], sj)
        s_int = _exact_int_scores(np.rint(c * 4), np.rint(qs[j] * 4))
        want = sorted(range(25), key=lambda r: (-s_int[r], r))[:6]
        assert list(idx[j]) == want


# ---------------------------------------------------------------- int32 pins

def pin_i32_closed_forms(o) -> None:
    """All-equal, strictly decreasing and strictly increasing arrays."""
    x = np.full(1000, 7, dtype=np.int32)
    val, pos = o.topk_int32(x, 20)
    assert list(pos) == list(range(20)) and np.all(val == 7)
    x = np.arange(500, 0, -1, dtype=np.int32)
    val, pos = o.topk_int32(x, 50)
    assert list(pos) == list(range(50)) and list(val) == list(range(500, 450, -1))
    x = np.arange(-250, 250, dtype=np.int32)
    val, pos = o.topk_int32(x, 20)
    assert list(pos) == list(range(499, 479, -1)) and list(val) == list(range(249, 229, -1))


def pin_i32_extremes(o) -> None:
    """INT32_MIN / INT32_MAX heavy arrays, planted ties at the K boundary."""
    x = np.full(300, INT32_MIN, dtype=np.int32)
    x[[5, 17, 250]] = INT32_MAX
    x[[3, 4]] = 0
    val, pos = o.topk_int32(x, 8)
    assert list(val) == [INT32_MAX] * 3 + [0, 0] + [INT32_MIN] * 3
    assert list(pos) == [5, 17, 250, 3, 4, 0, 1, 2]
    x = np.zeros(100, dtype=np.int32)
    x[[10, 20, 30, 40, 50]] = 9
    val, pos = o.topk_int32(x, 3)
    assert list(pos) == [10, 20, 30]


def pin_i32_lexsort(o) -> None:
    """Random narrow-range arrays against numpy's lexsort on (value, pos)."""
    for seed, lo, hi, n, k in [(121, -5, 5, 5000, 50), (122, INT32_MIN, INT32_MIN + 3, 777, 20),
                               (123, INT32_MAX - 2, INT32_MAX, 999, 64)]:
        x = workloads.int32_small_range(n, seed, lo, hi)
        order = np.lexsort((np.arange(n), -x.astype(np.int64)))
        val, pos = o.topk_int32(x, k)
        assert np.array_equal(pos, order[:k]) and np.array_equal(val, x[order[:k]])


def pin_i32_subsets(o) -> None:
    x = workloads.int32_small_range(9, 131, -2, 2)
    for k in range(1, 10):
        winners = [s for s in itertools.combinations(range(9), k)
                   if all(_better(int(x[a]), a, int(x[b]), b)
                          for a in s for b in range(9) if b not in s)]
        assert len(winners) == 1
        want = sorted(winners[0], key=lambda j: (-int(x[j]), j))
        _, pos = o.topk_int32(x, k)
        assert list(pos) == want


# ---------------------------------------------------------------- bf16 pin

def pin_bf16_rounding(o) -> None:
    """Hand values for round-to-nearest-even, then torch's CPU bf16 cast."""
    one = 1.0
    cases = {one + 2 ** -8: one, one + 3 * 2 ** -8: one + 2 ** -6,
             one + 2 ** -8 + 2 ** -20: one + 2 ** -7, -(one + 2 ** -8): -one,
             0.0: 0.0, 3.0: 3.0}
    xs = np.array(list(cases.keys()), dtype=np.float32)
    got = o.round_bf16(xs)
    assert np.array_equal(got, np.array(list(cases.values()), dtype=np.float32))
    import torch
    rng = np.random.default_rng(141)
    x = rng.standard_normal(20000).astype(np.float32)
    x[:200] = (rng.integers(-2 ** 15, 2 ** 15, 200) * 2.0 ** -12).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(o.round_bf16(x), ref)


# --------------------------------------------------------------- cosine pins
#
# Cosine similarity (GPU-Resident Top-K for Agentic RAG, section 4 step 2,
# cosine mode): inner product / (||q|| * ||c_i||), -inf when that denominator
# is not positive.

# Integer vectors with integer L2 norms: the cosine of any two is the exact
# rational dot / (|a| |b|).
_PYTH = [((3, 4, 0), 5), ((0, 3, 4), 5), ((2, 3, 6), 7), ((1, 4, 8), 9), ((4, 4, 7), 9),
         ((2, 6, 9), 11), ((6, 2, 3), 7), ((-2, 3, -6), 7), ((8, -4, 1), 9), ((0, 0, 5), 5)]


def pin_cosine_exact_rationals(o) -> None:
    """Integer rows and queries with integer norms: every cosine equals the
    rational dot / (|c| |q|) to within one rounding of each double step."""
    c = np.array([v for v, _ in _PYTH], dtype=np.float32)
    norms = [nv for _, nv in _PYTH]
    for qi, (qv, qn) in enumerate(_PYTH):
        q = np.array(qv, dtype=np.float32)
        got = o.scores_cosine(c, q)
        for i, (cv, cn) in enumerate(_PYTH):
            exact = Fraction(sum(a * b for a, b in zip(cv, qv)), cn * qn)
            assert abs(Fraction(float(got[i])) - exact) <= Fraction(4, 2 ** 53), (qi, i, got[i], exact)


def pin_cosine_parallel_and_orthogonal(o) -> None:
    """Rows alpha * q give +1 (alpha > 0) or -1 (alpha < 0), to rounding;
    with alpha a power of two they are bit-identical, so they tie and come
    first by index; rows orthogonal to q give exactly 0."""
    rng = np.random.default_rng(151)
    d = 24
    q = rng.standard_normal(d).astype(np.float32)
    q[5] = 0.0
    alphas = [4.0, 0.5, -2.0, 0.125, -7.5, 2.0, 3.0, 11.0]
    rows = [(a * q.astype(np.float64)).astype(np.float32) for a in alphas]
    e5 = np.zeros(d, dtype=np.float32)
    e5[5] = 4.0
    rows += [e5]
    c = np.stack(rows)
    got = o.scores_cosine(c, q)
    for a, g in zip(alphas, got[:8]):
        assert abs(g - np.sign(a)) < 1e-6, (a, g)
    assert got[0] == got[1] == got[3] == got[5]
    assert got[8] == 0.0
    idx, _ = o.topk_cosine(c[[0, 1, 2, 3, 4, 5, 8]], q, 4)
    assert list(idx) == [0, 1, 3, 5], list(idx)


def pin_cosine_zero_vectors(o) -> None:
    """A zero row scores -inf; a zero query scores every row -inf, so the
    top-K is rows 0..K-1 (ties by index)."""
    rng = np.random.default_rng(161)
    c = rng.standard_normal((30, 8)).astype(np.float32)
    c[4] = 0.0
    q = rng.standard_normal(8).astype(np.float32)
    got = o.scores_cosine(c, q)
    assert got[4] == -np.inf and np.all(np.isfinite(np.delete(got, 4)))
    idx, _ = o.topk_cosine(c, q, 30)
    assert idx[-1] == 4
    z = np.zeros(8, dtype=np.float32)
    assert np.all(o.scores_cosine(c, z) == -np.inf)
    idx, sc = o.topk_cosine(c, z, 6)
    assert list(idx) == list(range(6)) and np.all(sc == -np.inf)


def pin_cosine_scale_invariance(o) -> None:
    """Scaling a row or the query by a positive power of two changes no
    cosine (bit for bit: every double step scales exactly); any positive
    scale changes it by rounding only. Rows scaled by powers of two tie with
    their originals, and the lower index comes first."""
    rng = np.random.default_rng(171)
    n, d = 40, 33
    c = rng.standard_normal((n, d)).astype(np.float32)
    q = rng.standard_normal(d).astype(np.float32)
    base = o.scores_cosine(c, q)
    p2 = (2.0 ** rng.integers(-6, 7, size=n)).astype(np.float32)
    assert np.array_equal(o.scores_cosine(c * p2[:, None], q * np.float32(8.0)), base)
    s = rng.uniform(0.1, 10.0, size=n).astype(np.float64)
    cs = (c.astype(np.float64) * s[:, None]).astype(np.float32)
    np.testing.assert_allclose(o.scores_cosine(cs, q * np.float32(0.3)), base, rtol=1e-6, atol=1e-7)
    dup = np.concatenate([c, c[7:8] * np.float32(4.0), c[7:8] * np.float32(0.25)])
    idx, sc = o.topk_cosine(dup, c[7], 3)
    assert list(idx) == [7, n, n + 1] and sc[0] == sc[1] == sc[2]


def pin_cosine_unit_rows_match_ip_and_order(o) -> None:
    """On rows and a query normalised to unit length (in double, then fp32)
    the cosine equals the inner product to fp32 rounding of the norms; and
    K = N lists rows in numpy's stable descending order of the scores."""
    rng = np.random.default_rng(181)
    n, d = 300, 64
    c64 = rng.standard_normal((n, d))
    c = (c64 / np.linalg.norm(c64, axis=1, keepdims=True)).astype(np.float32)
    q64 = rng.standard_normal(d)
    q = (q64 / np.linalg.norm(q64)).astype(np.float32)
    np.testing.assert_allclose(o.scores_cosine(c, q), o.scores(c, q), rtol=0, atol=1e-6)
    c2 = rng.standard_normal((n, d)).astype(np.float32)
    c2[17] = c2[3]
    sig = o.scores_cosine(c2, q)
    idx, sc = o.topk_cosine(c2, q, n)
    assert np.array_equal(idx, np.argsort(-sig, kind="stable"))
    assert np.array_equal(sc, sig[idx])


ALL_PINS = [
    pin_subsets, pin_full_order_stable_sort, pin_d1_closed_form, pin_scaled_query_rows,
    pin_basis_rows, pin_duplicates_and_all_equal, pin_dyadic_exact, pin_planted,
    pin_error_bound, pin_invariants, pin_nan_and_signed_zero, pin_batch_matches_rows,
    pin_i32_closed_forms, pin_i32_extremes, pin_i32_lexsort, pin_i32_subsets,
    pin_bf16_rounding,
    pin_cosine_exact_rationals, pin_cosine_parallel_and_orthogonal, pin_cosine_zero_vectors,
    pin_cosine_scale_invariance, pin_cosine_unit_rows_match_ip_and_order,
]
