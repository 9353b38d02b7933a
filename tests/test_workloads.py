"""The seeded input generators: deterministic in (seed, sizes), independent
of the number of threads that fill them, and shaped as the pages' workloads
say (unit-norm Gaussian rows, raw 32-bit int32 draws, an exact dyadic grid,
planted near-duplicates that lead their query's list)."""
import numpy as np
import pytest

import workloads


@pytest.mark.parametrize("make", [
    lambda: workloads.unit_corpus(20_000, 48, seed=11),
    lambda: workloads.int32_uniform((1 << 22) + 12_345, seed=12),
    lambda: workloads.dyadic_grid(17_000, 24, seed=13),
])
def test_same_bytes_with_one_thread(make, monkeypatch):
    many = make()
    monkeypatch.setattr(workloads, "_threads", lambda: 1)
    one = make()
    assert many.dtype == one.dtype and np.array_equal(many.view(np.uint8), one.view(np.uint8))


def test_seeds_and_streams_differ():
    a = workloads.unit_corpus(100, 16, seed=1)
    assert np.array_equal(a, workloads.unit_corpus(100, 16, seed=1))
    assert not np.array_equal(a, workloads.unit_corpus(100, 16, seed=2))
    assert not np.array_equal(a, workloads.unit_queries(100, 16, seed=1))   # another stream


def test_unit_rows():
    c = workloads.unit_corpus(10_000, 384, seed=1).astype(np.float64)
    norms = np.sqrt((c * c).sum(axis=1))
    assert np.all(np.abs(norms - 1.0) < 1e-6)
    # N(0, 1) entries scaled by 1 / sqrt(D): the mean entry is ~0, the variance ~1 / D
    assert abs(c.mean()) < 1e-3 and abs(c.var() * 384 - 1.0) < 0.01


def test_int32_covers_the_full_range():
    x = workloads.int32_uniform(1_000_000, seed=1).astype(np.int64)
    assert x.min() < -(2**31) + 2**23 and x.max() > 2**31 - 2**23
    assert abs(x.mean()) < 2**31 * 0.01 and (x < 0).mean() == pytest.approx(0.5, abs=0.01)


def test_dyadic_grid_is_exact():
    g = workloads.dyadic_grid(5000, 64, seed=3)
    k = g.astype(np.float64) * 64
    assert np.array_equal(k, np.round(k)) and k.min() == -64 and k.max() == 64
    bf16 = (g.view(np.uint32) & 0xFFFF0000).view(np.float32)   # bf16 keeps the top 16 bits
    assert np.array_equal(bf16, g)


def test_planted_rows_are_distinct_and_lead():
    c = workloads.unit_corpus(50_000, 256, seed=1)
    qs = workloads.unit_queries(40, 256, seed=2)
    pos = workloads.plant_near_duplicates(c, qs, per_query=10, noise=0.05, seed=3)
    assert pos.shape == (40, 10) and len(np.unique(pos)) == 400
    scores = c.astype(np.float64) @ qs.astype(np.float64).T          # (N, 40)
    expect = 1.0 / np.sqrt(1.0 + 0.0025 * 256)
    for j in range(40):
        planted = scores[pos[j], j]
        assert np.all(np.abs(planted - expect) < 0.1)
        others = np.delete(scores[:, j], pos.reshape(-1))
        assert planted.min() > others.max()


def test_row_ranges_match_the_whole_corpus():
    """A shard generated on its own has the whole corpus's bytes in its range,
    and shard planting plants exactly what whole-corpus planting plants there."""
    full = workloads.unit_corpus(30_000, 40, seed=1)
    for r0, n in [(0, 30_000), (5, 100), (8190, 10), (8000, 17_000), (29_999, 1), (16_384, 8192)]:
        assert np.array_equal(workloads.unit_corpus_rows(r0, n, 40, seed=1), full[r0:r0 + n]), (r0, n)
    qs = workloads.unit_queries(7, 40, seed=2)
    whole = full.copy()
    pos = workloads.plant_near_duplicates(whole, qs, per_query=10, noise=0.05, seed=3)
    for r0, n in [(0, 12_000), (12_000, 18_000), (1000, 20_000)]:
        part = full[r0:r0 + n].copy()
        pos_s = workloads.plant_near_duplicates_shard(part, r0, 30_000, qs, per_query=10, noise=0.05, seed=3)
        assert np.array_equal(pos_s, pos) and np.array_equal(part, whole[r0:r0 + n])
