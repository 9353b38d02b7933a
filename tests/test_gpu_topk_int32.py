"""Flat int32 two-stage top-K through the C ABI against the oracle
(bit-exact values, positions and order)."""
import json
import os

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
INT32_MIN, INT32_MAX = -(2 ** 31), 2 ** 31 - 1


@pytest.fixture(scope="module")
def eng():
    import resident_brute_force_gb300 as rbf
    e = rbf.Engine(16, 16, 256)
    yield e
    e.close()


def _dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).cuda()


def _check(eng, d, x, k):
    val, pos = eng.topk_int32(d, k)
    o_val, o_pos = oracle.topk_int32(x, k)
    assert np.array_equal(pos, o_pos), (pos[:8], o_pos[:8])
    assert np.array_equal(val, o_val)


def test_golden(eng):
    with open(os.path.join(GOLDEN, "tiny_i32.json")) as f:
        g = json.load(f)
    x = np.array(g["x"], dtype=np.int32)
    for case in g["cases"]:
        val, pos = eng.topk_int32(_dev(x), case["k"])
        assert val.tolist() == case["val"] and pos.tolist() == case["pos"]


@pytest.mark.parametrize("n", [1, 3, 4, 5, 130, 4097, 100_003, 1_000_001])
@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_uniform_full_range_unaligned(eng, n, offset):
    x = workloads.int32_uniform(n + offset, seed=n)
    d = _dev(x)[offset:]          # 4-byte aligned, not 16-byte aligned
    for k in (1, 20, 50, 256):
        if k <= n:
            _check(eng, d, x[offset:], k)


def test_ties_and_extremes(eng):
    for lo, hi, n in [(-3, 3, 200_000), (INT32_MIN, INT32_MIN + 1, 50_000), (INT32_MAX - 1, INT32_MAX, 50_000)]:
        x = workloads.int32_small_range(n, seed=n, lo=lo, hi=hi)
        for k in (20, 50, 256):
            _check(eng, _dev(x), x, k)
    x = np.full(300_000, 5, dtype=np.int32)
    val, pos = eng.topk_int32(_dev(x), 256)
    assert pos.tolist() == list(range(256)) and np.all(val == 5)
    x = np.arange(1_000_000, 0, -1, dtype=np.int32)
    _check(eng, _dev(x), x, 50)
    x = np.arange(-500_000, 500_000, dtype=np.int32)
    _check(eng, _dev(x), x, 50)


def test_device_outputs_match_host(eng):
    import torch
    x = workloads.int32_uniform(2_000_000, seed=5)
    d = _dev(x)
    dv = torch.empty(50, dtype=torch.int32, device="cuda")
    dp = torch.empty(50, dtype=torch.int64, device="cuda")
    eng.topk_int32_dev(d, 50, dv, dp)
    torch.cuda.synchronize()
    val, pos = eng.topk_int32(d, 50)
    assert np.array_equal(dv.cpu().numpy(), val) and np.array_equal(dp.cpu().numpy(), pos)


def test_argument_errors(eng):
    import resident_brute_force_gb300 as rbf
    d = _dev(np.arange(10, dtype=np.int32))
    for k in (0, 11, 257):
        with pytest.raises(rbf.RbfError) as ei:
            eng.topk_int32(d, k)
        assert ei.value.status == rbf.RBF_ERR_INVALID_VALUE
    with pytest.raises(rbf.RbfError) as ei:
        eng.topk_int32(d[:0], 1)                                  # empty array
    assert ei.value.status == rbf.RBF_ERR_INVALID_VALUE


def test_full_size_1e8(eng):
    """100,000,000 int32 uniform over the full range, K = 20 and 50."""
    n = 100_000_000
    x = workloads.int32_uniform(n, seed=1)
    d = _dev(x)
    o_val, o_pos = oracle.topk_int32(x, 50)
    for k in (20, 50):
        val, pos = eng.topk_int32(d, k)
        assert np.array_equal(pos, o_pos[:k]) and np.array_equal(val, o_val[:k])


def test_sample_bound_cases(eng):
    """n >= 262,144: CTA b starts from a lower bound on the K-th key taken
    from its own slice of 32,768 values (vectors 8192 b .. 8192 b + 8191 of
    the 16-byte aligned body). Increasing arrays put every winner outside the
    early slices; constant arrays tie every key with the bound."""
    n = 600_000
    cases = [
        np.arange(n, dtype=np.int32),                                   # winners at the end
        np.arange(n, 0, -1, dtype=np.int32),                            # winners at the start
        np.full(n, 7, dtype=np.int32),                                  # every element ties
        workloads.int32_small_range(n, seed=77, lo=-3, hi=3),           # heavy ties
        np.where(np.arange(n) % 1000 == 999, np.int32(INT32_MAX), np.int32(INT32_MIN)).astype(np.int32),
    ]
    for x in cases:
        for k in (1, 20, 50, 256):
            _check(eng, _dev(x), x, k)


@pytest.mark.parametrize("offset", [0, 3])
def test_winners_inside_one_slice(eng, offset):
    """Every winner lies in one CTA's bound slice (slice 7), at random
    positions, with ties among them: that slice's bound is the exact K-th of
    its group maxima, the other slices' bounds are far below it."""
    n = 1_000_003
    rng = np.random.default_rng(8)
    x = workloads.int32_small_range(n + offset, seed=9, lo=-1000, hi=1000)
    lo = offset + ((16 - (offset * 4) % 16) % 16) // 4 + 7 * 32768
    hot = lo + rng.choice(32768, size=600, replace=False)
    x[hot] = INT32_MAX - rng.integers(0, 40, size=600).astype(np.int32)
    d = _dev(x)[offset:]
    for k in (1, 20, 50, 256):
        _check(eng, d, x[offset:], k)
