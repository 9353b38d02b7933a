"""The largest sizes the boundary accepts, through the C ABI: D = RBF_MAX_D
and K = RBF_MAX_K on the single-query path, a full max_batch of queries on
the batched path, and int32 positions past 2^31 (answers known by
construction where the oracle would need a sort of billions of pairs)."""
import numpy as np
import pytest

import oracle
import workloads
from tests.parity import check_exact

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rbf():
    import resident_brute_force_gb300 as rbf
    rbf.load_library()
    return rbf


def test_max_d_and_max_k_single_query(rbf):
    """D = 8192 (generic width, query in shared memory) and K = 256 on dyadic
    data, whose fp32 sums are exact: bit-exact against the oracle."""
    n, d = 20_001, rbf.RBF_MAX_D
    c = workloads.dyadic_grid(n, d, seed=201, bits=4)
    q = workloads.dyadic_grid(1, d, seed=202, bits=4)[0]
    with rbf.Engine(n, d, rbf.RBF_MAX_K) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident(q, rbf.RBF_MAX_K)
        check_exact(idx, sc, *oracle.topk(c, q, rbf.RBF_MAX_K))


def test_max_d_batched(rbf):
    """D = 8192 on the batched path: 128 K chunks per tile, dyadic data exact
    in bf16 with exact fp32 sums."""
    n, d, b = 3000, rbf.RBF_MAX_D, 130
    c = workloads.dyadic_grid(n, d, seed=203, bits=4)
    qs = workloads.dyadic_grid(b, d, seed=204, bits=4)
    with rbf.Engine(n, d, 32, max_batch=b, flags=rbf.RBF_FLAG_BF16_CORPUS) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, 32)
        for j in range(0, b, 9):
            check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], 32))


def test_max_batch(rbf):
    """4,096 queries in one call: 16 launches of 256 queries, every query
    bit-exact on dyadic data."""
    n, d, b = 5000, 64, 4096
    c = workloads.dyadic_grid(n, d, seed=205)
    qs = workloads.dyadic_grid(b, d, seed=206)
    with rbf.Engine(n, d, 32, max_batch=b, flags=rbf.RBF_FLAG_BF16_CORPUS) as e:
        e.upload_corpus_rowmajor(c)
        idx, sc = e.search_resident_batch(qs, 32)
        o_idx, o_sc = oracle.topk_batch(c, qs, 32)
        assert np.array_equal(idx.astype(np.int64), o_idx)
        assert np.array_equal(sc.astype(np.float64), o_sc)


def test_int32_positions_past_2_31(rbf):
    """n = 2^31 + 100 int32 values, all -5 except planted values, several of
    them (and a tie) at positions >= 2^31: the top K is the planted values by
    value then position, then the lowest positions holding -5."""
    import torch
    n = 2 ** 31 + 100
    x = torch.full((n,), -5, dtype=torch.int32, device="cuda")
    plant = {2 ** 31 + 99: 1000, 2 ** 31: 1000, 7: 1000, 2 ** 31 - 1: 999, 2 ** 30: 2 ** 31 - 1,
             2 ** 31 + 50: -(2 ** 31), 12345: 3}
    for p, v in plant.items():
        x[p] = v
    real = sorted((pv for pv in plant.items() if pv[1] > -5), key=lambda pv: (-pv[1], pv[0]))
    with rbf.Engine(16, 16, 256) as e:
        for k in (3, 6, 20, 100):
            val, pos = e.topk_int32(x, k)
            want = real[:k]
            fill = [p for p in range(k + len(plant)) if p not in plant][:k - len(want)]
            assert pos.tolist() == [p for p, _ in want] + fill, (k, pos.tolist())
            assert val.tolist() == [v for _, v in want] + [-5] * len(fill)
    del x
    torch.cuda.empty_cache()
