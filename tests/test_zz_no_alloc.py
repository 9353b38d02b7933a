"""topk_int32_noalloc: the int32 top-K for callers that may not allocate
device memory (for example a plugin whose GPU memory all comes from its host
application's allocator). Called through the C ABI twice in a row per case and
checked bit for bit against the oracle and against the engine's topk_int32.
This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu


def _call(lib, d, n, k, dv, dp, stream):
    return lib.topk_int32_noalloc(ctypes.c_void_p(d.data_ptr()), n, k, ctypes.c_void_p(dv.data_ptr()),
                                  ctypes.c_void_p(dp.data_ptr()), ctypes.c_void_p(stream))


def test_noalloc_matches_oracle_and_engine_on_two_calls():
    import torch

    import resident_brute_force_gb300 as rbf
    lib = rbf.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    # (n, start offset in elements, K): a ragged size with an unaligned start,
    # the full 1e8 workload, and a small array with the largest K.
    cases = [(3_000_001, 1, 50), (100_000_000, 0, 20), (777, 3, 256)]
    with rbf.Engine(16, 16, 256) as e:
        for n, offset, k in cases:
            x = workloads.int32_uniform(n + offset, seed=n)
            o_val, o_pos = oracle.topk_int32(x[offset:], k)
            d = torch.from_numpy(x).cuda()[offset:]
            e_val, e_pos = e.topk_int32(d, k)
            for _ in range(2):
                dv = torch.full((k,), -1, dtype=torch.int32, device="cuda")
                dp = torch.full((k,), -1, dtype=torch.int64, device="cuda")
                assert _call(lib, d, n, k, dv, dp, stream) == rbf.RBF_OK
                torch.cuda.synchronize()
                got_val, got_pos = dv.cpu().numpy(), dp.cpu().numpy()
                assert np.array_equal(got_val, o_val) and np.array_equal(got_pos, o_pos), (n, k)
                assert np.array_equal(got_val, e_val) and np.array_equal(got_pos, e_pos), (n, k)


def test_noalloc_rejects_oversized_k():
    import torch

    import resident_brute_force_gb300 as rbf
    lib = rbf.load_library()
    d = torch.zeros(1000, dtype=torch.int32, device="cuda")
    dv = torch.empty(300, dtype=torch.int32, device="cuda")
    dp = torch.empty(300, dtype=torch.int64, device="cuda")
    assert _call(lib, d, 1000, 257, dv, dp, 0) == rbf.RBF_ERR_INVALID_VALUE
    assert _call(lib, d, 1000, 0, dv, dp, 0) == rbf.RBF_ERR_INVALID_VALUE
    assert _call(lib, d, 100, 101, dv, dp, 0) == rbf.RBF_ERR_INVALID_VALUE
