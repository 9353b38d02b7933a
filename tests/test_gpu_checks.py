"""The checked build (-DRBF_CHECKS): every index a kernel derives for a list
slot, a list length, a per-query bound or a merge read is compared with the
buffer's capacity before the access; a miss skips the access and sets a bit
that the host returns as RBF_ERR_BOUNDS. (compute-sanitizer is not used; this
build stands in for its out-of-bounds checks on those accesses.)

The paths run in a child process that loads librbf_checks.so (RBF_LIB), so
that the test process keeps its own library:
- every single-query, batched, int32, cosine, no-alloc and view path on small
  cases must finish with no bounds report and with the oracle's results;
- with RBF_FAULT=bounds the engine understates its partials capacity to the
  kernels, and the checks must report it (and the process survive).
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PATHS = r"""
import numpy as np, torch
import resident_brute_force_gb300 as rbf, workloads, oracle
from tests.parity import check_exact, check_float_topk
rbf.load_library()
assert rbf.lib_path().endswith("librbf_checks.so"), rbf.lib_path()

def clean(e):
    st = e.check_device_error()
    assert st == rbf.RBF_OK, rbf.status_string(st)

# single query: registers (D = 384) and shared-memory query (D = 96), fused and two-step merges
for n, d in ((20_000, 96), (20_011, 384)):
    c = workloads.dyadic_grid(n, d, seed=n)
    q = workloads.dyadic_grid(2, d, seed=n + 1)
    with rbf.Engine(n, d, 256) as e:
        e.upload_corpus_rowmajor(c)
        for k in (8, 100, 256):
            check_exact(*e.search_resident(q[0], k), *oracle.topk(c, q[0], k))
            dq = torch.from_numpy(q[1]).cuda()
            di = torch.empty(k, dtype=torch.int32, device="cuda"); ds = torch.empty(k, dtype=torch.float32, device="cuda")
            e.score_select_partials_dev(dq, k); e.merge_partial_topk_dev(k, di, ds)
            torch.cuda.synchronize()  # the engine's own stream
            check_exact(di.cpu().numpy(), ds.cpu().numpy(), *oracle.topk(c, q[1], k))
            with e.view() as v:
                check_exact(*v.search_resident(q[0], k), *oracle.topk(c, q[0], k))
        clean(e)

# cosine
c = workloads.unit_corpus(8000, 128, seed=5); q = workloads.unit_queries(1, 128, seed=6)[0]
with rbf.Engine(8000, 128, 32, flags=rbf.RBF_FLAG_COSINE) as e:
    e.upload_corpus_rowmajor(c)
    idx, sc = e.search_resident(q, 32)
    check_float_topk(idx, sc, oracle.scores_cosine(c, q), 32)
    clean(e)

# batched: bf16 and tf32, with and without the bound pre-pass, register and global-memory lists, two groups
for flags in (rbf.RBF_FLAG_BF16_CORPUS, rbf.RBF_FLAG_FP32_CORPUS):
    for n in (5000, 70_144):
        c = workloads.dyadic_grid(n, 64, seed=n + 7)
        qs = workloads.dyadic_grid(300, 64, seed=n + 8)
        with rbf.Engine(n, 64, 256, max_batch=300, flags=flags) as e:
            e.upload_corpus_rowmajor(c)
            for b, k in ((5, 8), (300, 32), (40, 100), (3, 256)):
                idx, sc = e.search_resident_batch(qs[:b], k)
                for j in range(0, b, 37):
                    check_exact(idx[j], sc[j], *oracle.topk(c, qs[j], k))
            clean(e)

# int32: register-load stage 1 + merge kernel, stream kernel with its last-CTA merge, sample pass, no-alloc
x = workloads.int32_uniform(400_000, seed=9)
dx = torch.from_numpy(x).cuda()
with rbf.Engine(16, 16, 256) as e:
    for n, k in ((5000, 20), (400_000, 20), (400_000, 100), (400_000, 256)):
        v, p = e.topk_int32(dx[:n], k)
        ov, op = oracle.topk_int32(x[:n], k)
        assert np.array_equal(v, ov) and np.array_equal(p, op), (n, k)
    clean(e)
dv = torch.empty(20, dtype=torch.int32, device="cuda"); dp = torch.empty(20, dtype=torch.int64, device="cuda")
assert rbf.topk_int32_noalloc(dx, 20, dv, dp) == rbf.RBF_OK
torch.cuda.synchronize()
ov, op = oracle.topk_int32(x, 20)
assert np.array_equal(dv.cpu().numpy(), ov) and np.array_equal(dp.cpu().numpy(), op)
print("checked paths clean")
"""

FIRES = r"""
import resident_brute_force_gb300 as rbf, workloads
rbf.load_library()
c = workloads.dyadic_grid(50_000, 64, seed=3)
with rbf.Engine(50_000, 64, 8) as e:
    e.upload_corpus_rowmajor(c)
    try:
        e.search_resident(c[1], 8)
        raise SystemExit("no bounds report")
    except rbf.RbfError as ex:
        assert ex.status == rbf.RBF_ERR_BOUNDS, ex
print("bounds reported")
"""


def _run(script, **env):
    from resident_brute_force_gb300 import _build
    lib = _build.build(checks=True)
    full_env = dict(os.environ, RBF_LIB=lib, PYTHONPATH=ROOT, **env)
    r = subprocess.run([sys.executable, "-c", script], cwd=ROOT, env=full_env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    return r.stdout


def test_checked_build_paths_run_clean():
    assert "checked paths clean" in _run(PATHS)


def test_checked_build_reports_out_of_bounds():
    assert "bounds reported" in _run(FIRES, RBF_FAULT="bounds")
