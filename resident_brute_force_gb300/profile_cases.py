"""Small, L2-exceeding cases of each kernel for profiler captures.

    python -m resident_brute_force_gb300.profile_cases single   # scoring (+ merge kernel), 100k x 1024, K=8
    python -m resident_brute_force_gb300.profile_cases batch    # batched, 256 queries x 200k x 768, K=32
    python -m resident_brute_force_gb300.profile_cases batch_full  # 256 x 1M x 768, K=8/32/100 (launch lists)
    python -m resident_brute_force_gb300.profile_cases int32    # int32 top-K, 5e7 values, K=20

Each case holds a few hundred MB on the device and makes a handful of launches,
so a full-set capture of one launch ends in about a minute.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(part: str) -> None:
    import torch

    import resident_brute_force_gb300 as rbf
    import workloads

    if part == "single":
        n, d = 100_000, 1024
        c = workloads.unit_corpus(n, d, seed=1)
        qs = workloads.unit_queries(4, d, seed=2)
        e = rbf.Engine(n, d, 256)
        e.upload_corpus_rowmajor(c)
        dq = torch.from_numpy(qs).cuda()
        di = torch.empty(256, dtype=torch.int32, device="cuda")
        ds = torch.empty(256, dtype=torch.float32, device="cuda")
        for j in range(4):
            e.search_resident_dev(dq[j], 8, di, ds)  # one launch each (merge in the last CTA)
        for j in range(3):
            e.score_select_partials_dev(dq[j], 8)  # the two-step calls: the merge kernel
            e.merge_partial_topk_dev(8, di, ds)
    elif part == "batch":
        n, d, b = 200_000, 768, 256
        c = workloads.unit_corpus(n, d, seed=1)
        qs = workloads.unit_queries(b, d, seed=2)
        e = rbf.Engine(n, d, 32, max_batch=b, flags=rbf.RBF_FLAG_BF16_CORPUS)
        e.upload_corpus_rowmajor(c)
        dq = torch.from_numpy(qs).cuda()
        di = torch.empty((b, 32), dtype=torch.int32, device="cuda")
        ds = torch.empty((b, 32), dtype=torch.float32, device="cuda")
        for _ in range(2):
            e.search_resident_batch_dev(dq, 32, di, ds)
    elif part == "batch_full":
        # The full batched workload (about 4.6 GB on the device): for one-pass
        # launch lists only, never for multi-pass captures.
        n, d, b = 1_000_000, 768, 256
        c = workloads.unit_corpus(n, d, seed=1)
        qs = workloads.unit_queries(b, d, seed=2)
        e = rbf.Engine(n, d, 100, max_batch=b, flags=rbf.RBF_FLAG_BF16_CORPUS)
        e.upload_corpus_rowmajor(c)
        dq = torch.from_numpy(qs).cuda()
        for k in (8, 32, 100):
            di = torch.empty((b, k), dtype=torch.int32, device="cuda")
            ds = torch.empty((b, k), dtype=torch.float32, device="cuda")
            for _ in range(3):
                e.search_resident_batch_dev(dq, k, di, ds)
    elif part == "int32":
        x = torch.from_numpy(workloads.int32_uniform(50_000_000, seed=1)).cuda()
        e = rbf.Engine(16, 16, 64)
        dv = torch.empty(64, dtype=torch.int32, device="cuda")
        dp = torch.empty(64, dtype=torch.int64, device="cuda")
        for _ in range(2):
            e.topk_int32_dev(x, 20, dv, dp)
    else:
        raise SystemExit(f"unknown case {part!r}: single | batch | batch_full | int32")
    torch.cuda.synchronize()
    print("ok", part)


if __name__ == "__main__":
    main(sys.argv[1] if len(sys.argv) > 1 else "single")
