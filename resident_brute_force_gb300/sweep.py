"""The single-query sweep: N x D x K cells, one JSON line per cell.

    python -m resident_brute_force_gb300.sweep [--queries 200] [--n 10000,50000,...] [--d 384,768,1024] [--k 8,32,100]

Per cell (unit-norm Gaussian rows and queries, seeds 1 and 2): `queries` device
calls (`search_resident_dev`, CUDA events at call boundaries on the engine's
stream) and as many host calls (`search_resident`, host wall clock). Reports
p50/p99 of both, queries per second and the corpus read rate against the
measured HBM peak. A corpus smaller than twice the L2 stays in L2 between
calls; those cells say so ("l2_resident") rather than flushing.
"""
import argparse
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--queries", type=int, default=200)
    ap.add_argument("--n", default="10000,50000,100000,500000,1000000")
    ap.add_argument("--d", default="384,768,1024")
    ap.add_argument("--k", default="8,32,100")
    args = ap.parse_args(argv)
    import torch

    import resident_brute_force_gb300 as rbf
    import workloads
    from bench import hbm_peak, percentile

    ns = [int(x) for x in args.n.split(",")]
    ds = [int(x) for x in args.d.split(",")]
    ks = [int(x) for x in args.k.split(",")]
    hbm, hsrc = hbm_peak()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    for d in ds:
        full = workloads.unit_corpus(max(ns), d, seed=1)
        qs = workloads.unit_queries(args.queries, d, seed=2)
        dq = torch.from_numpy(qs).cuda()
        st = torch.cuda.Stream()
        eng = rbf.Engine(max(ns), d, max(ks), stream=st)
        for n in ns:
            eng.upload_corpus_rowmajor(full[:n])
            nbytes = n * d * 4
            for k in ks:
                di = torch.empty(k, dtype=torch.int32, device="cuda")
                dsc = torch.empty(k, dtype=torch.float32, device="cuda")
                with torch.cuda.stream(st):
                    for j in range(10):
                        eng.search_resident_dev(dq[j % args.queries], k, di, dsc)
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.queries + 1)]
                torch.cuda.synchronize()
                with torch.cuda.stream(st):
                    for j in range(args.queries):
                        ev[j].record(st)
                        eng.search_resident_dev(dq[j], k, di, dsc)
                    ev[args.queries].record(st)
                torch.cuda.synchronize()
                dev = [ev[j].elapsed_time(ev[j + 1]) * 1e-3 for j in range(args.queries)]
                host = []
                for j in range(args.queries):
                    t0 = time.perf_counter()
                    eng.search_resident(qs[j], k)
                    host.append(time.perf_counter() - t0)
                p50 = percentile(dev, 50)
                gbs = nbytes / statistics.mean(dev) / 1e9
                print(json.dumps({
                    "n": n, "d": d, "k": k, "queries": args.queries,
                    "p50_us": round(p50 * 1e6, 1), "p99_us": round(percentile(dev, 99) * 1e6, 1),
                    "qps": round(1.0 / statistics.mean(dev), 1), "gbs": round(gbs, 1),
                    "hbm_frac": round(gbs / hbm, 4), "hbm_peak_source": hsrc,
                    "e2e_p50_us": round(percentile(host, 50) * 1e6, 1),
                    "e2e_p99_us": round(percentile(host, 99) * 1e6, 1),
                    "l2_resident": nbytes < 2 * l2,
                }), flush=True)
        eng.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
