"""bench.py's host-side bookkeeping on CPU: the clock record of each timed
region and the configuration the two arms report."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_clock_regions_take_only_their_own_samples():
    s = bench.ClockSampler(0)
    s.source = "test"
    s.max_sm = 2070.0
    # (time, SM MHz, reasons, watts)
    s.samples = [(0.5, 900.0, set(), 100.0), (1.1, 2070.0, set(), 900.0), (1.2, 2055.0, {"sw_power_cap"}, 1300.0),
                 (1.3, 2070.0, set(), 950.0), (2.5, 1980.0, {"hw_slowdown"}, 800.0), (3.5, 300.0, set(), 90.0)]
    s.regions = [("headline.k8", 1.0, 1.25), ("headline.k32", 1.25, 1.4), ("batched.k32", 2.0, 3.0)]
    rep = s.report("headline.")
    assert rep["samples"] == 3 and rep["sm_mhz"] == 2070.0 and rep["sm_max_mhz"] == 2070.0
    assert rep["reasons"] == ["sw_power_cap"] and rep["rejectable"] is False
    regs = rep["regions"]
    assert regs["headline.k8"]["samples"] == 2 and regs["headline.k8"]["sm_mhz"] == (2070.0 + 2055.0) / 2
    assert regs["headline.k32"]["samples"] == 1
    assert regs["batched.k32"]["reasons"] == ["hw_slowdown"]


def test_clock_record_without_a_source():
    s = bench.ClockSampler(0)
    rep = s.report("headline.")
    assert rep["samples"] == 0 and rep["sm_mhz"] is None and rep["reasons"]


def test_both_arms_report_one_configuration():
    args = bench.parse(["--steps", "3"])
    assert bench.headline_config(args, 1) == {
        "workload": bench.WORKLOAD, "n": 1_000_000, "d": 1024, "k": 8, "queries": 1000,
        "parallelism": "single GPU", "l2": "inputs larger than L2 (4.1 GB corpus), no flush"}


def test_result_block_bytes():
    # [error word | pad] then K int32 indices (padded to 16 bytes) then K scores.
    assert bench.result_d2h_bytes(8) == 16 + 32 + 32
    assert bench.result_d2h_bytes(3) == 16 + 16 + 12
    assert bench.result_d2h_bytes(20, 8) == 16 + 80 + 160
