"""The oracle against the hand-worked fixtures in tests/golden/."""
import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_tiny_inner_product():
    g = _load("tiny_ip.json")
    c = np.array(g["corpus"], dtype=np.float32)
    for case in g["cases"]:
        idx, sc = oracle.topk(c, np.array(case["query"], np.float32), case["k"])
        assert idx.tolist() == case["idx"]
        assert sc.tolist() == case["score"]


def test_tiny_int32():
    g = _load("tiny_i32.json")
    x = np.array(g["x"], dtype=np.int32)
    for case in g["cases"]:
        val, pos = oracle.topk_int32(x, case["k"])
        assert val.tolist() == case["val"]
        assert pos.tolist() == case["pos"]
