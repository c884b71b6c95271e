"""Pins from numbers the pages print."""
import json
import os

import numpy as np

import oracle.draft_attn_oracle as orc

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_window_drops_99_percent_at_1m():
    g = json.load(open(os.path.join(GOLD, "windowed_mtp_kv_drop_1m.json")))
    L = g["context"]
    for W, ns in g["window_cases"]:
        kept = orc.select_keys("window", L, W, ns)["loc"].size
        assert kept == W + ns
        dropped = 1.0 - kept / L
        assert round(dropped, 2) >= g["dropped_fraction_approx"] and dropped < 1.0
    # the working set is constant: the same count at every context above W + sinks
    for L2 in (131072, 262144, 524288, L):
        assert orc.select_keys("window", L2, 4096, 4)["loc"].size == 4100
    # and full attention reads everything
    assert orc.select_keys("full", L, 0, 0)["loc"].size == L
