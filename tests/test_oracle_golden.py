"""The oracle still reproduces its recorded result on the tiny layer (regression guard)."""

import json
import os

from tests.golden.gen_golden import compute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_layer_oracle.json")


def test_tiny_layer_matches_recorded_oracle():
    with open(GOLDEN) as f:
        want = json.load(f)
    got = compute()
    for key in ("inputs", "packed", "qT", "sw", "xq", "sx", "acc", "y32", "ybf", "acc_00_01_10", "sx_0"):
        assert got[key] == want[key], key
    assert abs(got["rel_fro_vs_fp64"] - want["rel_fro_vs_fp64"]) < 1e-12
