"""The oracle still reproduces its locked table (tests/golden/oracle_lock.json).

A regression lock, not a pin: the table was written by
tests/golden/make_golden.py, which calls only the oracle on seeded inputs.
"""
import json
import os
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))
from make_golden import lock_inputs  # noqa: E402

with open(os.path.join(HERE, "golden", "oracle_lock.json")) as f:
    CASES = json.load(f)["cases"]


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_oracle_matches_lock(oracle_mod, case):
    x, y = lock_inputs(case["inputs"])
    assert list(x.shape) == case["shape"]
    if case["kind"] == "pyramid":
        means, maps = oracle_mod.ssim2d_pyramid(x, y, case["padding"], case["octaves"],
                                                want_maps=True)
        np.testing.assert_allclose(means.reshape(-1), case["means"], rtol=1e-12, atol=0)
        for m, pick in zip(maps, case["maps"]):
            np.testing.assert_allclose(m.reshape(-1)[pick["idx"]], pick["values"], rtol=1e-12,
                                       atol=0)
        return
    pad, dL = case["padding"], case["dL"]
    if case["kind"] == "2d":
        mean, smap = oracle_mod.ssim2d(x, y, pad, want_map=True)
        g1, g2 = oracle_mod.ssim2d_grad(x, y, dL, pad)
        np.testing.assert_allclose(smap.reshape(-1)[case["map_idx"]], case["map"],
                                   rtol=1e-12, atol=0)
    else:
        mean = oracle_mod.ssim3d(x, y, pad)
        g1, g2 = oracle_mod.ssim3d_grad(x, y, dL, pad)
    np.testing.assert_allclose(mean, case["mean"], rtol=1e-12, atol=0)
    scale = max(np.max(np.abs(case["grad1"])), 1e-30)
    np.testing.assert_allclose(g1.reshape(-1)[case["grad_idx"]], case["grad1"],
                               rtol=0, atol=1e-12 * scale)
    np.testing.assert_allclose(g2.reshape(-1)[case["grad_idx"]], case["grad2"],
                               rtol=0, atol=1e-12 * scale)
