"""Writes the oracle lock tables under tests/golden/.

It calls only the CPU oracle and the seeded input generators.  The tables lock
the oracle's outputs on small seeded inputs so that a later change to its
arithmetic shows up as a failing test (the practice of locking a validated
pipeline against a known-good table, from the zenmetrics ssim2-gpu handoff,
"Resume here" / validation plan).  They are not an independent pin: the pins
live in tests/test_oracle_pins.py.

Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from workloads import make_inputs, uniform_pair  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_lock.json")


def case_2d(name, x, y, padding, dL, n_idx=24, seed=0):
    mean, smap = oracle.ssim2d(x, y, padding, want_map=True)
    g1, g2 = oracle.ssim2d_grad(x, y, dL, padding)
    rng = np.random.default_rng(seed)
    idx = np.sort(rng.choice(x.size, n_idx, replace=False))
    midx = np.sort(rng.choice(smap.size, n_idx, replace=False))
    return {
        "name": name, "kind": "2d", "shape": list(x.shape), "padding": padding,
        "inputs": name, "dL": [float(v) for v in dL],
        "mean": [float(v) for v in mean],
        "map_idx": midx.tolist(), "map": smap.reshape(-1)[midx].tolist(),
        "grad_idx": idx.tolist(), "grad1": g1.reshape(-1)[idx].tolist(),
        "grad2": g2.reshape(-1)[idx].tolist(),
    }


def case_3d(name, x, y, padding, dL, n_idx=16, seed=0):
    mean = oracle.ssim3d(x, y, padding)
    g1, g2 = oracle.ssim3d_grad(x, y, dL, padding)
    idx = np.sort(np.random.default_rng(seed).choice(x.size, n_idx, replace=False))
    return {
        "name": name, "kind": "3d", "shape": list(x.shape), "padding": padding,
        "inputs": name, "dL": [float(v) for v in dL],
        "mean": [float(v) for v in mean],
        "grad_idx": idx.tolist(), "grad1": g1.reshape(-1)[idx].tolist(),
        "grad2": g2.reshape(-1)[idx].tolist(),
    }


def case_pyramid(name, x, y, padding, octaves, n_idx=12, seed=0):
    means, maps = oracle.ssim2d_pyramid(x, y, padding, octaves, want_maps=True)
    rng = np.random.default_rng(seed)
    picks = []
    for o in range(octaves):
        idx = np.sort(rng.choice(maps[o].size, n_idx, replace=False))
        picks.append({"idx": idx.tolist(), "values": maps[o].reshape(-1)[idx].tolist()})
    return {
        "name": name, "kind": "pyramid", "shape": list(x.shape), "padding": padding,
        "inputs": name, "octaves": octaves, "means": means.reshape(-1).tolist(), "maps": picks,
    }


def lock_inputs(name):
    """Inputs of each locked case, regenerated from their seeds."""
    if name == "tiny64_valid":
        return make_inputs("tiny64_valid")
    if name == "uniform_2x2x23x29_same":
        return uniform_pair((2, 2, 23, 29), 77, std=0.1)
    if name == "uniform_1x1x12x14x13_valid":
        return uniform_pair((1, 1, 12, 14, 13), 78, std=0.05)
    if name == "uniform_1x2x9x8x10_same":
        return uniform_pair((1, 2, 9, 8, 10), 79, std=0.05)
    if name == "uniform_2x2x45x50_pyramid":
        return uniform_pair((2, 2, 45, 50), 80, std=0.07)
    if name == "uniform_1x1x13x9_pyramid":
        return uniform_pair((1, 1, 13, 9), 81, std=0.07)
    raise KeyError(name)


def main():
    cases = []
    x, y = lock_inputs("tiny64_valid")
    cases.append(case_2d("tiny64_valid", x, y, "valid", [-1.0]))
    x, y = lock_inputs("uniform_2x2x23x29_same")
    cases.append(case_2d("uniform_2x2x23x29_same", x, y, "same", [-1.0, 0.5]))
    x, y = lock_inputs("uniform_1x1x12x14x13_valid")
    cases.append(case_3d("uniform_1x1x12x14x13_valid", x, y, "valid", [-1.0]))
    x, y = lock_inputs("uniform_1x2x9x8x10_same")
    cases.append(case_3d("uniform_1x2x9x8x10_same", x, y, "same", [-1.0]))
    x, y = lock_inputs("uniform_2x2x45x50_pyramid")
    cases.append(case_pyramid("uniform_2x2x45x50_pyramid", x, y, "valid", 3))
    x, y = lock_inputs("uniform_1x1x13x9_pyramid")
    cases.append(case_pyramid("uniform_1x1x13x9_pyramid", x, y, "same", 4))
    with open(OUT, "w") as f:
        json.dump({"generator": "tests/golden/make_golden.py", "cases": cases}, f, indent=1)
    print("wrote", OUT)


if __name__ == "__main__":
    main()
