"""Input builders for the golden fixtures (no method arithmetic: they only
place the fixture's chosen values into q / k / v arrays)."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def detector_2tile_inputs(fx=None):
    """q [1, 128, 1, 64], k, v as float32 for tests/golden/detector_2tile.json."""
    fx = fx or load("detector_2tile.json")
    d, n = fx["head_dim"], fx["seqlen"]
    q = np.zeros((1, n, 1, d), np.float32)
    k = np.zeros((1, n, 1, d), np.float32)
    for r in range(n):
        q[0, r, 0, (r % 64) // 16] = 8.0
    for s in range(4):
        spec = fx["logits"][f"strip{s}"]
        for t in range(2):
            tspec = spec[f"tile{t}"]
            for c in range(64 * t, 64 * t + 64):
                val = tspec.get(f"key{c}", tspec["default"])
                k[0, c, 0, s] = val
    rng = np.random.default_rng(7)
    v = rng.standard_normal((1, n, 1, d)).astype(np.float32)
    return q, k, v


def chunk32_inputs():
    """Inputs of chunk32_rounding.json: q, k, v float64 [1, 2, 1, 64]."""
    d = 64
    q = np.ones((1, 2, 1, d))
    k = np.zeros((1, 2, 1, d))
    k[0, 0, 0, :17] = 2.0
    k[0, 0, 0, 32:34] = 1.0
    v = np.zeros((1, 2, 1, d))
    v[0, 0, 0, 0] = 1.0
    v[0, 1, 0, 1] = 1.0
    return q, k, v
