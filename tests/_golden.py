"""Reader for the hand-derived fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, vals = line.partition(":")
            out[key.strip()] = [float(x) for x in vals.split()]
    out["shape"] = [int(x) for x in out["shape"]]
    return out


def f32(vals, shape):
    return np.asarray(vals, dtype=np.float32).reshape(shape)
