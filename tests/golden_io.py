"""Reader of the golden text fixtures under tests/golden/."""

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_fixture(window: int):
    path = os.path.join(GOLDEN, f"p1_fixture_bf16_w{window}.txt")
    lse, out = {}, {}
    with open(path) as f:
        for line in f:
            if line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "lse":
                lse[int(parts[1])] = np.array([float(x) for x in parts[2:]])
            elif parts[0] == "out":
                out[int(parts[1])] = np.array([float(x) for x in parts[2:]])
    return np.stack([lse[h] for h in sorted(lse)]), out
