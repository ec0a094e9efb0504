"""Parser for the hand-built block fixtures under tests/golden/."""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_cases(fname: str, block_bytes: int, block_weights: int):
    """Yield (name, row bytes uint8, expected float64 values, cols)."""
    cases = []
    cur = None
    with open(os.path.join(GOLDEN, fname)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest.strip(), "bytes": [], "expect": []}
            elif key == "nblocks":
                cur["nblocks"] = int(rest)
            elif key == "bytes":
                cur["bytes"] += rest.split()
            elif key == "expect":
                cur["expect"] += rest.split()
            elif key == "end":
                nb = cur["nblocks"]
                row = np.zeros(nb * block_bytes, dtype=np.uint8)
                for tok in cur["bytes"]:
                    off, val = tok.split(":")
                    row[int(off)] = int(val, 16)
                cols = nb * block_weights
                exp = np.zeros(cols, dtype=np.float64)
                for tok in cur["expect"]:
                    rng, val = tok.split(":")
                    lo, _, hi = rng.partition("-")
                    hi = hi or lo
                    exp[int(lo):int(hi) + 1] = float(val)
                cases.append((cur["name"], row, exp, cols))
                cur = None
            else:
                raise ValueError(f"bad fixture line in {fname}: {line}")
    return cases
