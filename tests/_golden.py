"""Reader for the small text fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#") or ":" not in line:
                continue
            key, vals = line.split(":", 1)
            out[key.strip()] = np.array([float(v) for v in vals.split()], dtype=np.float64)
    return out


def rows(name: str) -> list:
    """Whitespace-separated numeric rows (comment lines skipped)."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append([int(v) for v in line.split()])
    return out
