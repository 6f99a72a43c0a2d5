"""Reader for the worked-example fixtures in tests/golden/.

Each fixture is a small text file: ``#`` comment lines (the description and the
page it comes from), then blocks ``X r c`` / ``W r c`` / ``bias n`` / ``Y r c``
followed by their rows, a ``layout NK|KN`` line and optional extra keys.
"""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    path = os.path.join(GOLDEN, name)
    lines = [ln.strip() for ln in open(path, encoding="utf-8")]
    lines = [ln for ln in lines if ln and not ln.startswith("#")]
    out, i = {"extra": {}}, 0
    while i < len(lines):
        head = lines[i].split()
        key = head[0]
        if key == "layout":
            out["layout"] = {"NK": 0, "KN": 1}[head[1]]
            i += 1
        elif key in ("X", "W", "Y"):
            r, c = int(head[1]), int(head[2])
            rows = [[float(v) for v in lines[i + 1 + j].split()] for j in range(r)]
            out[key] = np.array(rows, dtype=np.float64).reshape(r, c)
            i += 1 + r
        elif key in ("bias", "partials"):
            n = int(head[1])
            out[key] = np.array([float(v) for v in lines[i + 1].split()], dtype=np.float64)
            assert out[key].size == n
            i += 2
        else:
            out["extra"].setdefault(key, []).append(head[1:])
            i += 1
    return out


# Fixtures that are not an X · Wᵀ = Y worked example (read by their own tests).
NOT_PRODUCTS = ("bf16_values.txt", "router_hilo.txt")


def names():
    """The worked-example fixtures with X, W and Y blocks."""
    return sorted(f for f in os.listdir(GOLDEN) if f.endswith(".txt") and f not in NOT_PRODUCTS)
