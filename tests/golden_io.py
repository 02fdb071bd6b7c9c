"""Reader for the hand-computed fixtures in tests/golden/hand_products.txt."""
from __future__ import annotations

import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _num(tok: str) -> float:
    if tok.startswith("p2(") and tok.endswith(")"):
        return 2.0 ** int(tok[3:-1])
    return float(tok)


def _rows(text: str, conv):
    return [[conv(t) for t in row.split()] for row in text.split(";")]


def hand_products(path: str | None = None):
    path = path or os.path.join(GOLDEN_DIR, "hand_products.txt")
    cases, cur = [], None
    with open(path) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                name, dtype, M, N, K = rest.split()
                cur = {"name": name, "dtype": dtype, "M": int(M), "N": int(N), "K": int(K)}
                cases.append(cur)
            elif key in ("A", "B", "D"):
                cur[key] = np.array(_rows(rest, _num), dtype=np.float64)
            elif key == "bits":
                cur["bits"] = np.array(_rows(rest, lambda t: int(t, 16)), dtype=np.uint16)
            else:
                raise ValueError(f"bad golden line: {raw!r}")
    for c in cases:
        assert c["A"].shape == (c["M"], c["K"]), c["name"]
        assert c["B"].shape == (c["N"], c["K"]), c["name"]
        assert c["D"].shape == (c["M"], c["N"]), c["name"]
        assert c["bits"].shape == (c["M"], c["N"]), c["name"]
    return cases
