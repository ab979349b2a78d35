"""Reader for the small text fixtures under tests/golden/ ("key: numbers" lines,
'#' comments; bf16_rne.txt is two columns per line)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _num(tok: str) -> float:
    return float(tok)  # accepts inf, -inf, -0.0


def load_kv(name: str) -> dict:
    """Return {key: [np.ndarray, ...]} (keys may repeat: one array per occurrence)."""
    out: dict = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, _, rest = line.partition(":")
            vals = np.array([_num(t) for t in rest.split()], dtype=np.float64)
            out.setdefault(key.strip(), []).append(vals)
    return out


def load_pairs(name: str):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                a, b = line.split()[:2]
                rows.append((_num(a), _num(b)))
    return rows
