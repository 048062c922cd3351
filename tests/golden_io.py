"""Readers for the text fixtures under tests/golden/ (no arithmetic of the method)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_kv(name):
    """key = rows separated by ';', values by spaces.  Returns dict of str -> list[list[str]]."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            out[key] = [r.split() for r in val.split(";")]
    return out


def as_array(rows, dtype):
    if dtype in (np.uint32,):
        return np.array([[int(v, 0) for v in r] for r in rows], dtype=np.uint64).astype(dtype)
    return np.array([[float(v) for v in r] for r in rows]).astype(dtype)


def read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split("|")])
    return rows
