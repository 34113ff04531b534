"""Reader for the small text fixtures in this folder.

Format: '#' starts a comment; ``key: v v v | v v`` gives a list of rows
separated by '|' (a single row when there is no '|').
"""
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def load(name):
    out = {}
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = line.split(":", 1)
            rows = [r.split() for r in val.split("|")]
            out[key.strip()] = rows if len(rows) > 1 else rows[0]
    return out


def as_array(rows, dtype):
    if rows and isinstance(rows[0], list):
        return np.array([[float(x) for x in r] for r in rows]).astype(dtype)
    return np.array([float(x) for x in rows]).astype(dtype)
