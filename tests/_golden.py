"""Loader for the hand-worked fixtures under tests/golden/."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _num(x):
    if isinstance(x, list):
        return [_num(y) for y in x]
    if isinstance(x, str):
        return float(x)      # "-inf", "nan"
    return x


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def arr(x, dtype=np.float64):
    return np.asarray(_num(x), dtype=dtype)
