"""Reader of the hand-worked fixtures under tests/golden/."""
import glob
import math
import os
from fractions import Fraction

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _value(tok: str) -> float:
    neg = tok.startswith("-")
    t = tok[1:] if neg else tok
    if t.startswith("ln(") and t.endswith(")"):
        v = math.log(float(Fraction(t[3:-1])))
    else:
        v = float(Fraction(t))
    return -v if neg else v


def load(path: str) -> dict:
    out = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, vals = line.split(":", 1)
            toks = vals.split()
            if key in ("op", "score_func"):
                out[key] = toks[0]
            elif key in ("K", "num_groups", "group_topk", "E"):
                out[key] = int(toks[0])
            elif key in ("scaling_factor", "coeff"):
                out[key] = _value(toks[0])
            elif "|" in vals:  # rows of a [T, ...] array, separated by "|"
                out[key] = np.array([[_value(t) for t in row.split()]
                                     for row in vals.split("|")], dtype=np.float64)
            else:
                out[key] = np.array([_value(t) for t in toks], dtype=np.float64)
    out.setdefault("num_groups", 0)
    out.setdefault("group_topk", 0)
    out.setdefault("scaling_factor", 1.0)
    out["name"] = os.path.basename(path)
    return out


def all_cases() -> list:
    return [load(p) for p in sorted(glob.glob(os.path.join(GOLDEN_DIR, "*.txt")))
            if not p.endswith("README.txt")]
