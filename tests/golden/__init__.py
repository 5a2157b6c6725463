"""Loader for the small text fixtures in this folder (``key = values`` lines, ``#`` comments)."""
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def _num(tok: str) -> float:
    neg = tok.startswith("-")
    t = tok[1:] if neg else tok
    if t.startswith("ln"):
        v = math.log(float(t[2:]))
    elif t.startswith("0x"):
        v = float(int(t, 16))
    elif "/" in t:
        a, b = t.split("/")
        v = float(a) / float(b)
    else:
        v = float(t)
    return -v if neg else v


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, vals = line.split("=", 1)
            out[key.strip()] = [_num(t) for t in vals.split()]
    return out
