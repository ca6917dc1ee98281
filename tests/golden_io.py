"""Readers for the text fixtures under tests/golden/."""
from __future__ import annotations

import math
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _num(tok: str) -> float:
    t = tok.strip()
    if t in ("-inf", "inf", "nan"):
        return float(t)
    return float(t)


def _matrix(s: str):
    return [[_num(x) for x in row.split()] for row in s.split(";")]


def hand_examples():
    """Parse hand_examples.txt into a list of dicts."""
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "hand_examples.txt")) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("[") and line.endswith("]"):
                cur = {"name": line[1:-1]}
                cases.append(cur)
                continue
            key, val = (x.strip() for x in line.split("=", 1))
            cur[key] = val
    out = []
    for c in cases:
        B, H, Sq, Sk, d = (int(x) for x in c["shape"].split())
        out.append(dict(
            name=c["name"], cite=c["cite"], B=B, H=H, Sq=Sq, Sk=Sk, d=d,
            causal=bool(int(c["causal"])), scale=float(c["scale"]),
            q=_matrix(c["q"]), k=_matrix(c["k"]), v=_matrix(c["v"]),
            o=_matrix(c["o"]), lse=[_num(x) for x in c["lse"].split(";")],
            tol=float(c["tol"])))
    return out


def pages_numbers():
    rows = {}
    with open(os.path.join(GOLDEN, "pages_numbers.txt")) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            name, inputs, value, rounding, cite = (x.strip() for x in line.split("|"))
            kv = dict(tok.split("=") for tok in inputs.split())
            rows[name] = dict(inputs={k: float(v) for k, v in kv.items()},
                              value=float(value.split()[0]), rounding=rounding, cite=cite)
    return rows


def isclose_or_both_inf(a: float, b: float, tol: float) -> bool:
    if math.isinf(a) or math.isinf(b):
        return a == b
    return abs(a - b) <= tol
