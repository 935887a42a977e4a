"""Parser for the hand-worked golden case files under tests/golden/.

Pure text parsing: no arithmetic of the method happens here.
"""
from __future__ import annotations

import os
from fractions import Fraction

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _expand(tokens):
    out = []
    for tok in tokens:
        if "*" in tok:
            v, c = tok.split("*")
            out.extend([v] * int(c))
        else:
            out.append(tok)
    return out


def read_cases(name):
    cases = []
    cur = None
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            if key == "case":
                cur = {"name": rest[0]}
            elif key == "end":
                cases.append(cur)
                cur = None
            else:
                cur.setdefault(key, []).extend(_expand(rest))
    return cases


def hex_bytes(vals):
    return [int(v, 16) for v in vals]


def fractions(vals):
    return [Fraction(v) for v in vals]
