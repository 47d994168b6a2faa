"""Readers for the hand-derived text fixtures in tests/golden/ (each cites its source)."""
from __future__ import annotations

import os
from fractions import Fraction

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if line:
                yield line.split()


def e4m3_values():
    """[(code, Fraction or None for NaN, negative_zero_flag)]"""
    out = []
    for code, val in _lines("e4m3_ocp_values.txt"):
        c = int(code, 16)
        if val == "nan":
            out.append((c, None, False))
            continue
        neg_zero = val == "-0"
        if "*2^" in val:
            mant, exp = val.split("*2^")
            v = Fraction(int(mant)) * Fraction(2) ** int(exp)
        else:
            v = Fraction(val)
        out.append((c, v, neg_zero))
    return out


def bf16_cases():
    """[(hi, lo, expected_bits)] with hi/lo as Python floats."""
    out = []
    for hi, lo, bits in _lines("bf16_rne_cases.txt"):
        out.append((float.fromhex(hi) if "0x" in hi else float(hi),
                    float.fromhex(lo) if "0x" in lo else float(lo), int(bits, 16)))
    return out


def tiny_problem(name):
    """Dict of the key -> values of tiny_stacked.txt / tiny_dynamic.txt."""
    d = {}
    for parts in _lines(name):
        key, vals = parts[0], parts[1:]
        if key in ("A", "B", "out"):
            d[key] = [int(v, 16) for v in vals]
        elif key in ("scale_a", "scale_b"):
            d[key] = [float(v) for v in vals]
        elif key in ("m_sizes", "zsi"):
            d[key] = [int(v) for v in vals]
        else:
            d[key] = int(vals[0])
    return d
