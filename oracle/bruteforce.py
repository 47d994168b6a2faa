"""Exact rational brute force of the FP8 rowwise-scaled grouped GEMM, pure Python.

TEST INFRASTRUCTURE ONLY; for tiny inputs (a few hundred output elements).

It restates the definition from MSLK #471 "Back the FP8 rowwise grouped GEMM ops with
FlyDSL on ROCm" (commit introducing the rowwise scaling scheme; PR Summary table):
per group g and owned row r,
    out[r, n] = bf16_rne(scale_a[r] * scale_b[g, n] * sum_k A[r, k] * B[g, n, k])
in exact rational arithmetic (fractions.Fraction), independently of oracle.c: the
E4M3 decode, the sum, the scaling and the bf16 rounding are all written again here
with no floating-point step at all.  NaN codes are reported as None.
"""
from __future__ import annotations

from fractions import Fraction


def e4m3_value(code: int):
    """OCP OFP8 E4M3: bias 7, no infinities, NaN = S.1111.111, max 448."""
    code &= 0xFF
    negative = bool(code & 0x80)
    exp_field = (code >> 3) & 0xF
    mant = code & 0x7
    if exp_field == 0xF and mant == 0x7:
        return None
    if exp_field == 0:
        v = Fraction(mant, 8) * Fraction(2) ** (1 - 7)
    else:
        v = (1 + Fraction(mant, 8)) * Fraction(2) ** (exp_field - 7)
    return -v if negative else v


def float_exact(x: float) -> Fraction:
    return Fraction(x)  # exact for every finite binary64 (and so binary32) value


def bf16_bits_exact(x) -> int:
    """Round the exact rational x to bfloat16, nearest-even; return the bit pattern."""
    if x is None:
        return 0x7FC0
    sign = 0x8000 if x < 0 else 0
    a = -x if x < 0 else x
    if a == 0:
        return sign
    # smallest e with 2^(e+1) > a, i.e. e = floor(log2(a))
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    if e < -126:
        step_exp = -133
    else:
        step_exp = e - 7
    t = a / Fraction(2) ** step_exp
    q = t.numerator // t.denominator
    rem = t - q
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and q % 2 == 1):
        q += 1
    value = q * Fraction(2) ** step_exp
    # encode an exactly representable value
    if value >= Fraction(2) ** 128:
        return sign | 0x7F80
    if value < Fraction(2) ** -126:
        return sign | int(value / Fraction(2) ** -133)
    e2 = e
    if value >= Fraction(2) ** (e + 1):
        e2 = e + 1
    if e2 > 127:
        return sign | 0x7F80
    mant = int(value / Fraction(2) ** (e2 - 7)) - 128
    return sign | ((e2 + 127) << 7) | mant


def dot_exact(arow, brow):
    s = Fraction(0)
    for ca, cb in zip(arow, brow):
        va, vb = e4m3_value(int(ca)), e4m3_value(int(cb))
        if va is None or vb is None:
            return None
        s += va * vb
    return s


def element(arow, brow, sa: float, sb: float) -> int:
    s = dot_exact(arow, brow)
    if s is None:
        return 0x7FC0
    return bf16_bits_exact(float_exact(float(sa)) * float_exact(float(sb)) * s)


def stacked(A, B, scale_a, scale_b, m_sizes, total_M):
    """Nested lists / arrays in, dict {(row, n): bits} out for every owned element."""
    G = len(B)
    N = len(B[0]) if G else 0
    out = {}
    start = 0
    for g in range(G):
        m = int(m_sizes[g])
        m = max(0, min(m, total_M - start))
        for r in range(start, start + m):
            for n in range(N):
                out[(r, n)] = element(A[r], B[g][n], scale_a[r], scale_b[g][n])
        start += m
    return out


def dynamic(A, B, scale_a, scale_b, zsi, expected_m):
    G = len(B)
    N = len(B[0]) if G else 0
    out = {}
    for g in range(G):
        v = max(0, min(int(zsi[g]), expected_m))
        for r in range(expected_m):
            row = g * expected_m + r
            for n in range(N):
                if r < v:
                    out[(row, n)] = element(A[row], B[g][n], scale_a[row], scale_b[g][n])
                else:
                    out[(row, n)] = 0x0000
    return out


def offsets(A, B, scale_a, scale_b, offsets_incl, total_M):
    """Group g owns rows [offsets[g-1], offsets[g]) (offsets[-1] = 0): the row counts are
    the steps between successive inclusive offsets."""
    counts = [int(offsets_incl[g]) - (int(offsets_incl[g - 1]) if g else 0)
              for g in range(len(offsets_incl))]
    return stacked(A, B, scale_a, scale_b, counts, total_M)


def batched(A, B, scale_a, scale_b, M):
    G = len(B)
    return dynamic(A, B, scale_a, scale_b, [M] * G, M)


def _bounds(offsets_incl, total):
    """Group ranges from an int32 inclusive prefix: the steps between successive offsets
    (offsets[-1] = 0), each clamped into [0, total - start]."""
    out, start = [], 0
    for g in range(len(offsets_incl)):
        c = int(offsets_incl[g]) - (int(offsets_incl[g - 1]) if g else 0)
        c = max(0, min(c, total - start))
        out.append((start, start + c))
        start += c
    return out


def n_offsets(A, B, scale_a, scale_b, offsets_incl, total_N):
    """Ragged N: A[g][m] rows (G slabs of M), B[n] rows (total_N), scale_a[g][m],
    scale_b[n]; group g owns output columns [c_g, c_{g+1}); out {(m, n): bits}."""
    G = len(A)
    M = len(A[0]) if G else 0
    out = {}
    for g, (c0, c1) in enumerate(_bounds(offsets_incl, total_N)):
        for m in range(M):
            for n in range(c0, c1):
                out[(m, n)] = element(A[g][m], B[n], scale_a[g][m], scale_b[n])
    return out


def k_offsets(A, B, scale_a, scale_b, offsets_incl, total_K):
    """Ragged K: A[m] and B[n] rows of total_K codes, scale_a[g][m], scale_b[g][n]; group
    g contracts over k in [k_g, k_{g+1}); out {(g*M + m, n): bits}."""
    M = len(A)
    N = len(B)
    out = {}
    for g, (k0, k1) in enumerate(_bounds(offsets_incl, total_K)):
        for m in range(M):
            for n in range(N):
                out[(g * M + m, n)] = element(list(A[m])[k0:k1], list(B[n])[k0:k1],
                                              scale_a[g][m], scale_b[g][n])
    return out


def blockwise_element(arow, brow, sa_row, sb_blk, block=128) -> int:
    """Block scaling: sum over K blocks of scale_a[kb] * scale_b[kb] * (exact block sum),
    all in exact rationals, rounded once to bf16."""
    total = Fraction(0)
    for kb in range(len(arow) // block):
        s = dot_exact(list(arow)[kb * block:(kb + 1) * block],
                      list(brow)[kb * block:(kb + 1) * block])
        if s is None:
            return 0x7FC0
        total += float_exact(float(sa_row[kb])) * float_exact(float(sb_blk[kb])) * s
    return bf16_bits_exact(total)


def blockwise_dynamic(A, B, scale_a, scale_b, zsi, expected_m, cols=None, block=128):
    """Block-scaled dynamic layout (zsi None: batched, every slab row valid): dict
    (row, n) -> bf16 bits, padding rows +0.0.  ``cols``: the columns to compute (all by
    default)."""
    G = len(B)
    N = len(B[0]) if G else 0
    out = {}
    for g in range(G):
        v = expected_m if zsi is None else max(0, min(int(zsi[g]), expected_m))
        for r in range(expected_m):
            row = g * expected_m + r
            for n in (range(N) if cols is None else cols):
                if r < v:
                    out[(row, n)] = blockwise_element(A[row], B[g][n], scale_a[row],
                                                      scale_b[g][n // block], block)
                else:
                    out[(row, n)] = 0x0000
    return out
