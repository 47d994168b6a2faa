"""Pins that tie the CPU oracle to facts outside itself.

Each pin is a function ``pin(orc)`` that raises AssertionError when the oracle build
``orc`` disagrees with something the format definitions, the mathematics or the
method's definition fix:

* library routines: torch's E4M3 decode and its binary32 -> bf16 round-to-nearest-even;
* hand-derived fixtures in tests/golden/ (OCP E4M3 values, bf16 rounding cases, and two
  tiny problems computed by hand);
* closed forms: K = 1, all-ones codes, B = identity, constant single-signed groups;
* an exact-rational brute force (oracle/bruteforce.py), written independently;
* invariants: exact K sum in any order and in integers, rowwise scales factoring out,
  empty groups and padding rows, agreement of the stacked and dynamic layouts.

The same battery runs against deliberately broken builds of the oracle (mutants) to
show that every planted mistake fails at least one pin.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import torch

from oracle import bruteforce as bf
import golden_io


def _torch_decode_table() -> np.ndarray:
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _rng(seed):
    return np.random.default_rng(seed)


def _random_codes(rng, shape, nan=False):
    c = rng.integers(0, 256, size=shape, dtype=np.int64)
    if not nan:
        c = np.where((c & 0x7F) == 0x7F, c ^ 1, c)
    return c.astype(np.uint8)


def _random_scales(rng, n):
    return np.exp(rng.normal(0.0, 3.0, size=n)).astype(np.float32) * \
        np.where(rng.random(n) < 0.2, -1.0, 1.0).astype(np.float32)


# ---------------------------------------------------------------------------------
# E4M3 decode
# ---------------------------------------------------------------------------------
def pin_decode_vs_torch(orc):
    mine = orc.decode_table()
    ref = _torch_decode_table()
    assert np.array_equal(np.isnan(mine), np.isnan(ref)), "NaN codes differ"
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok]), "decoded values differ from torch"
    assert np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok])), "zero signs differ"


def pin_decode_golden(orc):
    for code, val, neg_zero in golden_io.e4m3_values():
        got = orc.e4m3_to_double(code)
        if val is None:
            assert np.isnan(got), f"code {code:#04x} should be NaN"
        else:
            assert Fraction(got) == val, f"code {code:#04x}: {got} != {val}"
            if neg_zero:
                assert np.signbit(got), f"code {code:#04x} should be -0"


# ---------------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------------
def pin_bf16_golden(orc):
    for hi, lo, bits in golden_io.bf16_cases():
        got = orc.bf16_round(hi, lo)
        assert got == bits, f"bf16({hi!r} + {lo!r}) = {got:#06x}, expected {bits:#06x}"


def pin_bf16_vs_torch(orc, n=10_000_000, seed=11):
    """A 10^7-value sweep of binary32 (a quarter on exact bf16 midpoints, a quarter next to
    them, an eighth subnormal): the oracle's rounding equals torch's fp32 -> bf16 RNE."""
    rng = _rng(seed)
    bits = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
    # force a quarter of the sample onto exact bf16 midpoints, a quarter near them
    bits[: n // 4] = (bits[: n // 4] & 0xFFFF0000) | 0x8000
    bits[n // 4: n // 2] = (bits[n // 4: n // 2] & 0xFFFF0000) | \
        (0x8000 + rng.integers(-2, 3, size=n // 4)).astype(np.uint32)
    # subnormals
    bits[n // 2: n // 2 + n // 8] &= 0x807FFFFF
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy()
    ref = ref.astype(np.uint16)
    got = orc.bf16_round_array(f.astype(np.float64))
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (f"{bad.size} mismatches, first: {f[bad[0]]!r} "
                           f"got {got[bad[0]]:#06x} torch {ref[bad[0]]:#06x}")


# ---------------------------------------------------------------------------------
# the K sum
# ---------------------------------------------------------------------------------
def pin_dot_exact(orc, seed=5):
    """The fp64 K sum is exact: equal to integer arithmetic, to the reversed order and
    to a float64 matmul of torch-decoded operands."""
    rng = _rng(seed)
    tab = _torch_decode_table()
    for K in (1, 2, 3, 31, 128, 1000, 4096, 16384):
        a = _random_codes(rng, K)
        b = _random_codes(rng, K)
        if K == 16384:  # near the exactness limit: all codes at +-448
            a = np.full(K, 0x7E, np.uint8)
            b = np.where(rng.random(K) < 0.5, 0x7E, 0xFE).astype(np.uint8)
        s = orc.dot(a, b)
        ia = (tab[a] * 512).astype(np.int64)
        ib = (tab[b] * 512).astype(np.int64)
        exact_int = int(np.dot(ia, ib))
        assert orc.dot_int(a, b) == exact_int, f"K={K}: integer paths differ"
        assert Fraction(s) == Fraction(exact_int, 2 ** 18), f"K={K}: fp64 sum not exact"
        assert orc.dot(a[::-1].copy(), b[::-1].copy()) == s, f"K={K}: order dependent"
        m = torch.from_numpy(tab[a][None, :]) @ torch.from_numpy(tab[b][:, None])
        assert float(m.item()) == s, f"K={K}: differs from float64 matmul"


# ---------------------------------------------------------------------------------
# closed forms on small problems
# ---------------------------------------------------------------------------------
def pin_closed_form_k1(orc, seed=7):
    rng = _rng(seed)
    tab = _torch_decode_table()
    G, N = 3, 8
    m = np.array([2, 0, 3], np.int64)
    M = int(m.sum())
    A = _random_codes(rng, (M, 1))
    B = _random_codes(rng, (G, N, 1))
    sa = _random_scales(rng, M)
    sb = _random_scales(rng, G * N).reshape(G, N)
    out, _ = orc.stacked(A, B, sa, sb, m)
    grp = np.repeat(np.arange(G), m)
    for r in range(M):
        g = grp[r]
        for n in range(N):
            x = Fraction(float(sa[r])) * Fraction(float(sb[g, n])) * \
                Fraction(tab[A[r, 0]]) * Fraction(tab[B[g, n, 0]])
            assert out[r, n] == bf.bf16_bits_exact(x), f"K=1 mismatch at ({r},{n})"


def pin_closed_form_all_ones(orc):
    """A = B = 1.0 (code 0x38): out = sa * sb * K exactly, for power-of-two scales."""
    for K in (1, 7, 128, 200, 255, 256):
        G, N = 2, 8
        m = np.array([3, 2], np.int64)
        A = np.full((5, K), 0x38, np.uint8)
        B = np.full((G, N, K), 0x38, np.uint8)
        sa = np.array([1, 2, 0.5, 2 ** -10, 2 ** 20], np.float32)
        sb = np.array([[2.0 ** (j - 4) for j in range(N)], [0.25] * N], np.float32)
        out, _ = orc.stacked(A, B, sa, sb, m)
        grp = [0, 0, 0, 1, 1]
        for r in range(5):
            exp = torch.tensor(float(sa[r]) * sb[grp[r]].astype(np.float64) * K,
                               dtype=torch.float32).to(torch.bfloat16).view(torch.int16)
            assert np.array_equal(out[r], exp.numpy().astype(np.uint16)), f"K={K} row {r}"


def pin_closed_form_identity(orc, seed=3):
    """B = I (N = K, B[g, n, n] = 1): out[r, n] = bf16(sa * sb * A[r, n])."""
    rng = _rng(seed)
    K = 32
    G = 2
    m = np.array([4, 5], np.int64)
    A = _random_codes(rng, (9, K))
    B = np.zeros((G, K, K), np.uint8)
    for g in range(G):
        np.fill_diagonal(B[g], 0x38)
    sa = np.ones(9, np.float32)
    sa[4:] = 2.0 ** -3
    sb = np.ones((G, K), np.float32)
    sb[1] = 2.0 ** 5
    out, _ = orc.stacked(A, B, sa, sb, m)
    vals = torch.from_numpy(A.copy()).view(torch.float8_e4m3fn).to(torch.float32)
    vals = vals * torch.from_numpy(sa)[:, None]
    vals[4:] *= 2.0 ** 5
    exp = vals.to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    # code 0x80 (-0) times 1 plus +0 terms is the exact number 0, encoded +0.0
    exp[exp == 0x8000] = 0
    assert np.array_equal(out, exp), "B = I does not reproduce A"


def pin_coherent_groups(orc):
    """Constant, single-signed data per group (alternating groups): every element is
    the closed form sa * sb * K * a_g * b_g, so a row assigned to the wrong group or a
    read past a group's end shows up far outside rounding."""
    tab = _torch_decode_table()
    G, N, K = 4, 8, 96
    m = np.array([5, 1, 0, 7], np.int64)
    codes_a = [0x38, 0x44, 0x30, 0x40]
    codes_b = [0x40, 0xB8, 0x48, 0x38]
    A = np.concatenate([np.full((int(m[g]), K), codes_a[g], np.uint8) for g in range(G)])
    B = np.stack([np.full((N, K), codes_b[g], np.uint8) for g in range(G)])
    sa = np.ones(A.shape[0], np.float32)
    sb = np.ones((G, N), np.float32)
    out, _ = orc.stacked(A, B, sa, sb, m)
    r = 0
    for g in range(G):
        v = K * tab[codes_a[g]] * tab[codes_b[g]]
        exp = torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).view(torch.int16)
        for _ in range(int(m[g])):
            assert np.all(out[r] == np.uint16(exp.item() & 0xFFFF)), f"group {g} row {r}"
            r += 1


def pin_golden_tiny(orc):
    d = golden_io.tiny_problem("tiny_stacked.txt")
    G, N, K = d["G"], d["N"], d["K"]
    A = np.array(d["A"], np.uint8).reshape(-1, K)
    B = np.array(d["B"], np.uint8).reshape(G, N, K)
    out, _ = orc.stacked(A, B, np.array(d["scale_a"], np.float32),
                         np.array(d["scale_b"], np.float32).reshape(G, N), d["m_sizes"])
    assert out.ravel().tolist() == d["out"], f"tiny_stacked: {out.ravel()}"
    d = golden_io.tiny_problem("tiny_dynamic.txt")
    G, E, N, K = d["G"], d["E"], d["N"], d["K"]
    A = np.array(d["A"], np.uint8).reshape(-1, K)
    B = np.array(d["B"], np.uint8).reshape(G, N, K)
    out = orc.dynamic(A, B, np.array(d["scale_a"], np.float32),
                      np.array(d["scale_b"], np.float32).reshape(G, N), d["zsi"], E)
    assert out.ravel().tolist() == d["out"], f"tiny_dynamic: {out.ravel()}"


# ---------------------------------------------------------------------------------
# brute force on random tiny problems
# ---------------------------------------------------------------------------------
def _tiny_stacked_case(rng, nan=False):
    G = int(rng.integers(1, 5))
    N = int(rng.integers(1, 9))
    K = int(rng.choice([0, 1, 2, 5, 16, 33, 64]))
    m = rng.integers(0, 4, size=G)
    m[rng.random(G) < 0.3] = 0
    total = int(m.sum()) + int(rng.integers(0, 3))
    A = _random_codes(rng, (total, K), nan=nan)
    B = _random_codes(rng, (G, N, K), nan=nan)
    sa = _random_scales(rng, total)
    sb = _random_scales(rng, G * N).reshape(G, N)
    return A, B, sa, sb, m.astype(np.int64), total


def pin_bruteforce_stacked(orc, cases=40, seed=17):
    rng = _rng(seed)
    for i in range(cases):
        A, B, sa, sb, m, total = _tiny_stacked_case(rng, nan=(i % 10 == 9))
        poison = np.full((total, B.shape[1]), 0xDEAD, np.uint16)
        out, _ = orc.stacked(A, B, sa, sb, m, total_M=total, out=poison)
        ref = bf.stacked(A.tolist(), B.tolist(), sa.tolist(), sb.tolist(), m.tolist(), total)
        owned = np.zeros_like(out, dtype=bool)
        for (r, n), bits in ref.items():
            owned[r, n] = True
            got = int(out[r, n])
            if bits == 0x7FC0:
                assert (got & 0x7F80) == 0x7F80 and (got & 0x7F), f"case {i}: NaN expected"
            elif bits == 0x0000:
                # an exactly-zero product has no sign of its own: +0 and -0 both pass
                assert got in (0x0000, 0x8000), f"case {i} ({r},{n}): {got:#06x} != 0"
            else:
                assert got == bits, f"case {i} ({r},{n}): {got:#06x} != {bits:#06x}"
        assert np.all(out[~owned] == 0xDEAD), f"case {i}: unowned rows written"


def pin_bruteforce_dynamic(orc, cases=30, seed=19):
    rng = _rng(seed)
    for i in range(cases):
        G = int(rng.integers(1, 4))
        E = int(rng.integers(1, 6))
        N = int(rng.integers(1, 7))
        K = int(rng.choice([0, 1, 3, 16, 40]))
        zsi = rng.integers(-2, E + 3, size=G).astype(np.int64)
        A = _random_codes(rng, (G * E, K))
        B = _random_codes(rng, (G, N, K))
        sa = _random_scales(rng, G * E)
        sb = _random_scales(rng, G * N).reshape(G, N)
        out = orc.dynamic(A, B, sa, sb, zsi, E)
        ref = bf.dynamic(A.tolist(), B.tolist(), sa.tolist(), sb.tolist(), zsi.tolist(), E)
        for (r, n), bits in ref.items():
            got = int(out[r, n])
            if bits == 0x0000 and (r % E) < max(0, min(int(zsi[r // E]), E)):
                # computed exact zero: either sign passes (padding rows stay strict +0)
                assert got in (0x0000, 0x8000), f"case {i} ({r},{n}): {got:#06x} != 0"
            else:
                assert got == bits, f"case {i} ({r},{n}): {got:#06x} != {bits:#06x}"


# ---------------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------------
def pin_scale_factoring(orc, seed=23):
    """Power-of-two rowwise scales shift the result exactly: out(2^a, 2^b) equals
    2^(a+b) * out(1, 1) bit for bit, away from bf16 overflow and underflow."""
    rng = _rng(seed)
    G, N, K = 3, 8, 64
    m = np.array([3, 4, 2], np.int64)
    M = 9
    A = _random_codes(rng, (M, K))
    B = _random_codes(rng, (G, N, K))
    base, _ = orc.stacked(A, B, np.ones(M, np.float32), np.ones((G, N), np.float32), m)
    ea = rng.integers(-20, 21, size=M)
    eb = rng.integers(-20, 21, size=(G, N))
    sa = np.ldexp(np.ones(M), ea).astype(np.float32)
    sb = np.ldexp(np.ones((G, N)), eb).astype(np.float32)
    out, _ = orc.stacked(A, B, sa, sb, m)
    grp = np.repeat(np.arange(G), m)
    fb = np.array([orc.bf16_to_double(int(x)) for x in base.ravel()]).reshape(base.shape)
    fo = np.array([orc.bf16_to_double(int(x)) for x in out.ravel()]).reshape(out.shape)
    for r in range(M):
        for n in range(N):
            if fb[r, n] == 0 or not (2.0 ** -100 < abs(fb[r, n]) < 2.0 ** 100):
                continue
            want = np.ldexp(fb[r, n], int(ea[r] + eb[grp[r], n]))
            assert fo[r, n] == want, f"({r},{n}): {fo[r, n]} != {want}"


def pin_stacked_ownership(orc, seed=29):
    """Empty groups own no rows; rows past the last group stay untouched; counts that
    overrun total_M (or are negative) are clamped and reported."""
    rng = _rng(seed)
    G, N, K = 4, 8, 16
    A = _random_codes(rng, (10, K))
    B = _random_codes(rng, (G, N, K))
    sa = _random_scales(rng, 10)
    sb = _random_scales(rng, G * N).reshape(G, N)
    poison = np.full((10, N), 0xBEEF, np.uint16)
    out, clamped = orc.stacked(A, B, sa, sb, [0, 3, 0, 4], total_M=10, out=poison)
    assert not clamped
    assert np.all(out[7:] == 0xBEEF) and not np.any(out[:7] == 0xBEEF)
    off, clamped = orc.stacked_offsets([4, -1, 5, 9], 10)
    assert clamped and off.tolist() == [0, 4, 4, 9, 10]
    # rows 0..2 belong to group 1 ([0, 3, ...]): equal to a single-group problem
    single, _ = orc.stacked(A[:3], B[1:2], sa[:3], sb[1:2], [3], total_M=3)
    assert np.array_equal(out[:3], single)


def pin_padding_zero(orc, seed=31):
    """Dynamic padding rows are exactly +0.0 whatever the padding rows of A hold."""
    rng = _rng(seed)
    G, E, N, K = 3, 6, 8, 32
    zsi = np.array([0, 4, 6], np.int64)
    A = _random_codes(rng, (G * E, K))
    sa = _random_scales(rng, G * E)
    B = _random_codes(rng, (G, N, K))
    sb = _random_scales(rng, G * N).reshape(G, N)
    clean = orc.dynamic(A, B, sa, sb, zsi, E)
    for g in range(G):
        A[g * E + zsi[g]:(g + 1) * E] = 0x7F   # NaN codes
        sa[g * E + zsi[g]:(g + 1) * E] = np.nan
    poisoned = orc.dynamic(A, B, sa, sb, zsi, E)
    assert np.array_equal(clean, poisoned), "padding contents leaked into the output"
    for g in range(G):
        assert np.all(poisoned[g * E + zsi[g]:(g + 1) * E] == 0x0000)


def pin_layout_agreement(orc, seed=37):
    """The same valid rows give identical bits in the stacked and dynamic layouts."""
    rng = _rng(seed)
    G, N, K, E = 4, 8, 48, 5
    m = np.array([2, 0, 5, 3], np.int64)
    A = _random_codes(rng, (int(m.sum()), K))
    B = _random_codes(rng, (G, N, K))
    sa = _random_scales(rng, int(m.sum()))
    sb = _random_scales(rng, G * N).reshape(G, N)
    st, _ = orc.stacked(A, B, sa, sb, m)
    Ad = _random_codes(rng, (G * E, K))
    sad = _random_scales(rng, G * E)
    off = np.concatenate([[0], np.cumsum(m)])
    for g in range(G):
        Ad[g * E:g * E + m[g]] = A[off[g]:off[g + 1]]
        sad[g * E:g * E + m[g]] = sa[off[g]:off[g + 1]]
    dy = orc.dynamic(Ad, B, sad, sb, m, E)
    for g in range(G):
        assert np.array_equal(dy[g * E:g * E + m[g]], st[off[g]:off[g + 1]]), f"group {g}"


def pin_k_zero(orc):
    """A reduction over nothing gives +0.0 on every owned row."""
    G, N = 2, 8
    A = np.zeros((5, 0), np.uint8)
    B = np.zeros((G, N, 0), np.uint8)
    poison = np.full((5, N), 0x1234, np.uint16)
    out, _ = orc.stacked(A, B, np.ones(5, np.float32), np.ones((G, N), np.float32),
                         [2, 2], total_M=5, out=poison)
    assert np.all(out[:4] == 0) and np.all(out[4] == 0x1234)
    dy = orc.dynamic(np.zeros((6, 0), np.uint8), B, np.ones(6, np.float32),
                     np.ones((G, N), np.float32), [2, 3], 3)
    assert np.all(dy == 0)
    # +0.0 even with negative or NaN scales: the empty reduction is zeroed, not scaled
    out, _ = orc.stacked(A, B, np.array([-1, np.nan, 2, -3, 1], np.float32),
                         -np.ones((G, N), np.float32), [2, 2], total_M=5, out=poison)
    assert np.all(out[:4] == 0) and np.all(out[4] == 0x1234)


def pin_sampled_rows(orc, seed=41):
    """The row-sampling entry points equal the corresponding rows of the full oracle."""
    rng = _rng(seed)
    G, N, K = 3, 16, 40
    m = np.array([5, 0, 6], np.int64)
    A = _random_codes(rng, (13, K))
    B = _random_codes(rng, (G, N, K))
    sa = _random_scales(rng, 13)
    sb = _random_scales(rng, G * N).reshape(G, N)
    full, _ = orc.stacked(A, B, sa, sb, m, total_M=13)
    rows = np.array([0, 4, 5, 10, 12])
    part = orc.stacked_rows(A, B, sa, sb, m, rows)
    assert np.array_equal(part[:4], full[rows[:4]]) and np.all(part[4] == 0xFFFF)
    E = 7
    Ad = _random_codes(rng, (G * E, K))
    sad = _random_scales(rng, G * E)
    dy = orc.dynamic(Ad, B, sad, sb, [3, 7, 0], E)
    rows = np.array([0, 3, 6, 13, 14, 20])
    assert np.array_equal(orc.dynamic_rows(Ad, B, sad, sb, [3, 7, 0], E, rows), dy[rows])


def pin_offsets_layout(orc, cases=20, seed=43):
    """Offsets layout: brute force on tiny cases, and bit-equal to the stacked layout fed
    the steps between successive offsets."""
    rng = _rng(seed)
    for i in range(cases):
        A, B, sa, sb, m, total = _tiny_stacked_case(rng)
        incl = np.cumsum(m).astype(np.int32)
        out, _ = orc.offsets(A, B, sa, sb, incl, total_M=total,
                             out=np.full((total, B.shape[1]), 0xDEAD, np.uint16))
        ref = bf.offsets(A.tolist(), B.tolist(), sa.tolist(), sb.tolist(), incl.tolist(), total)
        for (r, n), bits in ref.items():
            got = int(out[r, n])
            assert got == bits or (bits == 0 and got == 0x8000), f"case {i} ({r},{n})"
        st, _ = orc.stacked(A, B, sa, sb, m, total_M=total,
                            out=np.full((total, B.shape[1]), 0xDEAD, np.uint16))
        assert np.array_equal(out, st), f"case {i}: offsets != stacked"


def pin_batched_layout(orc, cases=15, seed=47):
    """Batched layout: brute force on tiny cases, and bit-equal to the dynamic layout with
    every slab full."""
    rng = _rng(seed)
    for i in range(cases):
        G, M = int(rng.integers(1, 4)), int(rng.integers(1, 5))
        N, K = int(rng.integers(1, 7)), int(rng.choice([0, 1, 9, 32]))
        A = _random_codes(rng, (G * M, K))
        B = _random_codes(rng, (G, N, K))
        sa = _random_scales(rng, G * M)
        sb = _random_scales(rng, G * N).reshape(G, N)
        out = orc.batched(A, B, sa, sb)
        ref = bf.batched(A.tolist(), B.tolist(), sa.tolist(), sb.tolist(), M)
        for (r, n), bits in ref.items():
            got = int(out[r, n])
            assert got == bits or (bits == 0 and got == 0x8000), f"case {i} ({r},{n})"
        assert np.array_equal(out, orc.dynamic(A, B, sa, sb, [M] * G, M)), f"case {i}"


def _ragged_offsets(rng, G, total, step=1, over=False):
    """Random int32 inclusive offsets over `total` (multiples of `step`): some empty
    groups, optionally a last offset past `total` (clamped) or a decreasing step."""
    cuts = np.sort(rng.integers(0, total // step + 1, size=G)) * step
    if G > 1 and rng.random() < 0.5:
        cuts[rng.integers(0, G - 1)] = cuts[rng.integers(0, G - 1)]  # a repeated offset
    if over:
        cuts[-1] = total + step
    return cuts.astype(np.int32)


def pin_n_offsets_layout(orc, cases=20, seed=53):
    """Ragged-N layout: brute force on tiny cases (empty groups, columns past the last
    group untouched, clamping at total_N), and each group's columns bit-equal to the
    stacked layout with that group alone (A = the group's slab, B = its rows of B)."""
    rng = _rng(seed)
    for i in range(cases):
        G, M = int(rng.integers(1, 4)), int(rng.integers(1, 5))
        TN, K = int(rng.integers(1, 10)), int(rng.choice([0, 1, 9, 32]))
        A = _random_codes(rng, (G, M, K))
        B = _random_codes(rng, (TN, K))
        sa = _random_scales(rng, G * M).reshape(G, M)
        sb = _random_scales(rng, TN)
        off = _ragged_offsets(rng, G, TN, over=(i % 5 == 4))
        out, clamped = orc.n_offsets(A, B, sa, sb, off, out=np.full((M, TN), 0xDEAD, np.uint16))
        ref = bf.n_offsets(A.tolist(), B.tolist(), sa.tolist(), sb.tolist(), off.tolist(), TN)
        for (m, n), bits in ref.items():
            got = int(out[m, n])
            assert got == bits or (bits == 0 and got == 0x8000), f"case {i} ({m},{n})"
        owned = {n for (_, n) in ref}
        for n in range(TN):
            if n not in owned:
                assert np.all(out[:, n] == 0xDEAD), f"case {i}: column {n} written"
        assert clamped == (i % 5 == 4 and int(off[-1]) > TN), f"case {i}: clamp flag"
        start = 0
        for g in range(G):
            end = min(max(int(off[g]), start), TN)
            if end > start:
                st, _ = orc.stacked(A[g], B[start:end][None], sa[g], sb[start:end][None], [M],
                                    total_M=M)
                assert np.array_equal(out[:, start:end], st), f"case {i} group {g}"
            start = end


def pin_k_offsets_layout(orc, cases=20, seed=59):
    """Ragged-K layout: brute force on tiny cases (empty slices give +0.0, clamping at
    total_K), and each group's slab bit-equal to the stacked layout over its K slice; one
    group over all of K is the plain GEMM."""
    rng = _rng(seed)
    for i in range(cases):
        G, M, N = int(rng.integers(1, 4)), int(rng.integers(1, 5)), int(rng.integers(1, 6))
        TK = int(rng.choice([0, 16, 48, 64]))
        A = _random_codes(rng, (M, TK))
        B = _random_codes(rng, (N, TK))
        sa = _random_scales(rng, G * M).reshape(G, M)
        sb = _random_scales(rng, G * N).reshape(G, N)
        off = _ragged_offsets(rng, G, TK, step=int(rng.choice([1, 16])), over=(i % 5 == 4))
        out, clamped = orc.k_offsets(A, B, sa, sb, off)
        ref = bf.k_offsets(A.tolist(), B.tolist(), sa.tolist(), sb.tolist(), off.tolist(), TK)
        assert len(ref) == out.size
        for (r, n), bits in ref.items():
            got = int(out[r, n])
            assert got == bits or (bits == 0 and got == 0x8000), f"case {i} ({r},{n})"
        assert clamped == (i % 5 == 4 and int(off[-1]) > TK), f"case {i}: clamp flag"
        start = 0
        for g in range(G):
            end = min(max(int(off[g]), start), TK)
            st, _ = orc.stacked(A[:, start:end], B[None, :, start:end], sa[g], sb[g][None],
                                [M], total_M=M)
            assert np.array_equal(out[g * M:(g + 1) * M], st), f"case {i} group {g}"
            start = end
    # one group over all of K: the plain (dense) product
    A = _random_codes(rng, (3, 64))
    B = _random_codes(rng, (5, 64))
    sa, sb = _random_scales(rng, 3), _random_scales(rng, 5)
    out, _ = orc.k_offsets(A, B, sa, sb, [64])
    st, _ = orc.stacked(A, B[None], sa, sb[None], [3], total_M=3)
    assert np.array_equal(out, st)


def pin_ragged_sampled_rows(orc, seed=61):
    """The row-sampling forms of the ragged layouts equal rows of the full results."""
    rng = _rng(seed)
    A = _random_codes(rng, (3, 6, 32))
    B = _random_codes(rng, (11, 32))
    sa, sb = _random_scales(rng, 18).reshape(3, 6), _random_scales(rng, 11)
    off = np.array([4, 4, 11], np.int32)
    full, _ = orc.n_offsets(A, B, sa, sb, off)
    rows = np.array([5, 0, 3])
    part, _ = orc.n_offsets(A, B, sa, sb, off, rows=rows)
    assert np.array_equal(part, full[rows])
    A2, B2 = _random_codes(rng, (6, 64)), _random_codes(rng, (7, 64))
    sa2, sb2 = _random_scales(rng, 18).reshape(3, 6), _random_scales(rng, 21).reshape(3, 7)
    off2 = np.array([16, 48, 64], np.int32)
    full2, _ = orc.k_offsets(A2, B2, sa2, sb2, off2)
    rows2 = np.array([17, 0, 11, 6])
    part2, _ = orc.k_offsets(A2, B2, sa2, sb2, off2, rows=rows2)
    assert np.array_equal(part2, full2[rows2])


def _blockwise_case(rng, G, rows_per, N, K, pow2=False):
    m = [int(rows_per[g]) for g in range(G)]
    total = sum(m)
    A = _random_codes(rng, (total, K))
    B = _random_codes(rng, (G, N, K))
    nkb, nnb = K // 128, N // 128
    if pow2:
        sa = np.exp2(rng.integers(-3, 4, size=(total, nkb))).astype(np.float32)
        sb = np.exp2(rng.integers(-3, 4, size=(G, nnb, nkb))).astype(np.float32)
    else:
        sa = _random_scales(rng, total * nkb).reshape(total, nkb)
        sb = _random_scales(rng, G * nnb * nkb).reshape(G, nnb, nkb)
    return A, B, sa, sb, m, total


def pin_blockwise_bruteforce(orc, seed=67):
    """Block scaling: sampled elements bit-equal to the exact-rational sum over K blocks of
    scale_a[r, kb] * scale_b[g, n/128, kb] * (block sum), rounded once."""
    rng = _rng(seed)
    for i in range(3):
        G = int(rng.integers(1, 3))
        A, B, sa, sb, m, total = _blockwise_case(rng, G, rng.integers(0, 4, size=G) + (i == 0),
                                                 int(rng.choice([128, 256])), int(rng.choice([128, 256])))
        out, _ = orc.blockwise_stacked(A, B, sa, sb, m)
        N, K = B.shape[1], B.shape[2]
        start = 0
        for g in range(G):
            for r in range(start, start + m[g]):
                for n in rng.integers(0, N, size=6):
                    ref = bf.blockwise_element(A[r].tolist(), B[g, n].tolist(), sa[r].tolist(),
                                               sb[g, n // 128].tolist())
                    got = int(out[r, n])
                    assert got == ref or (ref == 0 and got == 0x8000), f"case {i} ({r},{n})"
            start += m[g]


def pin_blockwise_reduces_to_rowwise(orc, seed=71):
    """With scales constant over the K blocks (and over each 128-column block of B), block
    scaling is rowwise scaling: bit-equal to the rowwise oracle for power-of-two scales."""
    rng = _rng(seed)
    G, N, K = 2, 256, 384
    m = [3, 2]
    total = sum(m)
    A = _random_codes(rng, (total, K))
    B = _random_codes(rng, (G, N, K))
    sa_row = np.exp2(rng.integers(-4, 5, size=total)).astype(np.float32)
    sb_blk = np.exp2(rng.integers(-4, 5, size=(G, N // 128))).astype(np.float32)
    sa = np.repeat(sa_row[:, None], K // 128, axis=1)
    sb = np.repeat(sb_blk[:, :, None], K // 128, axis=2)
    out, _ = orc.blockwise_stacked(A, B, sa, sb, m)
    st, _ = orc.stacked(A, B, sa_row, np.repeat(sb_blk, 128, axis=1), m)
    assert np.array_equal(out, st)


def pin_blockwise_block_isolation(orc, seed=73):
    """A nonzero only in K block j: the result is that block's term alone, whatever the
    other blocks' scales hold (a scale indexed by the wrong block shows at once)."""
    rng = _rng(seed)
    G, N, K = 1, 128, 384
    A = np.zeros((3, K), np.uint8)
    B = _random_codes(rng, (G, N, K))
    for j in range(3):
        A[:] = 0
        A[:, j * 128:(j + 1) * 128] = _random_codes(rng, (3, 128))
        sa = np.full((3, 3), 1e30, np.float32)
        sb = np.full((G, 1, 3), 1e30, np.float32)
        sa[:, j] = np.float32(0.5)
        sb[:, :, j] = np.float32(2.0)
        out, _ = orc.blockwise_stacked(A, B, sa, sb, [3])
        ref, _ = orc.stacked(A[:, j * 128:(j + 1) * 128], B[:, :, j * 128:(j + 1) * 128],
                             np.ones(3, np.float32), np.ones((G, N), np.float32), [3])
        assert np.array_equal(out, ref), f"block {j}"


def _blockwise_dynamic_case(rng, G, E, N, K):
    A = _random_codes(rng, (G * E, K))
    B = _random_codes(rng, (G, N, K))
    sa = _random_scales(rng, G * E * (K // 128)).reshape(G * E, K // 128)
    sb = _random_scales(rng, G * (N // 128) * (K // 128)).reshape(G, N // 128, K // 128)
    return A, B, sa, sb


def pin_blockwise_dynamic_bruteforce(orc, seed=79):
    """Block-scaled dynamic and batched layouts: sampled columns of every slab row bit-equal
    to the exact-rational definition (padding rows +0.0; zsi clamped into [0, E])."""
    rng = _rng(seed)
    for i in range(4):
        G = int(rng.integers(2, 4))
        E = int(rng.integers(1, 4))
        N, K = int(rng.choice([128, 256])), int(rng.choice([128, 256]))
        A, B, sa, sb = _blockwise_dynamic_case(rng, G, E, N, K)
        zsi = None if i == 3 else rng.integers(-1, E + 2, size=G).astype(np.int64)
        if zsi is not None:
            zsi[0] = E  # one full slab at least
        out = (orc.blockwise_batched(A, B, sa, sb) if zsi is None
               else orc.blockwise_dynamic(A, B, sa, sb, zsi, E))
        cols = sorted(set(int(c) for c in rng.integers(0, N, size=5)) | {0, N - 1})
        ref = bf.blockwise_dynamic(A.tolist(), B.tolist(), sa.tolist(), sb.tolist(),
                                   None if zsi is None else zsi.tolist(), E, cols)
        for (r, n), bits in ref.items():
            got = int(out[r, n])
            valid = zsi is None or (r % E) < max(0, min(int(zsi[r // E]), E))
            if bits == 0x0000 and valid:
                assert got in (0x0000, 0x8000), f"case {i} ({r},{n}): {got:#06x} != 0"
            else:
                assert got == bits, f"case {i} ({r},{n}): {got:#06x} != {bits:#06x}"


def pin_blockwise_dynamic_layouts(orc, seed=83):
    """The valid rows of the block-scaled dynamic layout are the block-scaled stacked
    layout's rows bit for bit (rows scattered into slabs), padding rows are +0.0 whatever
    A and scale_a hold there, and the batched layout is the dynamic one with every slab
    full."""
    rng = _rng(seed)
    G, E, N, K = 3, 5, 256, 384
    zsi = np.array([2, 0, 5], np.int64)
    A, B, sa, sb = _blockwise_dynamic_case(rng, G, E, N, K)
    valid = np.concatenate([np.arange(g * E, g * E + zsi[g]) for g in range(G)])
    st, _ = orc.blockwise_stacked(A[valid], B, sa[valid], sb, zsi)
    dyn = orc.blockwise_dynamic(A, B, sa, sb, zsi, E)
    assert np.array_equal(dyn[valid], st)
    pad = np.setdiff1d(np.arange(G * E), valid)
    assert np.all(dyn[pad] == 0x0000)
    A2, sa2 = A.copy(), sa.copy()
    A2[pad] = 0x7F      # NaN codes
    sa2[pad] = np.nan
    assert np.array_equal(orc.blockwise_dynamic(A2, B, sa2, sb, zsi, E), dyn)
    full = orc.blockwise_dynamic(A, B, sa, sb, np.full(G, E, np.int64), E)
    assert np.array_equal(orc.blockwise_batched(A, B, sa, sb), full)
    rows = np.array([0, 4, 7, 11, 14], np.int64)
    assert np.array_equal(orc.blockwise_dynamic(A, B, sa, sb, zsi, E, rows=rows), dyn[rows])


PINS = [
    pin_decode_vs_torch, pin_decode_golden, pin_bf16_golden, pin_bf16_vs_torch,
    pin_dot_exact, pin_closed_form_k1, pin_closed_form_all_ones, pin_closed_form_identity,
    pin_coherent_groups, pin_golden_tiny, pin_bruteforce_stacked, pin_bruteforce_dynamic,
    pin_scale_factoring, pin_stacked_ownership, pin_padding_zero, pin_layout_agreement,
    pin_k_zero, pin_sampled_rows, pin_offsets_layout, pin_batched_layout,
    pin_n_offsets_layout, pin_k_offsets_layout, pin_ragged_sampled_rows,
    pin_blockwise_bruteforce, pin_blockwise_reduces_to_rowwise, pin_blockwise_block_isolation,
    pin_blockwise_dynamic_bruteforce, pin_blockwise_dynamic_layouts,
]
