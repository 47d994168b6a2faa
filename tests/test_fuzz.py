"""Seeded random problems through the planner's own choice of variant, compared with the
oracle element by element: random group counts and sizes (empty groups, single rows,
groups larger than a tile), N any multiple of 8, K any size (K % 16 != 0 takes the
cp.async loader), dynamic valid-row counts outside [0, E], scales over 16 binades.  Rows a
layout does not own must keep their contents."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
import fp8_rowwise_scaled_gb300 as fx
from fp8_rowwise_scaled_gb300 import build as fxbuild
from fp8_rowwise_scaled_gb300.synthetic import random_codes
from parity_util import Problem, bits_of, compare

pytestmark = pytest.mark.gpu

LAYOUTS = ("stacked", "dynamic", "offsets", "batched")
# cases per layout, and per ragged / block-scaled entry point; a longer run draws more seeds
# (e.g. MSLKB_FUZZ_CASES=2500 MSLKB_FUZZ_SIDE_CASES=800)
CASES_PER_LAYOUT = int(os.environ.get("MSLKB_FUZZ_CASES", "16"))
SIDE_CASES = int(os.environ.get("MSLKB_FUZZ_SIDE_CASES", "10"))
POISON = 0x5A5A


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fxbuild.build()
    fx.lib()
    fx.device_status()


@pytest.fixture(scope="module")
def orc():
    return oracle.load(0)


def _problem(layout: str, i: int) -> Problem:
    rng = np.random.default_rng(4000 + 97 * LAYOUTS.index(layout) + i)
    G = int(rng.integers(1, 17))
    N = 8 * int(rng.integers(1, 65))
    K = int(rng.integers(1, 41)) * 16 if rng.random() < 0.6 else int(rng.integers(1, 641))
    per = int(rng.choice([1, 3, 16, 40, 140]))
    g = torch.Generator().manual_seed(int(rng.integers(1 << 30)))
    if layout in ("stacked", "offsets"):
        counts = rng.integers(0, 2 * per + 1, size=G)
        counts[rng.random(G) < 0.25] = 0
        rows = int(counts.sum())
        meta = np.cumsum(counts).astype(np.int32) if layout == "offsets" else counts
        E = 0
    else:
        E = max(1, per)
        rows = G * E
        meta = rng.integers(-2, E + 3, size=G) if layout == "dynamic" else np.zeros(G, np.int64)
    A = random_codes((max(rows, 0), K), g).numpy()
    B = random_codes((G, N, K), g).numpy()
    sa = (np.exp2(rng.integers(-8, 8, size=rows)) * rng.uniform(0.5, 1.5, size=rows))
    sb = (np.exp2(rng.integers(-8, 8, size=(G, N))) * rng.uniform(0.5, 1.5, size=(G, N)))
    return Problem.from_numpy(layout, A, B, sa.astype(np.float32), sb.astype(np.float32),
                              meta, expected_m=E)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("i", range(CASES_PER_LAYOUT))
def test_fuzz(orc, layout, i):
    prob = _problem(layout, i)
    if prob.rows == 0:
        pytest.skip("no rows drawn")
    out = torch.full((prob.rows, prob.N), POISON, dtype=torch.int16, device="cuda")
    out = out.view(torch.bfloat16)
    res = prob.run_gpu(out=out)
    torch.cuda.synchronize()
    got = bits_of(res).reshape(prob.rows, prob.N)
    ref, ab = prob.oracle_full(orc, poison=np.full((prob.rows, prob.N), POISON, np.uint16))
    owned = prob.owned_rows_mask()
    what = f"{layout} #{i}: G={prob.G} N={prob.N} K={prob.K} rows={prob.rows}"
    compare(got[owned].ravel(), ref[owned].ravel(), ab[owned].ravel(), what)
    assert np.all(got[~owned] == POISON), f"{what}: rows it does not own were written"
    assert fx.device_status() == 0


# -- the ragged and block-scaled entry points, through their own parity helpers ---------

@pytest.mark.parametrize("i", range(SIDE_CASES))
def test_fuzz_ragged_n(orc, i):
    from test_ragged_layouts import _n_offsets_case
    rng = np.random.default_rng(5000 + i)
    G = int(rng.integers(1, 13))
    M = int(rng.choice([int(rng.integers(1, 33)), int(rng.integers(33, 300))]))
    K = 16 * int(rng.integers(1, 41))
    cols = rng.integers(0, 600, size=G)
    cols[rng.random(G) < 0.2] = 0
    total_N = 8 * (-(-int(cols.sum()) // 8)) + 8 * int(rng.integers(0, 4))
    if total_N == 0:
        pytest.skip("no columns drawn")
    _n_offsets_case(orc, G, M, total_N, K, cols.tolist(), seed=5100 + i)
    assert fx.device_status() == 0


@pytest.mark.parametrize("i", range(SIDE_CASES))
def test_fuzz_ragged_k(orc, i):
    from test_ragged_layouts import _k_offsets_case
    rng = np.random.default_rng(6000 + i)
    G = int(rng.integers(1, 13))
    M = int(rng.choice([int(rng.integers(1, 33)), int(rng.integers(33, 260))]))
    N = 8 * int(rng.integers(1, 49))
    ks = 16 * rng.integers(0, 60, size=G)
    ks[rng.random(G) < 0.2] = 0
    total_K = int(ks.sum()) + 16 * int(rng.integers(0, 8))
    if total_K == 0:
        pytest.skip("no K drawn")
    _k_offsets_case(orc, G, M, N, total_K, ks.tolist(), seed=6100 + i)
    assert fx.device_status() == 0


@pytest.mark.parametrize("i", range(SIDE_CASES))
def test_fuzz_groupwise(orc, i):
    from test_blockscale import _case, _check, _run
    rng = np.random.default_rng(7000 + i)
    G = int(rng.integers(1, 9))
    per = int(rng.choice([2, 16, 30, 150]))
    m = rng.integers(0, 2 * per + 1, size=G)
    m[rng.random(G) < 0.2] = 0
    if int(m.sum()) == 0:
        pytest.skip("no rows drawn")
    N = 128 * int(rng.integers(1, 5))
    K = 128 * int(rng.integers(1, 9))
    A, B, sa, sb, mm, rows = _case(7100 + i, G, m.tolist(), N, K, wide=bool(rng.random() < 0.5))
    got = _run(A, B, sa, sb, mm, rows, N)
    _check(orc, A, B, sa, sb, mm, rows, got, f"groupwise #{i}: G={G} N={N} K={K} m={m.tolist()}")
    assert fx.device_status() == 0


# -- random problems sized to land on each of the planner's choices ----------------------

PLAN_CASES = [
    # (layout, expected variant, per-group rows, G range, N choices, K choices, empty groups:
    # a fraction of G, or "one" -- exactly one, so that the mean the planner sees stays on
    # the branch)
    ("stacked", "stacked_swap_w128xa16_tma", (0, 16), (4, 32), (1024, 2048), (1024, 2048), 0.2),
    ("stacked", "stacked_swap_w128xa32_tma", (18, 32), (4, 16), (1024, 2048), (512, 1024), 0.0),
    # decode with long K ranges per CTA: weights of two K blocks per TMA operation (an odd
    # number of K blocks leaves a last single one)
    ("stacked", "stacked_swap_w128xa16_tma", (1, 16), (12, 16), (8192,), (8192, 8320, 6272), 0.2),
    ("stacked", "stacked_tile128x256_tma", (300, 480), (12, 16), (2048, 4096), (512, 1024), "one"),
    ("stacked", "stacked_pair256x256_tma", (1200, 1500), (16, 20), (1024, 2048), (256, 512), "one"),
    ("dynamic", "dynamic_pair256x256_tma", (520, 600), (16, 24), (2048,), (256, 512), 0.0),
    # skewed groups (a few large, many small: "zipf" draws rows ~ (rank + 1)^-1.1) with a
    # mean of at least 512 rows: CTA pairs, many groups ending in half-used pair tiles
    ("stacked", "stacked_pair256x256_tma", (600, 900), (16, 32), (2048,), (256, 512), "zipf"),
    ("stacked", "stacked_tile128x128_cpasync", (200, 600), (4, 8), (1024,),
     (1000, 1001, 1004, 1036), 0.2),
]


PLAN_DRAWS = int(os.environ.get("MSLKB_FUZZ_PLAN_DRAWS", "2"))


@pytest.mark.parametrize("case", range(len(PLAN_CASES) * PLAN_DRAWS))
def test_fuzz_planner_choices(orc, case):
    """Random groups around each branch of the planner (swap-AB 16 / 32, 128 x 256 tiles,
    CTA pairs claiming their tiles on the stacked layout and in a fixed stride on slabs,
    the cp.async loader), PLAN_DRAWS draws each: the planner must pick the expected kernel; the
    sampled rows (first, last and random rows of every group) must match the oracle and no
    owned element may keep the fill pattern."""
    layout, want, (lo, hi), (g_lo, g_hi), n_choices, k_choices, empty = \
        PLAN_CASES[case % len(PLAN_CASES)]
    rng = np.random.default_rng(8000 + case)
    G = int(rng.integers(g_lo, g_hi + 1))
    N = int(rng.choice(n_choices))
    K = int(rng.choice(k_choices))
    g = torch.Generator().manual_seed(8100 + case)
    if layout == "stacked":
        if empty == "zipf":   # G groups sharing G x mean rows, Zipf-sized, shuffled
            mean = int(rng.integers(lo, hi + 1))
            w = 1.0 / np.arange(1, G + 1) ** 1.1
            counts = np.floor(w / w.sum() * G * mean).astype(np.int64)
            rng.shuffle(counts)
        else:
            counts = rng.integers(lo, hi + 1, size=G)
            if empty == "one":
                counts[int(rng.integers(G))] = 0
            else:
                counts[rng.random(G) < empty] = 0
        rows, meta, E = int(counts.sum()), counts, 0
    else:
        E = int(rng.integers(lo, hi + 1))
        rows, meta = G * E, rng.integers(-2, E + 3, size=G)
    if rows == 0:
        pytest.skip("every group drawn empty")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = fx.mslkb_plan(0 if layout == "stacked" else 1, rows if layout == "stacked" else E,
                         G, N, K, sms)
    assert fx.variant_name(plan.variant) == want, (fx.variant_name(plan.variant), G, N, K, rows)
    A = random_codes((rows, K), g).numpy()
    B = random_codes((G, N, K), g).numpy()
    sa = (np.exp2(rng.integers(-6, 6, size=rows)) * rng.uniform(0.5, 1.5, size=rows))
    sb = (np.exp2(rng.integers(-6, 6, size=(G, N))) * rng.uniform(0.5, 1.5, size=(G, N)))
    prob = Problem.from_numpy(layout, A, B, sa.astype(np.float32), sb.astype(np.float32), meta,
                              expected_m=E)
    out = torch.full((rows, N), 0x7E7E, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    prob.run_gpu(out=out)
    torch.cuda.synchronize()
    assert fx.device_status() == 0
    owned = torch.from_numpy(prob.owned_rows_mask()).cuda()
    left = int((out.view(torch.int16)[owned] == 0x7E7E).sum().item())
    assert left == 0, f"{want}: {left} owned elements still hold the fill pattern"
    sample = prob.sample_rows(per_group_random=1, seed=case, cap=96)
    got = bits_of(out[torch.from_numpy(sample).cuda()]).reshape(sample.size, N)
    ref, ab = prob.oracle_rows(orc, sample)
    compare(got.ravel(), ref.ravel(), ab.ravel(), f"{want} G={G} N={N} K={K} rows={rows}")
