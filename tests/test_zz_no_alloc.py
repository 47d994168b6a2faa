"""The allocation-free stacked entry point, through the C ABI, against the oracle.

Some callers cannot allocate device memory when they call this library: plug-ins whose
host framework owns every device allocation, and serving loops that cannot take the
device-wide synchronisation a cudaMalloc can cause.  They use
mslkb_f8f8bf16_rowwise_grouped_stacked_noalloc, whose split-tile scratch is a static
device array instead of a workspace the library allocates.  Its output must match the
oracle within the parity tolerance on two calls in a row (the second call finds the array
holding the first call's leftovers), on every kind of plan it can take: split swap-AB
tiles (some or all tiles split), the cp.async loader for a K that is not a multiple of
16, K = 0, and CTA pairs (which take their tiles in a fixed stride here).  This file runs
last so that a failure here cannot hide any other test; it passes alone in a fresh
process as well.
"""
import numpy as np
import pytest
import torch

import oracle
import fp8_rowwise_scaled_gb300 as fx
from fp8_rowwise_scaled_gb300 import build as fxbuild
from fp8_rowwise_scaled_gb300.synthetic import random_codes
from parity_util import Problem, bits_of, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fxbuild.build()
    fx.lib()


@pytest.fixture(scope="module")
def orc():
    return oracle.load(0)


def _problem(G, N, K, m_sizes, seed):
    g = torch.Generator().manual_seed(seed)
    rows = int(sum(m_sizes))
    A = random_codes((rows, K), g).numpy()
    B = random_codes((G, N, K), g).numpy()
    sa = (torch.rand(rows, generator=g) + 0.5).numpy().astype(np.float32)
    sb = (torch.rand(G * N, generator=g) + 0.5).numpy().astype(np.float32).reshape(G, N)
    return Problem.from_numpy("stacked", A, B, sa, sb, m_sizes)


def _call(fn, prob, out):
    st = torch.cuda.current_stream().cuda_stream
    return fn(prob.A.data_ptr(), prob.B.data_ptr(), prob.sa.data_ptr(), prob.sb.data_ptr(),
              prob.meta.data_ptr(), out.data_ptr(), prob.rows, prob.G, prob.N, prob.K, st)


CASES = {
    # whole waves of swap-AB tiles, then a split remainder
    "split_remainder": (16, 4096, 4096, [3, 0, 1, 2, 0, 4, 1, 1, 0, 2, 1, 1, 0, 1, 2, 1], 41,
                        "stacked_swap_w128xa16_tma", True),
    # fewer tiles than SMs: every tile is split
    "every_tile_split": (4, 1024, 4096, [1, 0, 2, 0], 42, "stacked_swap_w128xa16_tma", True),
    # K = 1000 (8 mod 16): the cp.async loader, split too
    "cpasync_k_tail": (8, 2048, 1000, [2, 0, 1, 3, 0, 1, 4, 1], 44,
                       "stacked_swap_w128xa16_cpasync", True),
    # an empty reduction: every owned row +0.0
    "k_zero": (4, 512, 0, [5, 0, 9, 2], 45, None, False),
    # groups of ~1000 rows: CTA pairs, tiles in a fixed stride (no claim counter here)
    "cta_pairs": (2, 8192, 256, [1100, 1000], 46, "stacked_pair256x256_tma", False),
}


@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_matches_oracle_twice(orc, case):
    G, N, K, m_sizes, seed, variant, split = CASES[case]
    prob = _problem(G, N, K, m_sizes, seed)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = fx.mslkb_plan(0, prob.rows, prob.G, prob.N, prob.K, sms,
                         a_align=256, b_align=256)
    if variant is not None:
        assert fx.variant_name(plan.variant) == variant, "the case must take its plan"
    assert plan.split_k == int(split), "the case must (not) use the split-tile scratch"
    ref, ab = prob.oracle_full(orc)
    fx.device_status()
    for call in range(2):
        out = torch.full((prob.rows, prob.N), 0x7E7E, dtype=torch.int16,
                         device="cuda").view(torch.bfloat16)
        s = _call(fx.mslkb_f8f8bf16_rowwise_grouped_stacked_noalloc, prob, out)
        assert s == fx.MSLKB_OK, fx.mslkb_status_string(s)
        torch.cuda.synchronize()
        compare(bits_of(out).ravel(), ref.ravel(), ab.ravel(), f"{case}, call {call + 1}")
    assert fx.device_status() == 0


def test_noalloc_rejects_plans_beyond_its_scratch():
    # 256 rows per group plan 128-row activation tiles; when those are split too (policy
    # 2), their partial sums need more than the static array holds: a clear error,
    # nothing launched
    prob = _problem(2, 4096, 1024, [256, 256], 43)
    out = torch.zeros((prob.rows, prob.N), dtype=torch.bfloat16, device="cuda")
    fx.mslkb_set_split_k(2)
    try:
        s = _call(fx.mslkb_f8f8bf16_rowwise_grouped_stacked_noalloc, prob, out)
    finally:
        fx.mslkb_set_split_k(1)
    assert s == fx.MSLKB_ERR_TOO_LARGE
    assert "scratch" in fx.mslkb_status_string(s)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out.view(torch.int16)).item() == 0
