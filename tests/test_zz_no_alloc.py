"""The allocation-free stacked entry point, through the C ABI.

Callers that cannot allocate device memory -- code recording a CUDA graph, plug-ins whose
framework owns all device memory, serving loops that cannot take a cudaMalloc's device
synchronisation -- use mslkb_f8f8bf16_rowwise_grouped_stacked_noalloc, whose split-tile
scratch is a static device array.  Its output must match the regular stacked entry
point's within the parity tolerance, on two calls in a row (the second call finds the
array holding the first call's leftovers).  This file runs last so that a failure here
cannot hide any other test; it passes alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

import oracle
import fp8_rowwise_scaled_gb300 as fx
from fp8_rowwise_scaled_gb300 import build as fxbuild
from fp8_rowwise_scaled_gb300.synthetic import random_codes
from parity_util import Problem, abs_codes, bits_of, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fxbuild.build()
    fx.lib()


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


@pytest.mark.parametrize("shape", ["split_remainder", "every_tile_split"])
def test_noalloc_matches_stacked_twice(shape):
    if shape == "split_remainder":   # whole waves, then a split remainder
        prob = _problem(16, 4096, 4096, [3, 0, 1, 2, 0, 4, 1, 1, 0, 2, 1, 1, 0, 1, 2, 1], 41)
    else:                            # fewer tiles than SMs: every tile is split
        prob = _problem(4, 1024, 4096, [1, 0, 2, 0], 42)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = fx.mslkb_plan(0, prob.rows, prob.G, prob.N, prob.K, sms)
    assert plan.split_k == 1, "the shape must exercise the split-tile scratch"

    ref = torch.zeros((prob.rows, prob.N), dtype=torch.bfloat16, device="cuda")
    assert _call(fx.mslkb_f8f8bf16_rowwise_grouped_stacked, prob, ref) == fx.MSLKB_OK
    torch.cuda.synchronize()
    ref_bits = bits_of(ref).ravel()
    # tolerance term 1e-6 * |sa * sb| * sum_k |a_k b_k| from the oracle on |codes|, |scales|
    h = prob.host()
    orc = oracle.load(0)
    ab, _ = orc.stacked(abs_codes(h["A"]), abs_codes(h["B"]), np.abs(h["sa"]), np.abs(h["sb"]),
                        h["meta"])
    for call in range(2):
        out = torch.full((prob.rows, prob.N), 0x7E7E, dtype=torch.int16,
                         device="cuda").view(torch.bfloat16)
        s = _call(fx.mslkb_f8f8bf16_rowwise_grouped_stacked_noalloc, prob, out)
        assert s == fx.MSLKB_OK, fx.mslkb_status_string(s)
        torch.cuda.synchronize()
        compare(bits_of(out).ravel(), ref_bits, ab.ravel(), f"{shape}, call {call + 1}")
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
