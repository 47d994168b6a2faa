"""Failure detection without a GPU fault: every pipeline wait in the kernels is bounded.
A test hook makes CTA 0 of the next launch withhold one pipeline stage (a barrier that
nothing completes); its MMA wait runs out after the configured limit, the kernel records
MSLKB_DEV_TIMEOUT in the device status word, waits for its copies in flight, frees its
tensor memory and returns.  The host reads the status, and the context stays usable: the
same call then gives the oracle's result."""
import numpy as np
import pytest
import torch

import oracle
import fp8_rowwise_scaled_gb300 as fx
from fp8_rowwise_scaled_gb300 import build as fxbuild
from fp8_rowwise_scaled_gb300.synthetic import random_codes
from parity_util import Problem, abs_codes, bits_of, compare


@pytest.fixture(scope="module")
def L():
    fxbuild.build()
    return fx.lib()


def test_timeout_setting_arguments(L):
    with pytest.raises(fx.MslkbError):
        fx.mslkb_set_wait_timeout_us(-1)
    with pytest.raises(fx.MslkbError):
        fx.mslkb_set_wait_timeout_us(999)     # below 1 ms
    fx.mslkb_set_wait_timeout_us(5000)
    fx.mslkb_set_wait_timeout_us(0)           # back to the default


@pytest.mark.gpu
@pytest.mark.parametrize("shape", ["tiles", "swap"])
def test_wait_runs_out_and_the_context_survives(L, shape):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g = torch.Generator().manual_seed(77)
    if shape == "tiles":    # 128-row tiles, whole (no split tiles)
        G, N, K, m = 4, 1024, 1024, [300, 0, 257, 411]
    else:                   # swap-AB tiles, split along K over every CTA
        G, N, K, m = 8, 2048, 2048, [1, 0, 3, 2, 0, 1, 1, 2]
    rows = sum(m)
    A = random_codes((rows, K), g).numpy()
    B = random_codes((G, N, K), g).numpy()
    sa = (torch.rand(rows, generator=g) + 0.5).numpy().astype(np.float32)
    sb = (torch.rand(G * N, generator=g) + 0.5).numpy().astype(np.float32).reshape(G, N)
    prob = Problem.from_numpy("stacked", A, B, sa, sb, m)
    fx.device_status()                        # start clean
    fx.mslkb_set_wait_timeout_us(50_000)      # 50 ms
    try:
        fx.mslkb_test_stall_next_launch()
        prob.run_gpu()
        torch.cuda.synchronize()              # the launch returns: no hang, no fault
        assert fx.device_status() & fx.MSLKB_DEV_TIMEOUT
    finally:
        fx.mslkb_set_wait_timeout_us(0)
    # the context and the library keep working: the same call gives the oracle's result
    out = bits_of(prob.run_gpu()).reshape(rows, N)
    torch.cuda.synchronize()
    assert fx.device_status() == 0
    orc = oracle.load(0)
    h = prob.host()
    ref, _ = orc.stacked(h["A"], h["B"], h["sa"], h["sb"], h["meta"])
    ab, _ = orc.stacked(abs_codes(h["A"]), abs_codes(h["B"]), np.abs(h["sa"]), np.abs(h["sb"]),
                        h["meta"])
    compare(out.ravel(), ref.ravel(), ab.ravel(), f"after a timeout ({shape})")


@pytest.mark.gpu
@pytest.mark.parametrize("layout", ["stacked", "dynamic"])
def test_cta_pair_wait_runs_out_and_the_next_calls_are_right(L, layout):
    """The same on the CTA-pair kernels: both CTAs of the first pair skip one stage, so the
    leader's MMA wait runs out, the peer's waits run out after it, and both meet at the
    pair's teardown barriers, free their tensor memory and return.  The stacked plan takes
    its tiles from the stream's claim counter, which the last leader through teardown resets
    on the abort path too: the next call, enqueued right behind the stalled one (before the
    host reads the status word, which would also clear the counter), and one more after it
    must both match the oracle.  The dynamic plan takes its tiles in a fixed stride."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g = torch.Generator().manual_seed(78)
    if layout == "stacked":
        G, N, K, meta, E = 2, 8192, 1024, [1100, 1000], 0
        rows = sum(meta)
    else:
        G, N, K, meta, E = 4, 8192, 512, [600, 300, 0, 599], 600
        rows = G * E
    A = random_codes((rows, K), g).numpy()
    B = random_codes((G, N, K), g).numpy()
    sa = (torch.rand(rows, generator=g) + 0.5).numpy().astype(np.float32)
    sb = (torch.rand(G * N, generator=g) + 0.5).numpy().astype(np.float32).reshape(G, N)
    prob = Problem.from_numpy(layout, A, B, sa, sb, meta, expected_m=E)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = fx.mslkb_plan(0 if layout == "stacked" else 1, rows if layout == "stacked" else E,
                         G, N, K, sms)
    assert fx.variant_name(plan.variant) == f"{layout}_pair256x256_tma"
    orc = oracle.load(0)
    ref, ab = prob.oracle_full(orc)

    def poisoned():
        return torch.full((rows, N), 0x7E7E, dtype=torch.int16,
                          device="cuda").view(torch.bfloat16)

    fx.device_status()                        # start clean
    outs = [poisoned() for _ in range(3)]
    fx.mslkb_set_wait_timeout_us(50_000)      # 50 ms
    try:
        fx.mslkb_test_stall_next_launch()
        prob.run_gpu(out=outs[0])
    finally:
        fx.mslkb_set_wait_timeout_us(0)
    prob.run_gpu(out=outs[1])                 # right behind the stalled launch
    torch.cuda.synchronize()                  # both return: no hang, no fault
    assert fx.device_status() & fx.MSLKB_DEV_TIMEOUT
    compare(bits_of(outs[1]).ravel(), ref.ravel(), ab.ravel(),
            f"{layout} pairs, the call after a timeout")
    prob.run_gpu(out=outs[2])
    torch.cuda.synchronize()
    assert fx.device_status() == 0
    compare(bits_of(outs[2]).ravel(), ref.ravel(), ab.ravel(),
            f"{layout} pairs, the second call after a timeout")


def _stall_then_right(stalled_call, right_call, what):
    """The next launch withholds a stage: it must return with MSLKB_DEV_TIMEOUT set; then
    the same problem, called again, must match the oracle (right_call checks that)."""
    fx.device_status()                        # start clean
    fx.mslkb_set_wait_timeout_us(50_000)      # 50 ms
    try:
        fx.mslkb_test_stall_next_launch()
        stalled_call()
        torch.cuda.synchronize()              # the launch returns: no hang, no fault
        assert fx.device_status() & fx.MSLKB_DEV_TIMEOUT, what
    finally:
        fx.mslkb_set_wait_timeout_us(0)
    right_call()
    torch.cuda.synchronize()
    assert fx.device_status() == 0, what


@pytest.mark.gpu
@pytest.mark.parametrize("family", ["blockscale_tile128x256_tma",
                                    "dynamic_blockscale_swap_w128xa16_tma",
                                    "ragn_tile128x256_tma", "ragk_tile128x256_tma"])
def test_wait_runs_out_on_the_other_kernel_families(L, family):
    """The same on the block-scaled kernels (whose stages the epilogue frees, and whose
    128 x 256 tiles issue their K blocks from the unrolled runs: K = 2048 gives 16 blocks)
    and on the ragged-N and ragged-K kernels."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    orc = oracle.load(0)
    if family == "blockscale_tile128x256_tma":
        from test_blockscale import _case, _check, _run
        A, B, sa, sb, m, rows = _case(81, 4, [300, 0, 257, 411], 512, 2048)
        _stall_then_right(lambda: _run(A, B, sa, sb, m, rows, 512, family),
                          lambda: _check(orc, A, B, sa, sb, m, rows,
                                         _run(A, B, sa, sb, m, rows, 512, family), family),
                          family)
    elif family == "dynamic_blockscale_swap_w128xa16_tma":
        from test_blockscale_slabs import _case, _check, _run
        zsi = [16, 3, 0, 9, 16, 1, 12, 7]
        A, B, sa, sb = _case(82, 8, 16, 1024, 2048, zsi)
        _stall_then_right(lambda: _run(A, B, sa, sb, zsi, 16, family),
                          lambda: _check(orc, A, B, sa, sb, zsi, 16,
                                         _run(A, B, sa, sb, zsi, 16, family), family),
                          family)
    elif family == "ragn_tile128x256_tma":
        from test_ragged_layouts import _cuda, _data, _n_offsets_case, _run
        G, M, total_N, K, cols = 4, 300, 2048, 1024, [500, 0, 777, 600]
        A, B, sa, sb = _data(83, (G, M, K), (total_N, K), G * M, total_N)
        tA, tB, tsa, tsb, toff = _cuda(A, B, sa, sb, np.cumsum(cols).astype(np.int32))
        out = torch.empty((M, total_N), dtype=torch.bfloat16, device="cuda")
        _stall_then_right(
            lambda: _run(fx.f8f8bf16_rowwise_grouped_n_offsets, family, tA, tB, tsa, tsb, toff,
                         out),
            lambda: _n_offsets_case(orc, G, M, total_N, K, cols, seed=83, variant=family),
            family)
    else:
        from test_ragged_layouts import _cuda, _data, _k_offsets_case, _run
        G, M, N, ks = 4, 300, 512, [1024, 0, 2048, 512]
        total_K = sum(ks)
        A, B, sa, sb = _data(84, (M, total_K), (N, total_K), G * M, G * N)
        tA, tB, tsa, tsb, toff = _cuda(A, B, sa, sb, np.cumsum(ks).astype(np.int32))
        out = torch.empty((G, M, N), dtype=torch.bfloat16, device="cuda")
        _stall_then_right(
            lambda: _run(fx.f8f8bf16_rowwise_grouped_k_offsets, family, tA, tB, tsa, tsb, toff,
                         out),
            lambda: _k_offsets_case(orc, G, M, N, total_K, ks, seed=84, variant=family),
            family)
