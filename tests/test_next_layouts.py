"""GPU parity of the offsets (int32 inclusive prefix, 2D-3D) and batched (full slabs, 3D-3D)
layouts against the CPU oracle, and their agreement with the stacked and dynamic calls
they restate."""
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
    fx.device_status()


@pytest.fixture(scope="module")
def orc():
    return oracle.load(0)


def _variants(prefix):
    try:
        fxbuild.build()
        return [fx.variant_name(i) for i in range(fx.mslkb_num_variants())
                if fx.variant_name(i).startswith(prefix)
                and "blockscale" not in fx.variant_name(i)]   # rowwise variants only
    except Exception:  # noqa: BLE001 - collection must not depend on a toolchain
        return []


def _data(rows, G, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    A = random_codes((rows, K), g).numpy()
    B = random_codes((G, N, K), g).numpy()
    sa = (torch.rand(rows, generator=g) * 2 + 0.01).numpy().astype(np.float32)
    sb = (torch.rand(G * N, generator=g) * 2 + 0.01).numpy().astype(np.float32).reshape(G, N)
    return A, B, sa, sb


def _run_and_check(prob, orc, variant=None, poison=None, what=""):
    out = None
    if poison is not None:
        out = torch.full((prob.rows, prob.N), poison, dtype=torch.int16,
                         device="cuda").view(torch.bfloat16)
    res = prob.run_gpu(out=out, variant=variant)
    torch.cuda.synchronize()
    gb = bits_of(res).reshape(prob.rows, prob.N)
    ref, ab = prob.oracle_full(orc, poison=None if poison is None else
                               np.full((prob.rows, prob.N), poison & 0xFFFF, np.uint16))
    owned = prob.owned_rows_mask()
    compare(gb[owned].ravel(), ref[owned].ravel(), ab[owned].ravel(), what)
    if poison is not None:
        assert np.all(gb[~owned] == (poison & 0xFFFF)), f"{what}: unowned rows written"
    return gb


@pytest.mark.parametrize("variant", _variants("stacked"))
def test_offsets_every_variant(orc, variant):
    counts = [130, 0, 1, 257, 64, 0, 17]
    G, N, K = 7, 392, 688
    total = sum(counts) + 9
    A, B, sa, sb = _data(total, G, N, K, seed=51)
    incl = np.cumsum(counts).astype(np.int32)
    po = Problem.from_numpy("offsets", A, B, sa, sb, incl)
    got = _run_and_check(po, orc, variant=variant, poison=0x5A5A, what=f"offsets {variant}")
    ps = Problem.from_numpy("stacked", A, B, sa, sb, counts)
    ps.rows = po.rows = total
    out = torch.full((total, N), 0x5A5A, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    same = bits_of(ps.run_gpu(out=out, variant=variant)).reshape(total, N)
    assert np.array_equal(got, same), "offsets and stacked calls differ"


def test_offsets_non_monotonic_are_clamped(orc):
    # steps [5, -2, 7]: the negative step owns no rows, as a negative m_sizes entry
    G, N, K = 3, 64, 256
    A, B, sa, sb = _data(12, G, N, K, seed=52)
    po = Problem.from_numpy("offsets", A, B, sa, sb, [5, 3, 10])
    fx.device_status()
    _run_and_check(po, orc, poison=0x1234, what="non-monotonic offsets")
    assert fx.device_status() & fx.MSLKB_DEV_MSIZES_CLAMPED


@pytest.mark.parametrize("variant", _variants("dynamic"))
def test_batched_every_variant(orc, variant):
    G, M, N, K = 5, 200, 392, 688   # M does not divide a 128-row tile
    A, B, sa, sb = _data(G * M, G, N, K, seed=53)
    pb = Problem.from_numpy("batched", A, B, sa, sb, [], expected_m=M)
    got = _run_and_check(pb, orc, variant=variant, what=f"batched {variant}")
    pd = Problem.from_numpy("dynamic", A, B, sa, sb, [M] * G, expected_m=M)
    same = bits_of(pd.run_gpu(variant=variant)).reshape(G * M, N)
    assert np.array_equal(got, same), "batched and dynamic (full slabs) calls differ"


@pytest.mark.parametrize("K", [1000, 16, 0])
def test_batched_k_tails(orc, K):
    G, M, N = 3, 70, 136
    A, B, sa, sb = _data(G * M, G, N, K, seed=54 + K)
    pb = Problem.from_numpy("batched", A, B, sa, sb, [], expected_m=M)
    got = _run_and_check(pb, orc, what=f"batched K={K}")
    if K == 0:
        assert np.all(got == 0)


def test_offsets_and_batched_small_m_split(orc):
    # few rows per group: swap-AB tiles, split along K over all SMs
    counts = [1, 0, 2, 1]
    A, B, sa, sb = _data(4, 4, 1024, 4096, seed=55)
    po = Problem.from_numpy("offsets", A, B, sa, sb, np.cumsum(counts).astype(np.int32))
    _run_and_check(po, orc, what="offsets small M")
    A, B, sa, sb = _data(4 * 3, 4, 1024, 4096, seed=56)
    pb = Problem.from_numpy("batched", A, B, sa, sb, [], expected_m=3)
    _run_and_check(pb, orc, what="batched small M")
    assert fx.device_status() == 0
