"""GPU parity of the ragged layouts against the oracle, through the C ABI: ragged N (3D-2D,
groups partition the weight rows / output columns) and ragged K (2D-2D, groups slice the
contraction), on every kernel variant, with group extents that do not divide the tiles,
empty groups, a group narrower than one tile, slices whose end falls mid-way through a
32-byte MMA step, and the untouched / zeroed regions each layout defines."""
import numpy as np
import pytest
import torch

import oracle
import fp8_rowwise_scaled_gb300 as fx
from fp8_rowwise_scaled_gb300 import build as fxbuild
from fp8_rowwise_scaled_gb300.synthetic import random_codes
from parity_util import abs_codes, bits_of, compare

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
                if fx.variant_name(i).startswith(prefix)]
    except Exception:  # noqa: BLE001 - collection must not depend on a toolchain
        return []


def _data(seed, a_shape, b_shape, sa_n, sb_n, nan=False):
    g = torch.Generator().manual_seed(seed)
    A = random_codes(a_shape, g, allow_nan=nan).numpy()
    B = random_codes(b_shape, g, allow_nan=nan).numpy()
    sa = (torch.rand(sa_n, generator=g) * 2 + 0.01).numpy().astype(np.float32)
    sb = (torch.rand(sb_n, generator=g) * 2 + 0.01).numpy().astype(np.float32)
    return A, B, sa, sb


def _cuda(*arrs):
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrs]


def _run(fn, variant, *args):
    if variant is not None:
        fx.mslkb_force_variant(fx.variant_index(variant))
    try:
        return fn(*args)
    finally:
        if variant is not None:
            fx.mslkb_force_variant(-1)


def _n_offsets_case(orc, G, M, total_N, K, cols, seed, variant=None, poison=0x5A5A):
    """cols: column count per group (offsets are their inclusive prefix)."""
    A, B, sa, sb = _data(seed, (G, M, K), (total_N, K), G * M, total_N)
    off = np.cumsum(cols).astype(np.int32)
    tA, tB, tsa, tsb, toff = _cuda(A, B, sa, sb, off)
    out = torch.full((M, total_N), poison, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    _run(fx.f8f8bf16_rowwise_grouped_n_offsets, variant, tA, tB, tsa, tsb, toff, out)
    torch.cuda.synchronize()
    got = bits_of(out).reshape(M, total_N)
    ref, _ = orc.n_offsets(A, B, sa.reshape(G, M), sb, off,
                           out=np.full((M, total_N), poison, np.uint16))
    ab, _ = orc.n_offsets(abs_codes(A), abs_codes(B), np.abs(sa).reshape(G, M), np.abs(sb), off)
    owned = np.zeros(total_N, bool)
    owned[:min(int(off[-1]), total_N)] = True
    assert np.all(got[:, ~owned] == poison), f"{variant}: columns past the last group written"
    st = compare(got[:, owned].ravel(), ref[:, owned].ravel(), ab[:, owned].ravel(),
                 f"ragged N {variant} {cols}")
    return st


def _k_offsets_case(orc, G, M, N, total_K, ks, seed, variant=None):
    """ks: K extent per group (offsets are their inclusive prefix)."""
    A, B, sa, sb = _data(seed, (M, total_K), (N, total_K), G * M, G * N)
    off = np.cumsum(ks).astype(np.int32)
    tA, tB, tsa, tsb, toff = _cuda(A, B, sa, sb, off)
    out = torch.full((G, M, N), 0x5A5A, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    _run(fx.f8f8bf16_rowwise_grouped_k_offsets, variant, tA, tB, tsa, tsb, toff, out)
    torch.cuda.synchronize()
    got = bits_of(out).reshape(G * M, N)
    ref, _ = orc.k_offsets(A, B, sa.reshape(G, M), sb.reshape(G, N), off)
    ab, _ = orc.k_offsets(abs_codes(A), abs_codes(B), np.abs(sa).reshape(G, M),
                          np.abs(sb).reshape(G, N), off)
    return compare(got.ravel(), ref.ravel(), ab.ravel(), f"ragged K {variant} {ks}"), got


@pytest.mark.parametrize("variant", _variants("ragn_"))
def test_ragged_n_every_variant(orc, variant):
    # groups of 0, 3 (narrower than a store), 300 (a partial tile), 517, 1 and 203 columns;
    # the output is wider than the groups (columns past the last group stay untouched)
    cols = [0, 3, 300, 517, 1, 203]
    _n_offsets_case(orc, 6, 200, 1032, 400, cols, seed=1, variant=variant)
    assert fx.device_status() == 0


@pytest.mark.parametrize("variant", _variants("ragk_"))
def test_ragged_k_every_variant(orc, variant):
    # slices of 0, 16 (half a 32-byte MMA step), 128 (one block), 144, 400 (a block and a
    # half step) and 912 elements
    ks = [0, 16, 128, 144, 400, 912]
    _, got = _k_offsets_case(orc, 6, 200, 392, 1600, ks, seed=2, variant=variant)
    assert np.all(got[:200] == 0), "an empty slice must give +0.0"
    assert fx.device_status() == 0


def test_ragged_n_small_m_and_many_groups(orc):
    # few rows per slab (the swap-AB plan), 40 groups, some empty
    rng = np.random.default_rng(3)
    cols = rng.integers(0, 90, size=40)
    cols[::7] = 0
    total_N = int(-(-cols.sum() // 8) * 8) + 16
    st = _n_offsets_case(orc, 40, 12, total_N, 256, cols.tolist(), seed=3)
    assert st["elements"] == 12 * int(cols.sum())


def test_ragged_k_next_group_data_never_leaks(orc):
    # group 1's slice [48, 64) holds NaN codes in A: group 0's slice ends half-way through
    # the 32-byte MMA step over [32, 64), so any use of the bytes past its end would turn
    # group 0's results into NaN (group 1's own results are NaN, as the oracle's are)
    G, M, N, total_K = 3, 130, 264, 512
    ks = [48, 16, 448]
    A, B, sa, sb = _data(4, (M, total_K), (N, total_K), G * M, G * N)
    A[:, 48:64] = 0x7F
    off = np.cumsum(ks).astype(np.int32)
    tA, tB, tsa, tsb, toff = _cuda(A, B, sa, sb, off)
    out = fx.f8f8bf16_rowwise_grouped_k_offsets(tA, tB, tsa, tsb, toff)
    torch.cuda.synchronize()
    got = bits_of(out).reshape(G * M, N)
    ref, _ = orc.k_offsets(A, B, sa.reshape(G, M), sb.reshape(G, N), off)
    ab, _ = orc.k_offsets(abs_codes(A), abs_codes(B), np.abs(sa).reshape(G, M),
                          np.abs(sb).reshape(G, N), off)
    assert not np.isnan(oracle.bf16_bits_to_float(ref[:M])).any()
    assert np.isnan(oracle.bf16_bits_to_float(ref[M:2 * M])).all()
    compare(got.ravel(), ref.ravel(), ab.ravel(), "ragged K with poisoned neighbours")


def test_ragged_k_previous_group_data_never_leaks(orc):
    # group 0's slice [0, 48) ends in NaN codes over [32, 48); group 1's slice [48, 96)
    # starts half-way through the 32-byte MMA step over [32, 64) of the block that is
    # loaded from K = 0, so any use of the bytes before its start would turn group 1's
    # results into NaN (group 0's own results are NaN, as the oracle's are)
    G, M, N, total_K = 3, 130, 264, 512
    ks = [48, 48, 416]
    A, B, sa, sb = _data(5, (M, total_K), (N, total_K), G * M, G * N)
    A[:, 32:48] = 0x7F
    B[:, 40:48] = 0xFF
    off = np.cumsum(ks).astype(np.int32)
    tA, tB, tsa, tsb, toff = _cuda(A, B, sa, sb, off)
    out = fx.f8f8bf16_rowwise_grouped_k_offsets(tA, tB, tsa, tsb, toff)
    torch.cuda.synchronize()
    got = bits_of(out).reshape(G * M, N)
    ref, _ = orc.k_offsets(A, B, sa.reshape(G, M), sb.reshape(G, N), off)
    ab, _ = orc.k_offsets(abs_codes(A), abs_codes(B), np.abs(sa).reshape(G, M),
                          np.abs(sb).reshape(G, N), off)
    assert np.isnan(oracle.bf16_bits_to_float(ref[:M])).all()
    assert not np.isnan(oracle.bf16_bits_to_float(ref[M:])).any()
    compare(got.ravel(), ref.ravel(), ab.ravel(), "ragged K after poisoned neighbours")


def test_ragged_k_bad_slice_is_zero_and_flagged(orc):
    # a slice ending off the 16-element grid: that group is not computed (+0.0) and the
    # status bit is set; the other groups are unaffected
    G, M, N, total_K = 3, 64, 128, 256
    ks = [64, 24, 168]   # group 1 ends at 88 and group 2 starts there: both off the grid
    A, B, sa, sb = _data(5, (M, total_K), (N, total_K), G * M, G * N)
    off = np.cumsum(ks).astype(np.int32)
    tA, tB, tsa, tsb, toff = _cuda(A, B, sa, sb, off)
    fx.device_status()
    out = fx.f8f8bf16_rowwise_grouped_k_offsets(tA, tB, tsa, tsb, toff)
    torch.cuda.synchronize()
    assert fx.device_status() & fx.MSLKB_DEV_BAD_SLICE
    got = bits_of(out).reshape(G * M, N)
    assert np.all(got[M:] == 0)
    ref, _ = orc.k_offsets(A, B, sa.reshape(G, M), sb.reshape(G, N), off)
    ab, _ = orc.k_offsets(abs_codes(A), abs_codes(B), np.abs(sa).reshape(G, M),
                          np.abs(sb).reshape(G, N), off)
    compare(got[:M].ravel(), ref[:M].ravel(), ab[:M].ravel(), "ragged K good group")


def test_ragged_clamped_offsets(orc):
    # offsets past the end are clamped (status bit), as row counts are
    G, M, total_N, K = 3, 40, 64, 128
    A, B, sa, sb = _data(6, (G, M, K), (total_N, K), G * M, total_N)
    off = np.array([24, 20, 100], np.int32)   # a decreasing step and a last one past total_N
    tA, tB, tsa, tsb, toff = _cuda(A, B, sa, sb, off)
    fx.device_status()
    out = fx.f8f8bf16_rowwise_grouped_n_offsets(tA, tB, tsa, tsb, toff)
    torch.cuda.synchronize()
    assert fx.device_status() & fx.MSLKB_DEV_MSIZES_CLAMPED
    got = bits_of(out).reshape(M, total_N)
    ref, clamped = orc.n_offsets(A, B, sa.reshape(G, M), sb, off)
    assert clamped
    ab, _ = orc.n_offsets(abs_codes(A), abs_codes(B), np.abs(sa).reshape(G, M), np.abs(sb), off)
    compare(got.ravel(), ref.ravel(), ab.ravel(), "ragged N clamped")


def test_ragged_k_zero_total(orc):
    # total_K = 0: every slab +0.0
    out = fx.f8f8bf16_rowwise_grouped_k_offsets(
        torch.zeros((8, 0), dtype=torch.uint8, device="cuda"),
        torch.zeros((16, 0), dtype=torch.uint8, device="cuda"),
        torch.ones(16, device="cuda"), torch.ones(32, device="cuda"),
        torch.zeros(2, dtype=torch.int32, device="cuda"),
        out=torch.full((2, 8, 16), 1.0, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert torch.count_nonzero(out.view(torch.int16)).item() == 0


def test_ragged_graph_replay(orc):
    # both ragged calls captured in one CUDA graph and replayed: same bits as eager
    G, M, total_N, K = 4, 96, 512, 256
    A, B, sa, sb = _data(7, (G, M, K), (total_N, K), G * M, total_N)
    off = np.cumsum([100, 0, 250, 150]).astype(np.int32)
    tA, tB, tsa, tsb, toff = _cuda(A, B, sa, sb, off)
    A2, B2, sa2, sb2 = _data(8, (M, 512), (264, 512), G * M, G * 264)
    off2 = np.cumsum([128, 96, 32, 256]).astype(np.int32)
    uA, uB, usa, usb, uoff = _cuda(A2, B2, sa2, sb2, off2)
    eager_n = fx.f8f8bf16_rowwise_grouped_n_offsets(tA, tB, tsa, tsb, toff)
    eager_k = fx.f8f8bf16_rowwise_grouped_k_offsets(uA, uB, usa, usb, uoff)
    out_n = torch.zeros_like(eager_n)
    out_k = torch.zeros_like(eager_k)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fx.f8f8bf16_rowwise_grouped_n_offsets(tA, tB, tsa, tsb, toff, out=out_n)
        fx.f8f8bf16_rowwise_grouped_k_offsets(uA, uB, usa, usb, uoff, out=out_k)
    with torch.cuda.stream(s):
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_n.view(torch.int16), eager_n.view(torch.int16))
    assert torch.equal(out_k.view(torch.int16), eager_k.view(torch.int16))
