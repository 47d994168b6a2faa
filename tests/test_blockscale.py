"""GPU parity of the block-scaled (groupwise) stacked variant against the oracle, through the
C ABI: scale blocks of 128 along K and N, every K block's partial sum scaled on its way
into the fp32 accumulator."""
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


def _variants():
    try:
        fxbuild.build()
        return [fx.variant_name(i) for i in range(fx.mslkb_num_variants())
                if fx.variant_name(i).startswith("blockscale_")]
    except Exception:  # noqa: BLE001 - collection must not depend on a toolchain
        return []


def _case(seed, G, m_sizes, N, K, extra=0, wide=False):
    g = torch.Generator().manual_seed(seed)
    rows = int(sum(m_sizes)) + extra
    A = random_codes((rows, K), g).numpy()
    B = random_codes((G, N, K), g).numpy()
    nkb, nnb = K // 128, N // 128
    if wide:   # scales over many binades, so that a scale taken from the wrong block shows
        sa = np.exp2(torch.randint(-12, 12, (rows, nkb), generator=g).numpy()).astype(np.float32)
        sb = np.exp2(torch.randint(-12, 12, (G, nnb, nkb), generator=g).numpy()).astype(np.float32)
        sa *= (torch.rand((rows, nkb), generator=g).numpy() + 0.5).astype(np.float32)
    else:
        sa = (torch.rand((rows, nkb), generator=g) * 2 + 0.01).numpy().astype(np.float32)
        sb = (torch.rand((G, nnb, nkb), generator=g) * 2 + 0.01).numpy().astype(np.float32)
    return A, B, sa, sb, np.asarray(m_sizes, np.int64), rows


def _run(A, B, sa, sb, m, rows, N, variant=None, poison=0x5A5A):
    tA, tB, tsa, tsb, tm = [torch.from_numpy(np.ascontiguousarray(x)).cuda()
                            for x in (A, B, sa, sb, m)]
    out = torch.full((rows, N), poison, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    if variant is not None:
        fx.mslkb_force_variant(fx.variant_index(variant))
    try:
        fx.f8f8bf16_groupwise_grouped_stacked(tA, tB, tsa, tsb, tm, out=out)
    finally:
        if variant is not None:
            fx.mslkb_force_variant(-1)
    torch.cuda.synchronize()
    return bits_of(out).reshape(rows, N)


def _check(orc, A, B, sa, sb, m, rows, got, what, poison=0x5A5A):
    ref, _ = orc.blockwise_stacked(A, B, sa, sb, m, total_M=rows,
                                   out=np.full((rows, B.shape[1]), poison, np.uint16))
    ab, _ = orc.blockwise_stacked(abs_codes(A), abs_codes(B), np.abs(sa), np.abs(sb), m,
                                  total_M=rows)
    owned = int(np.clip(m, 0, None).sum())
    assert np.all(got[owned:] == poison), f"{what}: rows past the last group written"
    return compare(got[:owned].ravel(), ref[:owned].ravel(), ab[:owned].ravel(), what)


@pytest.mark.parametrize("variant", _variants())
def test_blockscale_every_variant(orc, variant):
    # groups ending inside tiles, an empty group, N of 3 scale blocks (a partial 256-wide
    # tile), 7 K blocks
    m = [130, 0, 1, 257, 64]
    A, B, sa, sb, m, rows = _case(11, 5, m, 384, 896, extra=5)
    got = _run(A, B, sa, sb, m, rows, 384, variant)
    _check(orc, A, B, sa, sb, m, rows, got, variant)
    assert fx.device_status() == 0


def test_blockscale_wide_scales(orc):
    # scales spread over 24 binades per block: a scale applied to the wrong K block or the
    # wrong 128-column block is off by orders of magnitude
    A, B, sa, sb, m, rows = _case(12, 3, [200, 70, 300], 512, 1024, wide=True)
    got = _run(A, B, sa, sb, m, rows, 512)
    _check(orc, A, B, sa, sb, m, rows, got, "wide scales")


def test_blockscale_equals_rowwise_for_constant_scales(orc):
    # scales constant over the K blocks: the block-scaled result agrees with the rowwise
    # kernel's within the parity tolerance of both
    A, B, sa, sb, m, rows = _case(13, 2, [300, 212], 256, 1024)
    sa[:] = sa[:, :1]
    sb[:] = sb[:, :, :1]
    got = _run(A, B, sa, sb, m, rows, 256)
    _check(orc, A, B, sa, sb, m, rows, got, "constant block scales")
    sa_row = np.ascontiguousarray(sa[:, 0])
    sb_gn = np.ascontiguousarray(np.repeat(sb[:, :, 0], 128, axis=1))
    tA, tB, tsa, tsb, tm = [torch.from_numpy(np.ascontiguousarray(x)).cuda()
                            for x in (A, B, sa_row, sb_gn, m)]
    row = bits_of(fx.f8f8bf16_rowwise_grouped_stacked(tA, tB, tsa, tsb, tm)).reshape(rows, 256)
    ref, _ = orc.stacked(A, B, sa_row, sb_gn, m)
    ab, _ = orc.stacked(abs_codes(A), abs_codes(B), np.abs(sa_row), np.abs(sb_gn), m)
    compare(row.ravel(), ref.ravel(), ab.ravel(), "rowwise on the same data")
    # the two oracles hold the same exact value here, so their bf16 bits agree
    assert np.array_equal(ref, orc.blockwise_stacked(A, B, sa, sb, m)[0])


@pytest.mark.parametrize("m", [[1, 0, 3, 2], [9, 16, 0, 30]])
def test_blockscale_decode_shapes(orc, m):
    # few rows per group: the planner's swap-AB tiles, split along K over every CTA
    A, B, sa, sb, m, rows = _case(14, 4, m, 1024, 2048, wide=True)
    got = _run(A, B, sa, sb, m, rows, 1024)
    _check(orc, A, B, sa, sb, m, rows, got, f"decode {m.tolist()}")
    assert fx.device_status() == 0


@pytest.mark.parametrize("K", [128, 384, 640])
@pytest.mark.parametrize("split", [0, 2])
def test_blockscale_swap_odd_block_counts(orc, K, split):
    # swap-AB tiles take two K blocks per chunk: 1, 3 and 5 blocks leave a chunk of one,
    # and split pieces may start on an odd block; both swap-AB widths, split or not
    A, B, sa, sb, m, rows = _case(16, 3, [5, 0, 19], 512, K, wide=True)
    fx.mslkb_set_split_k(split)
    try:
        for v in ("blockscale_swap_w128xa16_tma", "blockscale_swap_w128xa32_tma"):
            got = _run(A, B, sa, sb, m, rows, 512, v)
            _check(orc, A, B, sa, sb, m, rows, got, f"K={K} split={split} {v}")
    finally:
        fx.mslkb_set_split_k(1)
    assert fx.device_status() == 0


def test_blockscale_k_zero():
    out = fx.f8f8bf16_groupwise_grouped_stacked(
        torch.zeros((8, 0), dtype=torch.uint8, device="cuda"),
        torch.zeros((2, 128, 0), dtype=torch.uint8, device="cuda"),
        torch.ones(0, device="cuda"), torch.ones(0, device="cuda"),
        torch.tensor([5, 3], dtype=torch.int64, device="cuda"),
        out=torch.full((8, 128), 1.0, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert torch.count_nonzero(out.view(torch.int16)).item() == 0
